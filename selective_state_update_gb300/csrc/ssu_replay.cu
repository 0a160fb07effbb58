// ssu_replay.cu -- decode on the checkpoint + buffer form of the state.
//
// Article "ReplaySSM: Cache SSM Inputs, Not State", section 核心做法: the
// state of a slot is a checkpoint plus the inputs (v, dt', k) = (x, dt', B) of
// the steps since the last fold.  Unrolled, the state after the current step
// c is
//     S_c = gamma_{0:c} S_ckpt + sum_{j<=c} gamma_{j+1:c} dt'_j x_j B_j^T,
//     gamma_{i:c} = prod_{m=i..c} exp(A dt'_m),
// so y = S_c . C can be read out without forming S_c:
//     y = gamma_{0:c} (S_ckpt . C) + sum_j gamma_{j+1:c} dt'_j x_j (B_j . C).
// A step that does not fill the buffer does exactly that and appends its
// inputs; the checkpoint is read but not written.  The step that fills it
// folds the entries into the checkpoint in order (the plain update, carried in
// fp32), reads y out of the result and writes the checkpoint back once.
// Section 数据与边界: the checkpoint is read every step and written once every
// L steps, so the state traffic per step drops from a read and a write to
// about a read.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows), one CTA each.
// One thread requests the checkpoint tile and every buffered entry of the
// tile (x rows, dt' rows, B of the group) as bulk asynchronous copies (TMA
// engine) completing on one mbarrier, so all of a unit's reads are in flight
// together; meanwhile the CTA loads the current token and computes its row
// scalars.
#include <atomic>

#include "ssu_device.cuh"

namespace ssu {

// Dynamic shared memory for a buffer of `len` entries: the checkpoint tile;
// the buffered entries as stored (x rows and dt' rows of this tile, B of the
// group); C and the current token's B as fp32; the B.C dot products; per-row
// per-entry decays and input terms (for a fold); the current token's row
// scalars and each row's readout coefficients; the mbarrier.
template <typename TS, int L>
struct ReplaySmem {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kTileBytes = kTileRows * kN * static_cast<int>(sizeof(TS));
    int tile, xe, de, be, cs, bc, dots, rowa, rowb, rowq, rowg, bar, bytes;
    __host__ __device__ static int up(int v) { return (v + 127) / 128 * 128; }
    __host__ __device__ ReplaySmem(int len, int io) {
        tile = 0;
        xe = up(kTileBytes);                      // io   [len][kTileRows]
        de = up(xe + len * kTileRows * io);       // f32  [len][kTileRows]
        be = up(de + len * kTileRows * 4);        // io   [len][N]
        cs = up(be + len * kN * io);              // f32  [N]
        bc = up(cs + kN * 4);                     // f32  [N]
        dots = up(bc + kN * 4);                   // f32  [len]
        rowa = up(dots + len * 4);                // f32  [len][kTileRows]
        rowb = up(rowa + len * kTileRows * 4);    // f32  [len][kTileRows]
        rowq = up(rowb + len * kTileRows * 4);    // f32x4 [kTileRows]
        rowg = up(rowq + kTileRows * 16);         // f32x2 [kTileRows]
        bar = up(rowg + kTileRows * 8);           // u64
        bytes = bar + 16;
    }
};

__device__ __forceinline__ float raw_to_float(const unsigned char *base, int i, int io_dtype) {
    if (io_dtype == kF32) return reinterpret_cast<const float *>(base)[i];
    return bits_to_float(reinterpret_cast<const unsigned short *>(base)[i], io_dtype);
}

// Not inlined: the readout walk of a row from the newest entry to the oldest,
// w = gamma_{j+1:c} along the way and gamma_{0:c} at the end.
static __device__ __noinline__ float2 readout_walk(int c, int r, float Ah, float dA_now, float dtx_now,
                                                   const float *de, const unsigned char *xe, const float *dots,
                                                   int io_dtype) {
    float w = 1.f;
    float hist = fmaf(w * dtx_now, dots[c], 0.f);
    w *= dA_now;
    for (int j = c - 1; j >= 0; --j) {
        const float d = de[j * kTileRows + r];
        const float x = raw_to_float(xe, j * kTileRows + r, io_dtype);
        hist = fmaf(w * (d * x), dots[j], hist);
        w *= decay(Ah, d);
    }
    return make_float2(w, hist);
}

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads)
    ssu_replay_kernel(const KParams p) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    const int len = p.rlen;
    const int io = p.io_dtype == kF32 ? 4 : 2;
    const ReplaySmem<TS, L> lay(len, io);
    TS *tile = reinterpret_cast<TS *>(smem + lay.tile);
    unsigned char *xe = smem + lay.xe;
    float *de = reinterpret_cast<float *>(smem + lay.de);
    unsigned char *be = smem + lay.be;
    float *sC = reinterpret_cast<float *>(smem + lay.cs);
    float *sBc = reinterpret_cast<float *>(smem + lay.bc);
    float *dots = reinterpret_cast<float *>(smem + lay.dots);
    float *rowa = reinterpret_cast<float *>(smem + lay.rowa);
    float *rowb = reinterpret_cast<float *>(smem + lay.rowb);
    float4 *rowq = reinterpret_cast<float4 *>(smem + lay.rowq);
    float2 *rowg = reinterpret_cast<float2 *>(smem + lay.rowg);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bar);

    const int64_t unit = blockIdx.x;
    const int ptile = static_cast<int>(unit % p.ptiles);
    const int64_t bh = unit / p.ptiles;
    const int h = static_cast<int>(bh % p.H);
    const int64_t b = bh / p.H;
    const int g = h / p.heads_per_group;
    const int tid = threadIdx.x;

    // Slot and buffered count (uniform over the CTA).
    int64_t s;
    if (!table_slot(p, p.rd, b, 0, b, b, &s) || !slot_ok(p, s)) return;
    const bool pad = s == p.pad;
    int c = 0;
    if (!pad) {
        c = __ldg(p.cnt_in + b);
        if (c < 0 || c >= len) {
            flag(p.status, kDevBadCount);
            return;
        }
    }
    const bool fold = pad || c + 1 == len;
    if (tid == 0 && h == 0 && ptile == 0) p.cnt_out[b] = fold ? 0 : c + 1;

    const int row0 = ptile * kTileRows;
    const int rows_here = min(kTileRows, p.P - row0);
    const int64_t head_row0 = static_cast<int64_t>(h) * p.P + row0;
    // Everything the unit reads from the slot -- the checkpoint tile and each
    // buffered entry's x rows, dt' rows and B -- is requested at once, as
    // bulk asynchronous copies completing on one mbarrier.
    const bool bulk_entries = p.rbulk != 0;
    if (tid == 0 && !pad) {
        uint32_t bytes = static_cast<uint32_t>(rows_here) * N * sizeof(TS);
        if (bulk_entries) bytes += static_cast<uint32_t>(c) * (rows_here * (io + 4) + N * io);
        mbar_init(bar, 1);
        mbar_arrive_expect(bar, bytes);
        bulk_load(tile, static_cast<const TS *>(p.state) + (s * p.H * p.P + head_row0) * N,
                  static_cast<uint32_t>(rows_here) * N * sizeof(TS), bar);
        if (bulk_entries) {
            for (int j = 0; j < c; ++j) {
                const int64_t e = ((s * len + j) * p.H + h) * static_cast<int64_t>(p.P) + row0;
                bulk_load(xe + j * kTileRows * io, static_cast<const unsigned char *>(p.xbuf) + e * io,
                          static_cast<uint32_t>(rows_here) * io, bar);
                bulk_load(de + j * kTileRows, p.dtbuf + e, static_cast<uint32_t>(rows_here) * 4, bar);
                const int64_t eb = ((s * len + j) * p.G + g) * static_cast<int64_t>(N);
                bulk_load(be + j * N * io, static_cast<const unsigned char *>(p.Bbuf) + eb * io,
                          static_cast<uint32_t>(N) * io, bar);
            }
        }
    }
    if (!pad && !bulk_entries) {
        // Unaligned buffers: plain loads of the same entries.
        for (int i = tid; i < c * rows_here; i += NT) {
            const int j = i / rows_here, r = i % rows_here;
            const int64_t e = ((s * len + j) * p.H + h) * static_cast<int64_t>(p.P) + row0 + r;
            de[j * kTileRows + r] = __ldg(p.dtbuf + e);
            if (io == 4)
                reinterpret_cast<unsigned int *>(xe)[j * kTileRows + r] = load_bits<true>(p.xbuf, e);
            else
                reinterpret_cast<unsigned short *>(xe)[j * kTileRows + r] =
                    static_cast<unsigned short>(load_bits<false>(p.xbuf, e));
        }
        for (int i = tid; i < c * N; i += NT) {
            const int j = i / N, n = i % N;
            const int64_t eb = ((s * len + j) * p.G + g) * static_cast<int64_t>(N) + n;
            if (io == 4)
                reinterpret_cast<unsigned int *>(be)[j * N + n] = load_bits<true>(p.Bbuf, eb);
            else
                reinterpret_cast<unsigned short *>(be)[j * N + n] = static_cast<unsigned short>(load_bits<false>(p.Bbuf, eb));
        }
    }

    // The current token: B, C, and the row scalars; its entry is appended
    // when the buffer does not fill.
    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    const int64_t bo = b * p.Bs[0] + g * p.Bs[1];
    const int64_t co = b * p.Cs[0] + g * p.Cs[1];
    const bool append_b = !fold && h % p.heads_per_group == 0 && ptile == 0;
    for (int n = tid; n < N; n += NT) {
        const uint32_t bb = io == 4 ? load_bits<true>(p.B, bo + n * p.Bs[2]) : load_bits<false>(p.B, bo + n * p.Bs[2]);
        const uint32_t cb = io == 4 ? load_bits<true>(p.C, co + n * p.Cs[2]) : load_bits<false>(p.C, co + n * p.Cs[2]);
        sBc[n] = bits_to_float(bb, p.io_dtype);
        sC[n] = bits_to_float(cb, p.io_dtype);
        if (append_b) {
            const int64_t e = ((s * len + c) * p.G + g) * static_cast<int64_t>(N) + n;
            if (io == 4)
                static_cast<unsigned int *>(p.Bbuf)[e] = bb;
            else
                static_cast<unsigned short *>(p.Bbuf)[e] = static_cast<unsigned short>(bb);
        }
    }
    for (int r = tid; r < rows_here; r += NT) {
        const int pr = row0 + r;
        const int64_t xo = b * p.xs[0] + h * p.xs[1] + pr * p.xs[2];
        const int64_t dto = b * p.dts[0] + h * p.dts[1] + pr * p.dts[2];
        const int64_t zo = b * p.zs[0] + h * p.zs[1] + pr * p.zs[2];
        const uint32_t xb = io == 4 ? load_bits<true>(p.x, xo) : load_bits<false>(p.x, xo);
        const uint32_t db = p.dt_dtype == kF32 ? load_bits<true>(p.dt, dto) : load_bits<false>(p.dt, dto);
        const uint32_t zb = p.z ? (io == 4 ? load_bits<true>(p.z, zo) : load_bits<false>(p.z, zo)) : 0u;
        const float dtv = bits_to_float(db, p.dt_dtype);
        rowq[r] = row_scalars(RowInputs{dtv, bits_to_float(xb, p.io_dtype), bits_to_float(zb, p.io_dtype)}, Ah, bias,
                              p.softplus, p.z != nullptr);
        if (!fold) {
            const int64_t e = ((s * len + c) * p.H + h) * static_cast<int64_t>(p.P) + pr;
            p.dtbuf[e] = processed_step(dtv, bias, p.softplus);
            if (io == 4)
                static_cast<unsigned int *>(p.xbuf)[e] = xb;
            else
                static_cast<unsigned short *>(p.xbuf)[e] = static_cast<unsigned short>(xb);
        }
    }
    __syncthreads();
    int timed_out = 0;
    if (!pad && !mbar_wait_bounded(bar, 0)) timed_out = 1;
    if (__syncthreads_or(timed_out)) {
        if (tid == 0) flag(p.status, kDevTimeout);
        return;
    }

    if (!fold) {
        // B_j . C for the entries and the current token: one warp (or the
        // whole CTA when it is narrower than a warp) per dot.
        constexpr int W = NT < 32 ? NT : 32;
        constexpr unsigned kMask = W == 32 ? 0xffffffffu : (1u << W) - 1u;
        const int warp = tid / W, wl = tid % W;
        for (int j = warp; j <= c; j += NT / W) {
            float acc = 0.f;
            for (int n = wl; n < N; n += W)
                acc = fmaf(j < c ? raw_to_float(be, j * N + n, p.io_dtype) : sBc[n], sC[n], acc);
#pragma unroll
            for (int off = W / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kMask, acc, off);
            if (wl == 0) dots[j] = acc;
        }
        __syncthreads();
        for (int r = tid; r < rows_here; r += NT) {
            const float4 q = rowq[r];
            rowg[r] = readout_walk(c, r, Ah, q.x, q.y, de, xe, dots, p.io_dtype);
        }
        __syncthreads();
    } else if (c > 0) {
        // Decay and input term of every entry and row, for the fold.
        for (int i = tid; i < c * rows_here; i += NT) {
            const int j = i / rows_here, r = i % rows_here;
            const float d = de[j * kTileRows + r];
            rowa[j * kTileRows + r] = decay(Ah, d);
            rowb[j * kTileRows + r] = d * raw_to_float(xe, j * kTileRows + r, p.io_dtype);
        }
        __syncthreads();
    }

    const int lane = tid % L;
    const int slot_row = tid / L;
    float cv[kElemsPerThread];
    T::gather(sC, lane, cv);
    TS *ckpt = static_cast<TS *>(p.state) + (s * p.H * p.P + head_row0) * N;
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int rr = slot_row + j * kRowSlots;  // row within the tile
        const bool live = rr < rows_here;
        const int rq = live ? rr : 0;
        float sv[kElemsPerThread];
        if (!pad && live) {
            T::load_row_smem(tile + rr * N, lane, sv);
        } else {
#pragma unroll
            for (int i = 0; i < kElemsPerThread; ++i) sv[i] = 0.f;
        }
        const float4 q = rowq[rq];
        float y;
        if (fold) {
            float bv[kElemsPerThread];
            // The buffered steps in order, as the plain update made them ...
            for (int e = 0; e < c; ++e) {
#pragma unroll
                for (int i = 0; i < kElemsPerThread; ++i) bv[i] = raw_to_float(be, e * N + T::elem(lane, i), p.io_dtype);
                const float a = rowa[e * kTileRows + rq], dx = rowb[e * kTileRows + rq];
#pragma unroll
                for (int i = 0; i < kElemsPerThread; ++i) sv[i] = fmaf(sv[i], a, dx * bv[i]);
            }
            // ... then the current token, whose state y is read from.
            T::gather(sBc, lane, bv);
            const float sum = row_sum<L>(update_elems(sv, bv, cv, q.x, q.y));
            y = output(sum, Dh, q.z, q.w);
            if (live && !pad) T::store_row(ckpt + rr * N, lane, sv);
        } else {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kElemsPerThread; ++i) acc = fmaf(sv[i], cv[i], acc);
            const float sum = row_sum<L>(acc);
            const float2 gw = rowg[rq];
            y = output(fmaf(gw.x, sum, gw.y), Dh, q.z, q.w);
        }
        if (live && lane == 0) store_small(p.y, b * p.ys[0] + h * p.ys[1] + (row0 + rr) * p.ys[2], p.io_dtype, y);
    }
}

template <typename TS, int L>
static cudaError_t smem_opt_in() {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(ssu_replay_kernel<TS, L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ReplaySmem<TS, L>(kMaxReplayLen, 4).bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, int64_t batch, cudaStream_t stream) {
    cudaError_t e = smem_opt_in<TS, L>();
    if (e != cudaSuccess) return e;
    const int64_t units = batch * p.H * p.ptiles;
    ssu_replay_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads,
                               ReplaySmem<TS, L>(p.rlen, p.io_dtype == kF32 ? 4 : 2).bytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename TS>
static cudaError_t launch_lanes(int lanes, const KParams &p, int64_t batch, cudaStream_t stream) {
    switch (lanes) {
    case 1: return launch_t<TS, 1>(p, batch, stream);
    case 2: return launch_t<TS, 2>(p, batch, stream);
    case 4: return launch_t<TS, 4>(p, batch, stream);
    case 8: return launch_t<TS, 8>(p, batch, stream);
    case 16: return launch_t<TS, 16>(p, batch, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_replay(int state_dtype, int lanes, const KParams &p, int64_t batch, cudaStream_t stream) {
    switch (state_dtype) {
    case kF32: return launch_lanes<float>(lanes, p, batch, stream);
    case kF16: return launch_lanes<__half>(lanes, p, batch, stream);
    case kBF16: return launch_lanes<__nv_bfloat16>(lanes, p, batch, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
