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
// The checkpoint tile arrives by one bulk asynchronous copy (TMA engine,
// mbarrier completion) while the CTA stages the entries' B vectors, C and
// the per-row, per-entry scalars {exp(A dt'_j), dt'_j x_j} in shared memory.
#include <atomic>

#include "ssu_device.cuh"

namespace ssu {

// Dynamic shared memory for a buffer of `len` entries: the checkpoint tile,
// B of every entry and the current token, C, the B.C dot products, the
// per-row per-entry decays and input terms, the current token's row scalars
// and the readout coefficients of each row, the mbarrier.
template <typename TS, int L>
struct ReplaySmem {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kTileBytes = kTileRows * kN * static_cast<int>(sizeof(TS));
    int tile, bs, cs, dots, rowa, rowb, rowq, rowg, bar, bytes;
    __host__ __device__ explicit ReplaySmem(int len) {
        tile = 0;
        bs = kTileBytes;                          // float [len][N]
        cs = bs + len * kN * 4;                   // float [N]
        dots = cs + kN * 4;                       // float [len], padded to 32
        rowa = dots + ((len + 31) / 32) * 32 * 4;  // float [len][kTileRows]
        rowb = rowa + len * kTileRows * 4;        // float [len][kTileRows]
        rowq = rowb + len * kTileRows * 4;        // float4 [kTileRows]
        rowg = rowq + kTileRows * 16;             // float2 [kTileRows]
        bar = rowg + kTileRows * 8;               // uint64
        bytes = bar + 16;
    }
};

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads)
    ssu_replay_kernel(const KParams p) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    const int len = p.rlen;
    const ReplaySmem<TS, L> lay(len);
    TS *tile = reinterpret_cast<TS *>(smem + lay.tile);
    float *sB = reinterpret_cast<float *>(smem + lay.bs);
    float *sC = reinterpret_cast<float *>(smem + lay.cs);
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
    if (tid == 0 && !pad) {
        const uint32_t bytes = static_cast<uint32_t>(rows_here) * N * sizeof(TS);
        mbar_init(bar, 1);
        mbar_arrive_expect(bar, bytes);
        bulk_load(tile, static_cast<const TS *>(p.state) + (s * p.H * p.P + head_row0) * N, bytes, bar);
    }

    // B of the entries and of the current token (entry c), C.
    const int64_t bo = b * p.Bs[0] + g * p.Bs[1];
    for (int i = tid; i < (c + 1) * N; i += NT) {
        const int j = i / N, n = i % N;
        float v;
        if (j < c) {
            const int64_t e = ((s * len + j) * p.G + g) * static_cast<int64_t>(N) + n;
            v = bits_to_float(p.io_dtype == kF32 ? load_bits<true>(p.Bbuf, e) : load_bits<false>(p.Bbuf, e),
                              p.io_dtype);
        } else {
            v = bits_to_float(p.io_dtype == kF32 ? load_bits<true>(p.B, bo + n * p.Bs[2])
                                                 : load_bits<false>(p.B, bo + n * p.Bs[2]),
                              p.io_dtype);
        }
        sB[j * N + n] = v;
    }
    const int64_t co = b * p.Cs[0] + g * p.Cs[1];
    for (int n = tid; n < N; n += NT)
        sC[n] = bits_to_float(p.io_dtype == kF32 ? load_bits<true>(p.C, co + n * p.Cs[2])
                                                 : load_bits<false>(p.C, co + n * p.Cs[2]),
                              p.io_dtype);
    // Per row and entry: exp(A dt'_j) and dt'_j x_j.
    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    for (int i = tid; i < c * rows_here; i += NT) {
        const int j = i / rows_here, r = i % rows_here;
        const int64_t e = ((s * len + j) * p.H + h) * static_cast<int64_t>(p.P) + row0 + r;
        const float d = __ldg(p.dtbuf + e);
        const float x = bits_to_float(p.io_dtype == kF32 ? load_bits<true>(p.xbuf, e) : load_bits<false>(p.xbuf, e),
                                      p.io_dtype);
        rowa[j * kTileRows + r] = decay(Ah, d);
        rowb[j * kTileRows + r] = d * x;
    }
    // The current token: row scalars, and its entry when it is buffered.
    for (int r = tid; r < rows_here; r += NT) {
        const int pr = row0 + r;
        const uint32_t xb = p.io_dtype == kF32 ? load_bits<true>(p.x, b * p.xs[0] + h * p.xs[1] + pr * p.xs[2])
                                               : load_bits<false>(p.x, b * p.xs[0] + h * p.xs[1] + pr * p.xs[2]);
        const float dtv = bits_to_float(
            p.dt_dtype == kF32 ? load_bits<true>(p.dt, b * p.dts[0] + h * p.dts[1] + pr * p.dts[2])
                               : load_bits<false>(p.dt, b * p.dts[0] + h * p.dts[1] + pr * p.dts[2]),
            p.dt_dtype);
        float zv = 0.f;
        if (p.z)
            zv = bits_to_float(p.io_dtype == kF32 ? load_bits<true>(p.z, b * p.zs[0] + h * p.zs[1] + pr * p.zs[2])
                                                  : load_bits<false>(p.z, b * p.zs[0] + h * p.zs[1] + pr * p.zs[2]),
                               p.io_dtype);
        const float4 q = row_scalars(RowInputs{dtv, bits_to_float(xb, p.io_dtype), zv}, Ah, bias, p.softplus,
                                     p.z != nullptr);
        rowq[r] = q;
        rowa[c * kTileRows + r] = q.x;
        rowb[c * kTileRows + r] = q.y;
        if (!fold) {
            const int64_t e = ((s * len + c) * p.H + h) * static_cast<int64_t>(p.P) + pr;
            p.dtbuf[e] = processed_step(dtv, bias, p.softplus);
            if (p.io_dtype == kF32)
                static_cast<unsigned int *>(p.xbuf)[e] = xb;
            else
                static_cast<unsigned short *>(p.xbuf)[e] = static_cast<unsigned short>(xb);
        }
    }
    // The group's B is appended once, by the first head of the group.
    if (!fold && h % p.heads_per_group == 0 && ptile == 0) {
        for (int n = tid; n < N; n += NT) {
            const int64_t e = ((s * len + c) * p.G + g) * static_cast<int64_t>(N) + n;
            if (p.io_dtype == kF32)
                static_cast<unsigned int *>(p.Bbuf)[e] = load_bits<true>(p.B, bo + n * p.Bs[2]);
            else
                static_cast<unsigned short *>(p.Bbuf)[e] =
                    static_cast<unsigned short>(load_bits<false>(p.B, bo + n * p.Bs[2]));
        }
    }
    __syncthreads();

    if (!fold) {
        // B_j . C for every entry and the current token: one warp (or the
        // whole CTA when it is narrower than a warp) per dot.
        constexpr int W = NT < 32 ? NT : 32;
        constexpr unsigned kMask = W == 32 ? 0xffffffffu : (1u << W) - 1u;
        const int warp = tid / W, wl = tid % W;
        for (int j = warp; j <= c; j += NT / W) {
            float acc = 0.f;
            for (int n = wl; n < N; n += W) acc = fmaf(sB[j * N + n], sC[n], acc);
#pragma unroll
            for (int off = W / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kMask, acc, off);
            if (wl == 0) dots[j] = acc;
        }
        __syncthreads();
        // Readout coefficients of each row: walk the entries from the newest
        // (the current token) to the oldest; w = gamma_{j+1:c}, and after the
        // walk w = gamma_{0:c}, the weight of the checkpoint.
        for (int r = tid; r < rows_here; r += NT) {
            float w = 1.f, hist = 0.f;
            for (int j = c; j >= 0; --j) {
                hist = fmaf(w * rowb[j * kTileRows + r], dots[j], hist);
                w *= rowa[j * kTileRows + r];
            }
            rowg[r] = make_float2(w, hist);
        }
    }
    int timed_out = 0;
    if (!pad && !mbar_wait_bounded(bar, 0)) timed_out = 1;
    if (__syncthreads_or(timed_out)) {
        if (tid == 0) flag(p.status, kDevTimeout);
        return;
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
                T::gather(sB + e * N, lane, bv);
                const float a = rowa[e * kTileRows + rq], dx = rowb[e * kTileRows + rq];
#pragma unroll
                for (int i = 0; i < kElemsPerThread; ++i) sv[i] = fmaf(sv[i], a, dx * bv[i]);
            }
            // ... then the current token, whose state y is read from.
            T::gather(sB + c * N, lane, bv);
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
                             ReplaySmem<TS, L>(kMaxReplayLen).bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, int64_t batch, cudaStream_t stream) {
    cudaError_t e = smem_opt_in<TS, L>();
    if (e != cudaSuccess) return e;
    const int64_t units = batch * p.H * p.ptiles;
    ssu_replay_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads,
                               ReplaySmem<TS, L>(p.rlen).bytes, stream>>>(p);
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
