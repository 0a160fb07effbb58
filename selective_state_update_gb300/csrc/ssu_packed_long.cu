// ssu_packed_long.cu -- packed decode for calls whose sequences are long
// (on average kLongRowsPerSeq tokens or more; ssu_packed.cu takes the rest).
//
// MATE documentation, page "Mamba / SSU", "SSU at a glance", rows Sequence
// layout, Slot semantics and Variable-length and MTP decode: cu_seqlens splits
// the packed rows between sequences; the read slot is seeded at
// max(num_accepted - 1, 0); every token publishes its state to its own
// destination entry (or its own read-table entry without a destination
// table); pad destinations are never written; empty sequences are skipped.
// Section Graph capture: one launch, no host/device scalar copies.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows), one CTA each;
// small CTAs, many resident per SM, so that the stores of many units are in
// flight at once and the block scheduler balances the units' lengths.
// The seed tile arrives in shared memory by one bulk asynchronous copy (TMA
// engine, mbarrier completion); the unit's state then stays in shared memory
// as fp32 across the sequence's tokens (each thread only ever touches its own
// elements), so it is read from HBM once and written once per token, with
// 16-byte streaming stores.  Each token's B, C and per-row scalars {dA,
// dt' x, x, gate} are loaded two tokens ahead and staged in shared memory
// (double-buffered, one barrier per token); every row's scalars are computed
// once, by one thread.
#include "ssu_device.cuh"

namespace ssu {

namespace {

template <typename TS, int L>
struct PackedSmem {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kCarryBytes = kTileRows * kN * 4;
    static constexpr int kSeedBytes = sizeof(TS) == 4 ? 0 : kTileRows * kN * static_cast<int>(sizeof(TS));
    static constexpr int kBCOffset = kCarryBytes + kSeedBytes;             // B[2][N], C[2][N]
    static constexpr int kRowQOffset = kBCOffset + 4 * kN * 4;             // float4 [2][kTileRows]
    static constexpr int kBarOffset = kRowQOffset + 2 * kTileRows * 16;
    static constexpr int kBytes = kBarOffset + 16;
};

// The fp32 carry uses the element order of Tile<TS, L> (16-byte chunks of
// kVec state elements), stored as kVec floats per chunk.
template <typename TS, int L>
__device__ __forceinline__ void carry_load(const float *row, int lane, float *s) {
    constexpr int kVec = Tile<TS, L>::kVec;
#pragma unroll
    for (int k = 0; k < Tile<TS, L>::kChunks; ++k)
#pragma unroll
        for (int q = 0; q < kVec / 4; ++q) {
            const float4 f = *reinterpret_cast<const float4 *>(row + (lane + L * k) * kVec + 4 * q);
            s[k * kVec + 4 * q + 0] = f.x;
            s[k * kVec + 4 * q + 1] = f.y;
            s[k * kVec + 4 * q + 2] = f.z;
            s[k * kVec + 4 * q + 3] = f.w;
        }
}

template <typename TS, int L>
__device__ __forceinline__ void carry_store(float *row, int lane, const float *s) {
    constexpr int kVec = Tile<TS, L>::kVec;
#pragma unroll
    for (int k = 0; k < Tile<TS, L>::kChunks; ++k)
#pragma unroll
        for (int q = 0; q < kVec / 4; ++q)
            *reinterpret_cast<float4 *>(row + (lane + L * k) * kVec + 4 * q) =
                make_float4(s[k * kVec + 4 * q + 0], s[k * kVec + 4 * q + 1], s[k * kVec + 4 * q + 2],
                            s[k * kVec + 4 * q + 3]);
}

// One token's small operands, loaded into registers ahead of time (as raw
// bits, back to back, so that they are in flight together) and staged in
// shared memory afterwards, converted to fp32 and turned into row scalars.
template <int N, int NT>
struct TokenOperands {
    static constexpr int kPerB = (N + NT - 1) / NT;
    static constexpr int kPerRow = (kTileRows + NT - 1) / NT;
    uint32_t b[kPerB], c[kPerB];
    uint32_t dt[kPerRow], x[kPerRow], z[kPerRow];

    template <bool WIO, bool WDT>
    __device__ __forceinline__ void load_t(const KParams &p, int64_t r, int g, int h, int row0, int rows_here) {
        const int64_t bo = r * p.Bs[0] + g * p.Bs[1];
        const int64_t co = r * p.Cs[0] + g * p.Cs[1];
#pragma unroll
        for (int i = 0; i < kPerB; ++i) {
            const int n = threadIdx.x + i * NT;
            if (n < N) {
                b[i] = load_bits<WIO>(p.B, bo + n * p.Bs[2]);
                c[i] = load_bits<WIO>(p.C, co + n * p.Cs[2]);
            }
        }
#pragma unroll
        for (int i = 0; i < kPerRow; ++i) {
            const int rr = threadIdx.x + i * NT;
            if (rr < rows_here) {
                const int pr = row0 + rr;
                dt[i] = load_bits<WDT>(p.dt, r * p.dts[0] + h * p.dts[1] + pr * p.dts[2]);
                x[i] = load_bits<WIO>(p.x, r * p.xs[0] + h * p.xs[1] + pr * p.xs[2]);
                z[i] = p.z ? load_bits<WIO>(p.z, r * p.zs[0] + h * p.zs[1] + pr * p.zs[2]) : 0u;
            }
        }
    }

    __device__ __forceinline__ void load(const KParams &p, int64_t r, int g, int h, int row0, int rows_here) {
        const bool wio = p.io_dtype == kF32, wdt = p.dt_dtype == kF32;
        if (wio) {
            if (wdt) load_t<true, true>(p, r, g, h, row0, rows_here);
            else load_t<true, false>(p, r, g, h, row0, rows_here);
        } else {
            if (wdt) load_t<false, true>(p, r, g, h, row0, rows_here);
            else load_t<false, false>(p, r, g, h, row0, rows_here);
        }
    }

    __device__ __forceinline__ void stage(const KParams &p, float *sB, float *sC, float4 *rowq, int rows_here,
                                          float Ah, float bias) const {
#pragma unroll
        for (int i = 0; i < kPerB; ++i) {
            const int n = threadIdx.x + i * NT;
            if (n < N) {
                sB[n] = bits_to_float(b[i], p.io_dtype);
                sC[n] = bits_to_float(c[i], p.io_dtype);
            }
        }
#pragma unroll
        for (int i = 0; i < kPerRow; ++i) {
            const int rr = threadIdx.x + i * NT;
            if (rr < rows_here) {
                const RowInputs in{bits_to_float(dt[i], p.dt_dtype), bits_to_float(x[i], p.io_dtype),
                                   bits_to_float(z[i], p.io_dtype)};
                rowq[rr] = row_scalars(in, Ah, bias, p.softplus, p.z != nullptr);
            }
        }
    }
};

// One token applied to this thread's rows.  FIRST: the state comes from the
// seed tile (state dtype; zeros when the seed is the pad slot); later tokens
// read the fp32 carry.  The carry is written back (fp32, never re-rounded) and
// the rounded copy is published to the destination rows when `dst` is set.
template <typename TS, int L, bool FIRST>
__device__ __forceinline__ void token_rows(const KParams &p, int64_t r, int h, int row0, int rows_here,
                                           int slot_row, int lane, const TS *seed, bool seeded, float *carry,
                                           TS *dst, const float *bv, const float *cv, const float4 *rowq,
                                           float Dh) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
#pragma unroll 2
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int rr = slot_row + j * kRowSlots;  // row within the tile
        const bool live = rr < rows_here;
        const float4 q = rowq[live ? rr : 0];
        float s[kElemsPerThread];
        if (FIRST) {
            if (seeded && live) {
                T::load_row_smem(seed + rr * N, lane, s);
            } else {
#pragma unroll
                for (int i = 0; i < kElemsPerThread; ++i) s[i] = 0.f;
            }
        } else {
            carry_load<TS, L>(carry + rr * N, lane, s);
        }
        const float sum = row_sum<L>(update_elems(s, bv, cv, q.x, q.y));
        if (live) {
            if (lane == 0)
                store_small(p.y, r * p.ys[0] + h * p.ys[1] + (row0 + rr) * p.ys[2], p.io_dtype,
                            output(sum, Dh, q.z, q.w));
            carry_store<TS, L>(carry + rr * N, lane, s);
            if (dst != nullptr) T::store_row(dst + rr * N, lane, s);
        }
    }
}

// CTAs per SM that the shared memory of one CTA allows (228 KB per SM, 1 KB
// of it reserved per CTA), at most 8: the register allocation is held to
// what that many resident CTAs can share.
template <typename TS, int L>
constexpr int packed_min_ctas() {
    constexpr int fit = (228 * 1024) / (PackedSmem<TS, L>::kBytes + 1024);
    return fit < 1 ? 1 : (fit > 8 ? 8 : fit);
}

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads, (packed_min_ctas<TS, L>()))
    ssu_packed_long_kernel(const KParams p) {
    using T = Tile<TS, L>;
    using SM = PackedSmem<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    float *carry = reinterpret_cast<float *>(smem);
    TS *seed = sizeof(TS) == 4 ? reinterpret_cast<TS *>(smem) : reinterpret_cast<TS *>(smem + SM::kCarryBytes);
    float *sB = reinterpret_cast<float *>(smem + SM::kBCOffset);  // [2][N]
    float *sC = sB + 2 * N;                                        // [2][N]
    float4 *rowq = reinterpret_cast<float4 *>(smem + SM::kRowQOffset);  // [2][kTileRows]
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + SM::kBarOffset);

    const int64_t unit = blockIdx.x;
    const int ptile = static_cast<int>(unit % p.ptiles);
    const int64_t bh = unit / p.ptiles;
    const int h = static_cast<int>(bh % p.H);
    const int64_t b = bh / p.H;
    const int g = h / p.heads_per_group;

    // Rows of the sequence (uniform over the CTA).
    int64_t start, end;
    if (p.cu != nullptr) {
        start = load_index(p.cu, b, p.meta_is_i64);
        end = load_index(p.cu, b + 1, p.meta_is_i64);
    } else {
        start = b * p.steps;
        end = start + p.steps;
    }
    if (start < 0 || end < start || end > p.rows) {
        flag(p.status, kDevBadSeqlen);
        return;
    }
    const int64_t len = end - start;
    if (len == 0) return;

    // Read slot at step max(num_accepted - 1, 0).
    int64_t t_seed = 0;
    if (p.acc != nullptr) {
        t_seed = load_index(p.acc, b, p.meta_is_i64) - 1;
        if (t_seed < 0) t_seed = 0;
    }
    // Per-row tables hold one entry per packed row: the seed step must be
    // one of the sequence's own rows.
    if (p.rd.entries != nullptr && p.rd.per_row && t_seed >= len) {
        if (threadIdx.x == 0) flag(p.status, kDevBadEntry);
        return;
    }
    int64_t rs;
    if (!table_slot(p, p.rd, b, t_seed, start, b, &rs) || !slot_ok(p, rs)) return;
    // Every destination of the sequence is checked before anything is written.
    const SlotTab &wt = (p.wr.entries != nullptr) ? p.wr : p.rd;
    int bad = 0;
    for (int64_t t = threadIdx.x; t < len; t += NT) {
        int64_t w;
        if (!table_slot(p, wt, b, t, start, b, &w) || !slot_ok(p, w)) bad = 1;
    }
    if (__syncthreads_or(bad)) return;

    const int tid = threadIdx.x;
    const int lane = tid % L;
    const int slot_row = tid / L;
    const int row0 = ptile * kTileRows;
    const int rows_here = min(kTileRows, p.P - row0);
    const int64_t head_row0 = static_cast<int64_t>(h) * p.P + row0;
    const bool seeded = rs != p.pad;

    if (tid == 0 && seeded) {
        const uint32_t bytes = static_cast<uint32_t>(rows_here) * N * sizeof(TS);
        mbar_init(bar, 1);
        mbar_arrive_expect(bar, bytes);
        bulk_load(seed, static_cast<const TS *>(p.state) + (rs * p.H * p.P + head_row0) * N, bytes, bar);
    }
    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    // Two operand sets in turn: the operands of token t + 2 are loaded while
    // token t computes and staged at the end of token t + 1, so their loads
    // have two tokens' time to arrive.
    TokenOperands<N, NT> ops0, ops1;
    ops0.load(p, start, g, h, row0, rows_here);
    ops0.stage(p, sB, sC, rowq, rows_here, Ah, bias);
    if (len > 1) ops1.load(p, start + 1, g, h, row0, rows_here);
    __syncthreads();
    int timed_out = 0;
    if (seeded && !mbar_wait_bounded(bar, 0, p.wait_cycles)) timed_out = 1;
    if (__syncthreads_or(timed_out)) {
        // The seed copy may still be in flight: thread 0 keeps the CTA alive
        // for one more bounded wait so that it does not retire under it.
        if (tid == 0) {
            flag(p.status, kDevTimeout);
            mbar_wait_bounded(bar, 0, p.wait_cycles);
        }
        return;
    }

    // Token t reads staging buffers t & 1; the staging of token t + 1 goes to
    // the other buffers, last read before the previous barrier.
    auto token = [&](int64_t t, int buf) {
        const int64_t r = start + t;
        int64_t ws;
        table_slot(p, wt, b, t, start, b, &ws);
        TS *dst = (!p.disable && ws != p.pad)
                      ? static_cast<TS *>(p.state) + (ws * p.H * p.P + head_row0) * N
                      : nullptr;
        float bv[kElemsPerThread], cv[kElemsPerThread];
        T::gather(sB + buf * N, lane, bv);
        T::gather(sC + buf * N, lane, cv);
        if (t == 0)
            token_rows<TS, L, true>(p, r, h, row0, rows_here, slot_row, lane, seed, seeded, carry, dst, bv, cv,
                                    rowq + buf * kTileRows, Dh);
        else
            token_rows<TS, L, false>(p, r, h, row0, rows_here, slot_row, lane, seed, seeded, carry, dst, bv, cv,
                                     rowq + buf * kTileRows, Dh);
    };
    for (int64_t t = 0; t < len; t += 2) {
        if (t + 2 < len) ops0.load(p, start + t + 2, g, h, row0, rows_here);
        token(t, 0);
        if (t + 1 < len) ops1.stage(p, sB + N, sC + N, rowq + kTileRows, rows_here, Ah, bias);
        __syncthreads();
        if (t + 1 >= len) break;
        if (t + 3 < len) ops1.load(p, start + t + 3, g, h, row0, rows_here);
        token(t + 1, 1);
        if (t + 2 < len) ops0.stage(p, sB, sC, rowq, rows_here, Ah, bias);
        __syncthreads();
    }
}

}  // namespace

template <typename TS, int L>
static cudaError_t set_smem_attr() {
    constexpr int bytes = PackedSmem<TS, L>::kBytes;
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(ssu_packed_long_kernel<TS, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, cudaStream_t stream) {
    cudaError_t e = set_smem_attr<TS, L>();
    if (e != cudaSuccess) return e;
    const int64_t units = p.nseq * p.H * p.ptiles;
    ssu_packed_long_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads, PackedSmem<TS, L>::kBytes,
                               stream>>>(p);
    return cudaGetLastError();
}

template <typename TS>
static cudaError_t launch_lanes(int lanes, const KParams &p, cudaStream_t stream) {
    switch (lanes) {
    case 1: return launch_t<TS, 1>(p, stream);
    case 2: return launch_t<TS, 2>(p, stream);
    case 4: return launch_t<TS, 4>(p, stream);
    case 8: return launch_t<TS, 8>(p, stream);
    case 16: return launch_t<TS, 16>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_packed_long(int state_dtype, int lanes, const KParams &p, cudaStream_t stream) {
    switch (state_dtype) {
    case kF32: return launch_lanes<float>(lanes, p, stream);
    case kF16: return launch_lanes<__half>(lanes, p, stream);
    case kBF16: return launch_lanes<__nv_bfloat16>(lanes, p, stream);
    }
    return cudaErrorInvalidValue;
}

template <typename TS, int L>
static cudaError_t attrs_t() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, ssu_packed_long_kernel<TS, L>);
    return e != cudaSuccess ? e : set_smem_attr<TS, L>();
}

template <typename TS>
static cudaError_t attrs_lanes(int lanes) {
    switch (lanes) {
    case 1: return attrs_t<TS, 1>();
    case 2: return attrs_t<TS, 2>();
    case 4: return attrs_t<TS, 4>();
    case 8: return attrs_t<TS, 8>();
    case 16: return attrs_t<TS, 16>();
    }
    return cudaErrorInvalidValue;
}

cudaError_t prewarm_packed_long(int state_dtype, int lanes) {
    switch (state_dtype) {
    case kF32: return attrs_lanes<float>(lanes);
    case kF16: return attrs_lanes<__half>(lanes);
    case kBF16: return attrs_lanes<__nv_bfloat16>(lanes);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
