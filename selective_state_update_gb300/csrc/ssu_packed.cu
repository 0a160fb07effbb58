// ssu_packed.cu -- packed variable-length and multi-token (MTP) decode.
//
// MATE documentation, page "Mamba / SSU", "SSU at a glance", rows Sequence
// layout, Slot semantics and Variable-length and MTP decode: cu_seqlens splits
// the packed rows between sequences; the read slot is seeded at
// max(num_accepted - 1, 0); every token publishes its state to its own
// destination entry (or its own read-table entry without a destination
// table); pad destinations are never written; empty sequences are skipped.
// Section Graph capture: one launch, no host/device scalar copies.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows).  The seed tile
// arrives in shared memory by one bulk asynchronous copy (TMA engine); the
// unit's state then stays in shared memory as fp32 across the sequence's
// tokens (each thread only ever touches its own elements), so it is read
// from HBM once and written once per token, with 16-byte streaming stores.
// B and C of each token are staged in shared memory, double-buffered so that
// one barrier per token suffices.
#include "ssu_device.cuh"

namespace ssu {

// Dynamic shared memory of a CTA: the fp32 carried state tile (the seed lands
// in it directly for an fp32 pool), the seed tile for a 16-bit pool, B and C
// double-buffered as fp32, the mbarrier.
template <typename TS, int L>
struct PackedSmem {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kCarryBytes = kTileRows * kN * 4;
    static constexpr int kSeedBytes = sizeof(TS) == 4 ? 0 : kTileRows * kN * static_cast<int>(sizeof(TS));
    static constexpr int kBCOffset = kCarryBytes + kSeedBytes;
    static constexpr int kBytes = kBCOffset + 4 * kN * 4 + 16;
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

// One token applied to this thread's rows.  FIRST: the state comes from the
// seed tile (state dtype; zeros when the seed is the pad slot); later tokens
// read the fp32 carry.  The carry is written back (fp32, never re-rounded) and
// the rounded copy is published to the destination row when `dst` is set.
template <typename TS, int L, bool FIRST>
__device__ __forceinline__ void token_rows(const KParams &p, int64_t r, int h, int row0, int rows_here,
                                           int slot_row, int lane, const TS *seed, bool seeded,
                                           float *carry, TS *dst, const float *bv, const float *cv,
                                           float Ah, float Dh, float bias) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
#pragma unroll(kPackedUnroll)
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int rr = slot_row + j * kRowSlots;  // row within the tile
        const RowScalars q = row_scalars(p, r, h, row0 + (rr < rows_here ? rr : 0), Ah, bias);
        float s[kElemsPerThread];
        if (FIRST) {
            if (seeded && rr < rows_here) {
                T::load_row_smem(seed + rr * N, lane, s);
            } else {
#pragma unroll
                for (int i = 0; i < kElemsPerThread; ++i) s[i] = 0.f;
            }
        } else {
            carry_load<TS, L>(carry + rr * N, lane, s);
        }
        const float part = update_elems(s, bv, cv, q.dA, q.dtx);
        const float sum = row_sum<L>(part);
        if (rr < rows_here) {
            if (lane == 0) {
                const float y = output(sum, Dh, q.x, p.z != nullptr, q.z);
                store_small(p.y, r * p.ys[0] + h * p.ys[1] + (row0 + rr) * p.ys[2], p.io_dtype, y);
            }
            carry_store<TS, L>(carry + rr * N, lane, s);
            if (dst != nullptr) T::store_row(dst + rr * N, lane, s);
        }
    }
}

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads)
    ssu_packed_kernel(const KParams p) {
    using T = Tile<TS, L>;
    using SM = PackedSmem<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    float *carry = reinterpret_cast<float *>(smem);
    TS *seed = sizeof(TS) == 4 ? reinterpret_cast<TS *>(smem) : reinterpret_cast<TS *>(smem + SM::kCarryBytes);
    float *sB = reinterpret_cast<float *>(smem + SM::kBCOffset);  // [2][N]
    float *sC = sB + 2 * N;                                        // [2][N]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sC + 2 * N);

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
    stage_bc<N, NT>(p, start, g, sB, sC);
    __syncthreads();
    int timed_out = 0;
    if (seeded && !mbar_wait_bounded(bar, 0)) timed_out = 1;
    if (__syncthreads_or(timed_out)) {
        if (tid == 0) flag(p.status, kDevTimeout);
        return;
    }

    for (int64_t t = 0; t < len; ++t) {
        const int64_t r = start + t;
        const int buf = static_cast<int>(t & 1);
        // Prefetch the next token's B and C into the other buffer; its last
        // readers finished before the barrier that ended the previous token.
        if (t + 1 < len) stage_bc<N, NT>(p, r + 1, g, sB + (buf ^ 1) * N, sC + (buf ^ 1) * N);

        int64_t ws;
        table_slot(p, wt, b, t, start, b, &ws);
        TS *dst = (!p.disable && ws != p.pad)
                      ? static_cast<TS *>(p.state) + (ws * p.H * p.P + head_row0) * N
                      : nullptr;
        float bv[kElemsPerThread], cv[kElemsPerThread];
        T::gather(sB + buf * N, lane, bv);
        T::gather(sC + buf * N, lane, cv);
        if (t == 0)
            token_rows<TS, L, true>(p, r, h, row0, rows_here, slot_row, lane, seed, seeded, carry, dst, bv,
                                    cv, Ah, Dh, bias);
        else
            token_rows<TS, L, false>(p, r, h, row0, rows_here, slot_row, lane, seed, seeded, carry, dst, bv,
                                     cv, Ah, Dh, bias);
        __syncthreads();
    }
}

template <typename TS, int L>
static cudaError_t set_smem_attr() {
    constexpr int bytes = PackedSmem<TS, L>::kBytes;
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(ssu_packed_kernel<TS, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, cudaStream_t stream) {
    cudaError_t e = set_smem_attr<TS, L>();
    if (e != cudaSuccess) return e;
    const int64_t units = p.nseq * p.H * p.ptiles;
    ssu_packed_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads, PackedSmem<TS, L>::kBytes,
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

cudaError_t launch_packed(int state_dtype, int lanes, const KParams &p, cudaStream_t stream) {
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
    cudaError_t e = cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, L>);
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

cudaError_t prewarm_packed(int state_dtype, int lanes) {
    switch (state_dtype) {
    case kF32: return attrs_lanes<float>(lanes);
    case kF16: return attrs_lanes<__half>(lanes);
    case kBF16: return attrs_lanes<__nv_bfloat16>(lanes);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
