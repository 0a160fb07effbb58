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
// Work unit: (sequence b, head h, tile of kTileRows dim rows).  The unit's
// state tile stays in registers (fp32) across the sequence's tokens; it is
// read from HBM once and written once per token.  B and C of each token are
// staged in shared memory, double-buffered so that one barrier per token
// suffices.
#include "ssu_device.cuh"

namespace ssu {

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads)
    ssu_packed_kernel(const KParams p) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    __shared__ __align__(16) float sB[2][N];
    __shared__ __align__(16) float sC[2][N];

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
        flag(p.status, 0x4);
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
    const int64_t head_rows = static_cast<int64_t>(h) * p.P;

    float s[kRowsPerThread][kElemsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int pr = ptile * kTileRows + slot_row + j * kRowSlots;
        const TS *row = nullptr;
        if (pr < p.P && rs != p.pad)
            row = static_cast<const TS *>(p.state) + ((rs * p.H) * p.P + head_rows + pr) * N;
        T::load_row(row, lane, s[j]);
    }

    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    stage_bc<N, NT>(p, start, g, sB[0], sC[0]);
    __syncthreads();

    for (int64_t t = 0; t < len; ++t) {
        const int64_t r = start + t;
        const int buf = static_cast<int>(t & 1);
        // Prefetch the next token's B and C into the other buffer; its last
        // readers finished before the barrier that ended the previous token.
        if (t + 1 < len) stage_bc<N, NT>(p, r + 1, g, sB[buf ^ 1], sC[buf ^ 1]);

        int64_t ws;
        table_slot(p, wt, b, t, start, b, &ws);
        const bool write_state = !p.disable && ws != p.pad;

        float bv[kElemsPerThread], cv[kElemsPerThread];
        T::gather(sB[buf], lane, bv);
        T::gather(sC[buf], lane, cv);
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) {
            const int pr = ptile * kTileRows + slot_row + j * kRowSlots;
            const RowScalars q = row_scalars(p, r, h, pr < p.P ? pr : 0, Ah, bias);
            const float part = update_elems(s[j], bv, cv, q.dA, q.dtx);
            const float sum = row_sum<L>(part);
            if (pr < p.P) {
                if (lane == 0) {
                    const float y = output(sum, Dh, q.x, p.z != nullptr, q.z);
                    store_small(p.y, r * p.ys[0] + h * p.ys[1] + pr * p.ys[2], p.io_dtype, y);
                }
                if (write_state)
                    T::store_row(static_cast<TS *>(p.state) + ((ws * p.H) * p.P + head_rows + pr) * N,
                                 lane, s[j]);
            }
        }
        __syncthreads();
    }
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, cudaStream_t stream) {
    const int64_t units = p.nseq * p.H * p.ptiles;
    ssu_packed_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads, 0, stream>>>(p);
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

template <typename TS>
static cudaError_t attrs_lanes(int lanes) {
    cudaFuncAttributes a;
    switch (lanes) {
    case 1: return cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, 1>);
    case 2: return cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, 2>);
    case 4: return cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, 4>);
    case 8: return cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, 8>);
    case 16: return cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, 16>);
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
