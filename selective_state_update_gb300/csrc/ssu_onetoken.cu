// ssu_onetoken.cu -- one decode token per sequence.
//
// MATE documentation, page "Mamba / SSU": intro paragraph (a one-token kernel
// for the plain decode step), "SSU at a glance" (rows State, B / C, Slot
// semantics).  The update itself is the recurrence of the ReplaySSM article,
// section 三个瓶颈: read the state, decay it, add the rank-1 term, read y out
// of the updated state, write the state back.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows); one CTA each,
// ptile fastest so that neighbouring CTAs stream neighbouring bytes of the
// same slot.  The path is HBM-bound: every state byte is read once and
// written once with 16-byte streaming accesses; B and C of the unit's group
// are staged once in shared memory; y is reduced over dstate with shuffles.
#include "ssu_device.cuh"

namespace ssu {

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads)
    ssu_onetoken_kernel(const KParams p) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    __shared__ __align__(16) float sB[N];
    __shared__ __align__(16) float sC[N];

    const int64_t unit = blockIdx.x;
    const int ptile = static_cast<int>(unit % p.ptiles);
    const int64_t bh = unit / p.ptiles;
    const int h = static_cast<int>(bh % p.H);
    const int64_t b = bh / p.H;
    const int g = h / p.heads_per_group;

    // Slots (uniform over the CTA).  One token: entry (b, 0), row_start b.
    int64_t rs, ws;
    if (!table_slot(p, p.rd, b, 0, b, b, &rs)) return;
    if (p.wr.entries != nullptr) {
        if (!table_slot(p, p.wr, b, 0, b, b, &ws)) return;
    } else {
        ws = rs;
    }
    if (!slot_ok(p, rs) || !slot_ok(p, ws)) return;

    const int tid = threadIdx.x;
    const int lane = tid % L;
    const int slot_row = tid / L;
    const int64_t head_rows = (static_cast<int64_t>(h)) * p.P;

    // Issue the state loads of all this thread's rows first.
    float s[kRowsPerThread][kElemsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int pr = ptile * kTileRows + slot_row + j * kRowSlots;
        const TS *row = nullptr;
        if (pr < p.P && rs != p.pad)
            row = static_cast<const TS *>(p.state) + ((rs * p.H) * p.P + head_rows + pr) * N;
        T::load_row(row, lane, s[j]);
    }

    stage_bc<N, NT>(p, b, g, sB, sC);
    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    RowScalars q[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int pr = ptile * kTileRows + slot_row + j * kRowSlots;
        q[j] = row_scalars(p, b, h, pr < p.P ? pr : 0, Ah, bias);
    }
    __syncthreads();
    float bv[kElemsPerThread], cv[kElemsPerThread];
    T::gather(sB, lane, bv);
    T::gather(sC, lane, cv);

    const bool write_state = !p.disable && ws != p.pad;
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int pr = ptile * kTileRows + slot_row + j * kRowSlots;
        const float part = update_elems(s[j], bv, cv, q[j].dA, q[j].dtx);
        const float sum = row_sum<L>(part);
        if (pr < p.P) {
            if (lane == 0) {
                const float y = output(sum, Dh, q[j].x, p.z != nullptr, q[j].z);
                store_small(p.y, b * p.ys[0] + h * p.ys[1] + pr * p.ys[2], p.io_dtype, y);
            }
            if (write_state)
                T::store_row(static_cast<TS *>(p.state) + ((ws * p.H) * p.P + head_rows + pr) * N,
                             lane, s[j]);
        }
    }
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, int64_t batch, cudaStream_t stream) {
    const int64_t units = batch * p.H * p.ptiles;
    ssu_onetoken_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads, 0, stream>>>(p);
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

cudaError_t launch_onetoken(int state_dtype, int lanes, const KParams &p, int64_t batch,
                            cudaStream_t stream) {
    switch (state_dtype) {
    case kF32: return launch_lanes<float>(lanes, p, batch, stream);
    case kF16: return launch_lanes<__half>(lanes, p, batch, stream);
    case kBF16: return launch_lanes<__nv_bfloat16>(lanes, p, batch, stream);
    }
    return cudaErrorInvalidValue;
}

template <typename TS>
static cudaError_t attrs_lanes(int lanes) {
    cudaFuncAttributes a;
    switch (lanes) {
    case 1: return cudaFuncGetAttributes(&a, ssu_onetoken_kernel<TS, 1>);
    case 2: return cudaFuncGetAttributes(&a, ssu_onetoken_kernel<TS, 2>);
    case 4: return cudaFuncGetAttributes(&a, ssu_onetoken_kernel<TS, 4>);
    case 8: return cudaFuncGetAttributes(&a, ssu_onetoken_kernel<TS, 8>);
    case 16: return cudaFuncGetAttributes(&a, ssu_onetoken_kernel<TS, 16>);
    }
    return cudaErrorInvalidValue;
}

cudaError_t prewarm_onetoken(int state_dtype, int lanes) {
    switch (state_dtype) {
    case kF32: return attrs_lanes<float>(lanes);
    case kF16: return attrs_lanes<__half>(lanes);
    case kBF16: return attrs_lanes<__nv_bfloat16>(lanes);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
