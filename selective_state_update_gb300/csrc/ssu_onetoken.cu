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
// written once.  The tile (contiguous in the pool) arrives in shared memory
// by one bulk asynchronous copy (TMA engine, mbarrier completion), so the
// bytes in flight per SM are bounded by shared memory, not by registers;
// meanwhile the CTA stages B and C of the unit's group in shared memory and
// the per-row scalars in registers.  Results leave with 16-byte streaming
// stores; y is reduced over dstate with shuffles.
#include "ssu_device.cuh"

namespace ssu {

// Dynamic shared memory of a CTA: the state tile, B and C as fp32, the mbarrier.
template <typename TS, int L>
struct OnetokenSmem {
    static constexpr int kTileBytes = kTileRows * Tile<TS, L>::kN * static_cast<int>(sizeof(TS));
    static constexpr int kBytes = kTileBytes + 2 * Tile<TS, L>::kN * 4 + 16;
};

template <typename TS, int L>
__global__ void __launch_bounds__(Tile<TS, L>::kThreads)
    ssu_onetoken_kernel(const KParams p) {
    using T = Tile<TS, L>;
    constexpr int N = T::kN;
    constexpr int NT = T::kThreads;
    extern __shared__ __align__(128) unsigned char smem[];
    TS *tile = reinterpret_cast<TS *>(smem);
    float *sB = reinterpret_cast<float *>(smem + OnetokenSmem<TS, L>::kTileBytes);
    float *sC = sB + N;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sC + N);

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
    const int row0 = ptile * kTileRows;
    const int rows_here = min(kTileRows, p.P - row0);
    const int64_t head_row0 = (static_cast<int64_t>(h)) * p.P + row0;
    const bool seeded = rs != p.pad;

    // One thread starts the bulk copy of the tile (rows_here contiguous rows);
    // the others stage B, C and the per-row scalars meanwhile.
    if (tid == 0 && seeded) {
        const uint32_t bytes = static_cast<uint32_t>(rows_here) * N * sizeof(TS);
        mbar_init(bar, 1);
        mbar_arrive_expect(bar, bytes);
        bulk_load(tile, static_cast<const TS *>(p.state) + (rs * p.H * p.P + head_row0) * N, bytes, bar);
    }
    stage_bc<N, NT>(p, b, g, sB, sC);
    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
    RowScalars q[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int pr = row0 + slot_row + j * kRowSlots;
        q[j] = row_scalars(p, b, h, pr < p.P ? pr : 0, Ah, bias);
    }
    __syncthreads();
    float bv[kElemsPerThread], cv[kElemsPerThread];
    T::gather(sB, lane, bv);
    T::gather(sC, lane, cv);
    if (seeded && !mbar_wait_bounded(bar, 0)) {
        flag(p.status, kDevTimeout);
        return;
    }

    const bool write_state = !p.disable && ws != p.pad;
    TS *dst = static_cast<TS *>(p.state) + (ws * p.H * p.P + head_row0) * N;
#pragma unroll(kOnetokenUnroll)
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = slot_row + j * kRowSlots;  // row within the tile
        float s[kElemsPerThread];
        if (seeded && r < rows_here) {
            T::load_row_smem(tile + r * N, lane, s);
        } else {
#pragma unroll
            for (int i = 0; i < kElemsPerThread; ++i) s[i] = 0.f;
        }
        const float part = update_elems(s, bv, cv, q[j].dA, q[j].dtx);
        const float sum = row_sum<L>(part);
        if (r < rows_here) {
            if (lane == 0) {
                const float y = output(sum, Dh, q[j].x, p.z != nullptr, q[j].z);
                store_small(p.y, b * p.ys[0] + h * p.ys[1] + (row0 + r) * p.ys[2], p.io_dtype, y);
            }
            if (write_state) T::store_row(dst + r * N, lane, s);
        }
    }
}

// Dynamic shared memory above the 48 KiB default needs an opt-in per kernel.
template <typename TS, int L>
static cudaError_t set_smem_attr() {
    constexpr int bytes = OnetokenSmem<TS, L>::kBytes;
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(ssu_onetoken_kernel<TS, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, int64_t batch, cudaStream_t stream) {
    cudaError_t e = set_smem_attr<TS, L>();
    if (e != cudaSuccess) return e;
    const int64_t units = batch * p.H * p.ptiles;
    ssu_onetoken_kernel<TS, L><<<static_cast<unsigned>(units), Tile<TS, L>::kThreads,
                                 OnetokenSmem<TS, L>::kBytes, stream>>>(p);
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

template <typename TS, int L>
static cudaError_t attrs_t() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, ssu_onetoken_kernel<TS, L>);
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

cudaError_t prewarm_onetoken(int state_dtype, int lanes) {
    switch (state_dtype) {
    case kF32: return attrs_lanes<float>(lanes);
    case kF16: return attrs_lanes<__half>(lanes);
    case kBF16: return attrs_lanes<__nv_bfloat16>(lanes);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
