// ssu_onetoken.cu -- one decode token per sequence.
//
// MATE documentation, page "Mamba / SSU": intro paragraph (a one-token kernel
// for the plain decode step), "SSU at a glance" (rows State, B / C, Slot
// semantics).  The update itself is the recurrence of the ReplaySSM article,
// section 三个瓶颈: read the state, decay it, add the rank-1 term, read y out
// of the updated state, write the state back.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows), numbered with
// the dim tile fastest, then the head, then the sequence, so that units next
// to each other in the numbering read neighbouring blocks of a slot.
//
// The kernel is persistent and warp-specialised.  Each CTA (one or two per
// SM) walks the units u = blockIdx.x + k * gridDim.x through a ring of
// kStages shared-memory stages:
//   producer warp  pure data movement, one unit ahead: resolves the unit's
//                  read/destination slots, copies B and C of the unit's group
//                  and the per-row inputs dt, x, z into the stage, and starts
//                  the bulk asynchronous copy (TMA engine) of the unit's state
//                  tile (contiguous in the pool) into the stage; completion
//                  arrives on the stage's "full" mbarrier;
//   consumer warps wait for "full", turn each row's inputs into its scalars
//                  {dA, dt' x, x, silu gate} (one thread per row), update the
//                  tile rows in registers, write y (one store per row) and
//                  the new state back into the stage; one thread then starts
//                  a bulk asynchronous copy of the stage to the destination
//                  slot and, once the previous unit's copy has read its stage
//                  out, releases that stage on its "empty" mbarrier.
// The producer runs up to kStages units ahead, so state reads stay in flight
// while the consumers compute, and the TMA engine moves the state both ways:
// the bytes in flight per SM are set by the ring size, not by registers, by
// store issue or by CTA launch latency.  The path is HBM-bound; every state
// byte is read once and written once.
#include <atomic>

#include "ssu_device.cuh"

namespace ssu {

constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Size of the pieces a state tile is moved in by the TMA engine.
constexpr int kLoadChunk = 32768;
constexpr int kStoreChunk = 32768;

template <typename TS, int L>
struct OnetokenPipe {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kTileBytes = kTileRows * kN * static_cast<int>(sizeof(TS));
    static constexpr int kStageBytes = align_up(kTileBytes + 2 * kN * 4 + kTileRows * 16 + 32, 128);
    // Dynamic shared memory an SM can give its CTAs (228 KB less the 1 KB
    // each CTA reserves, less a margin).  Small (16-bit) stages: three CTAs
    // of four stages, so three consumer groups share the SM; fp32 stages: two
    // CTAs of three.  The launcher reads how many CTAs the device really
    // holds.
    static constexpr int kSmemPerSm = 222 * 1024;
    static constexpr int kCtasPerSm = (kSmemPerSm / 3 - 1024) / kStageBytes >= 4   ? 3
                                      : (kSmemPerSm / 2 - 1024) / kStageBytes >= 3 ? 2
                                                                                   : 1;
    static constexpr int kRingBytes = kSmemPerSm / kCtasPerSm - 1024;
    static constexpr int kStages = (kRingBytes / kStageBytes) < 6 ? (kRingBytes / kStageBytes) : 6;
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kExitOffset = kBarOffset + kStages * 16;
    static constexpr int kBytes = kExitOffset + static_cast<int>(sizeof(RingExit));
    static constexpr int kConsumerWarps = (Tile<TS, L>::kThreads + 31) / 32;
    static constexpr int kProducerWarps = 2;
    static constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
    static_assert(kStages >= 2 && kStages <= kMaxRingStages, "state tile too large for a pipelined ring");
    // A producer waits for stage s to be free by the parity of the "empty"
    // phase it needs.  When it starts unit k it has finished its previous unit
    // k - kProducerWarps, whose wait guaranteed that every unit up to
    // k - kProducerWarps - kStages had been released; the parity test is
    // unambiguous once unit k - 2 kStages is released, hence this bound.
    static_assert(kProducerWarps <= kStages, "more producer warps than stages breaks the parity waits");
};

// Per-stage header written by the producer.
struct UnitHeader {
    int64_t ws;        // destination slot
    int32_t flags;     // kUnit* bits
    float Dh, Ah, bias;  // D[h] (0 without D), A[h], dt_bias[h] (0 without)
    int32_t reserved;
};
enum : int32_t { kUnitValid = 1, kUnitSeeded = 2, kUnitWrite = 4 };

template <typename TS, int L>
struct StageView {
    using PS = OnetokenPipe<TS, L>;
    TS *tile;
    float *B, *C;
    float4 *rowq;
    UnitHeader *hd;
    __device__ __forceinline__ StageView(unsigned char *smem, int s) {
        unsigned char *base = smem + s * PS::kStageBytes;
        tile = reinterpret_cast<TS *>(base);
        B = reinterpret_cast<float *>(base + PS::kTileBytes);
        C = B + PS::kN;
        rowq = reinterpret_cast<float4 *>(C + PS::kN);
        hd = reinterpret_cast<UnitHeader *>(rowq + kTileRows);
    }
};

// Stage one unit (global index u): header, B, C, row inputs, then the tile
// copy (or a plain arrival when there is nothing to copy).  Returns false
// when the CTA stops: a wait gave up or another role did.
template <typename TS, int L>
__device__ __forceinline__ bool produce_unit(const KParams &p, const UnitOperands<TS, L> &op, int k, int64_t u,
                                             unsigned char *smem, uint64_t *full, uint64_t *empty, RingExit *rx,
                                             int lane) {
    using PS = OnetokenPipe<TS, L>;
    constexpr int N = PS::kN;
    constexpr int S = PS::kStages;
    const int s = k % S;
    const int round = k / S;
    if (ring_aborted(rx)) return false;
    if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, p.wait_cycles)) {
        if (lane == 0) {
            flag(p.status, kDevTimeout);
            ring_abort(rx);
        }
        return false;
    }
    // Self-test of the exit path: this unit's stage is never filled, so the
    // consumers' wait for it runs out with no copy pending.
    if (u == p.withhold_unit) return true;
    const StageView<TS, L> st(smem, s);
    int32_t flags = 0;
    if (lane == 0) {
        const int64_t ws = (p.wr.entries != nullptr) ? op.ws : op.rs;
        if (op.entries_ok && slot_ok(p, op.rs) && slot_ok(p, ws)) {
            flags = kUnitValid;
            if (op.rs != p.pad) flags |= kUnitSeeded;
            if (!p.disable && ws != p.pad) flags |= kUnitWrite;
        }
        st.hd->ws = ws;
        st.hd->flags = flags;
        st.hd->Dh = op.Dh;
        st.hd->Ah = op.Ah;
        st.hd->bias = op.bias;
    }
#pragma unroll
    for (int i = 0; i < UnitOperands<TS, L>::kPerB; ++i) {
        const int n = lane + 32 * i;
        if (n < N) {
            st.B[n] = bits_to_float(op.b[i], p.io_dtype);
            st.C[n] = bits_to_float(op.cc[i], p.io_dtype);
        }
    }
#pragma unroll
    for (int i = 0; i < UnitOperands<TS, L>::kPerRow; ++i) {
        const int r = lane + 32 * i;
        if (r < op.c.rows_here)
            st.rowq[r] = make_float4(bits_to_float(op.dt[i], p.dt_dtype), bits_to_float(op.x[i], p.io_dtype),
                                     bits_to_float(op.z[i], p.io_dtype), 0.f);
    }
    flags = __shfl_sync(0xffffffffu, flags, 0);
    if (flags & kUnitSeeded) {
        // The tile is copied as kLoadChunk-byte pieces issued by all lanes;
        // lane 0 registers the total before any piece can complete.
        const uint32_t bytes = static_cast<uint32_t>(op.c.rows_here) * N * sizeof(TS);
        const int64_t rs = __shfl_sync(0xffffffffu, op.rs, 0);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(
            static_cast<const TS *>(p.state) + ((rs * p.H + op.c.h) * static_cast<int64_t>(p.P) + op.c.row0) * N);
        if (lane == 0) mbar_arrive_expect(&full[s], bytes);
        __syncwarp();
        unsigned char *dst = reinterpret_cast<unsigned char *>(st.tile);
        for (uint32_t off = static_cast<uint32_t>(lane) * kLoadChunk; off < bytes; off += 32u * kLoadChunk) {
            const uint32_t n = bytes - off < static_cast<uint32_t>(kLoadChunk) ? bytes - off : kLoadChunk;
            bulk_load(dst + off, src + off, n, &full[s]);
        }
        if (lane == 0) ring_note_fill(rx, s, round);
        if (lane != 0) mbar_arrive(&full[s]);
    } else {
        if (lane == 0) ring_note_fill(rx, s, round);
        mbar_arrive(&full[s]);
    }
    return true;
}

// Producer warp `w` of kProducerWarps stages the CTA's units k = w, w + P,
// w + 2P, ... (P = kProducerWarps), i.e. global units blockIdx.x + k * gridDim.x.
template <typename TS, int L>
__device__ __forceinline__ void onetoken_producer(const KParams &p, int64_t units, unsigned char *smem,
                                                  uint64_t *full, uint64_t *empty, RingExit *rx, int w) {
    constexpr int P = OnetokenPipe<TS, L>::kProducerWarps;
    const int lane = threadIdx.x & 31;
    const int64_t step = static_cast<int64_t>(P) * gridDim.x;
    // Two operand sets used in turn: the next unit's loads are issued before
    // the current unit is staged (no register copies between them).
    UnitOperands<TS, L> a, b;
    int64_t u = blockIdx.x + static_cast<int64_t>(w) * gridDim.x;
    UnitWalker walk(p, u, step);
    if (u < units) a.load(p, walk.coords(p), lane);
    for (int k = w; u < units; k += 2 * P, u += 2 * step) {
        walk.advance(p);
        if (u + step < units) b.load(p, walk.coords(p), lane);
        if (!produce_unit<TS, L>(p, a, k, u, smem, full, empty, rx, lane)) return;
        if (u + step >= units) break;
        walk.advance(p);
        if (u + 2 * step < units) a.load(p, walk.coords(p), lane);
        if (!produce_unit<TS, L>(p, b, k + P, u + step, smem, full, empty, rx, lane)) return;
    }
}

// Returns the ring index of the first unit not consumed.
template <typename TS, int L>
__device__ __forceinline__ int onetoken_consumer(const KParams &p, int64_t units, unsigned char *smem,
                                                 uint64_t *full, uint64_t *empty, RingExit *rx) {
    using T = Tile<TS, L>;
    using PS = OnetokenPipe<TS, L>;
    constexpr int N = PS::kN;
    constexpr int S = PS::kStages;
    constexpr int kConsumers = 32 * PS::kConsumerWarps;
    const int tid = threadIdx.x;
    const bool active = tid < T::kThreads;
    const int lane = tid % L;
    const int slot_row = tid / L;
    int prev_s = -1;
    int k = 0;
    UnitWalker walk(p, blockIdx.x, gridDim.x);
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++k, walk.advance(p)) {
        const int s = k % S;
        const bool ok = mbar_wait_bounded(&full[s], (k / S) & 1, p.wait_cycles);
        if (barrier_or(1, kConsumers, !ok)) {  // a wait gave up: every consumer stops here
            if (tid == 0) {
                flag(p.status, kDevTimeout);
                ring_abort(rx);
                bulk_wait_all();
            }
            return k;
        }
        const StageView<TS, L> st(smem, s);
        const int32_t flags = st.hd->flags;
        const UnitCoords c = walk.coords(p);
        if (flags & kUnitValid) {
            // Row scalars, one thread per row, in place of the row inputs.
            const float Ah = st.hd->Ah, bias = st.hd->bias;
            for (int r = tid; r < c.rows_here; r += kConsumers) {
                const float4 in = st.rowq[r];
                st.rowq[r] = row_scalars(RowInputs{in.x, in.y, in.z}, Ah, bias, p.softplus, p.z != nullptr);
            }
            named_barrier(1, kConsumers);
            if (active) {
                const float Dh = st.hd->Dh;
                float bv[kElemsPerThread], cv[kElemsPerThread];
                T::gather(st.B, lane, bv);
                T::gather(st.C, lane, cv);
#pragma unroll(kOnetokenUnroll)
                for (int j = 0; j < kRowsPerThread; ++j) {
                    const int rr = slot_row + j * kRowSlots;  // row within the tile
                    const bool live = rr < c.rows_here;
                    const float4 q = st.rowq[live ? rr : 0];
                    float sv[kElemsPerThread];
                    if ((flags & kUnitSeeded) && live) {
                        T::load_row_smem(st.tile + rr * N, lane, sv);
                    } else {
#pragma unroll
                        for (int i = 0; i < kElemsPerThread; ++i) sv[i] = 0.f;
                    }
                    const float sum = row_sum<L>(update_elems(sv, bv, cv, q.x, q.y));
                    if (live) {
                        if (lane == 0)
                            store_small(p.y, c.b * p.ys[0] + c.h * p.ys[1] + (c.row0 + rr) * p.ys[2], p.io_dtype,
                                        output(sum, Dh, q.z, q.w));
                        // The new state goes back into the stage; the TMA
                        // engine writes the whole tile to its destination.
                        T::store_row_smem(st.tile + rr * N, lane, sv);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        named_barrier(1, kConsumers);
        if (tid == 0) {
            if ((flags & kUnitValid) && (flags & kUnitWrite)) {
                unsigned char *dst = reinterpret_cast<unsigned char *>(
                    static_cast<TS *>(p.state) + ((st.hd->ws * p.H + c.h) * static_cast<int64_t>(p.P) + c.row0) * N);
                const unsigned char *src = reinterpret_cast<const unsigned char *>(st.tile);
                const uint32_t bytes = static_cast<uint32_t>(c.rows_here) * N * sizeof(TS);
                for (uint32_t off = 0; off < bytes; off += kStoreChunk)
                    bulk_store(dst + off, src + off, bytes - off < static_cast<uint32_t>(kStoreChunk) ? bytes - off
                                                                                                    : kStoreChunk);
            }
            bulk_commit();
            // The previous unit's tile has been read out by its store: its
            // stage may be refilled.
            if (prev_s >= 0) {
                bulk_wait_read<1>();
                mbar_arrive(&empty[prev_s]);
            }
        }
        prev_s = s;
    }
    if (tid == 0) bulk_wait_all();
    return k;
}

// Register budget of the kernel (the min-CTAs launch bound): for 16-bit pools
// the CTAs per SM the ring allows (three); for fp32 pools the budget of up to
// four CTAs but never under 80 registers a thread, which measured faster than
// the larger allocation two CTAs would permit.
template <typename TS, int L>
constexpr int onetoken_min_ctas() {
    constexpr int threads = OnetokenPipe<TS, L>::kThreads;
    constexpr int by_regs = 65536 / (threads * 80);
    return sizeof(TS) != 4 ? OnetokenPipe<TS, L>::kCtasPerSm : (by_regs < 1 ? 1 : (by_regs > 4 ? 4 : by_regs));
}

template <typename TS, int L>
__global__ void __launch_bounds__(OnetokenPipe<TS, L>::kThreads, (onetoken_min_ctas<TS, L>()))
    ssu_onetoken_kernel(const KParams p, int64_t units) {
    using PS = OnetokenPipe<TS, L>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + PS::kBarOffset);
    uint64_t *empty = full + PS::kStages;
    RingExit *rx = reinterpret_cast<RingExit *>(smem + PS::kExitOffset);
    if (threadIdx.x == 0) {
        for (int s = 0; s < PS::kStages; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], 1);
        }
        ring_init(rx);
    }
    __syncthreads();
    const int warp = threadIdx.x / 32;
    int consumed = 0;
    if (warp >= PS::kConsumerWarps)
        onetoken_producer<TS, L>(p, units, smem, full, empty, rx, warp - PS::kConsumerWarps);
    else
        consumed = onetoken_consumer<TS, L>(p, units, smem, full, empty, rx);
    __syncthreads();
    if (threadIdx.x == 0) ring_drain(rx, full, PS::kStages, consumed, p.wait_cycles, p.status);
}

// Number of SMs of the current device (cached per device).
static int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The ring needs more than the 48 KiB default of dynamic shared memory: opt
// in once per device, then read how many CTAs of the kernel an SM of this
// device holds (cached per device).
template <typename TS, int L>
static cudaError_t resident_ctas(int *ctas) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        using PS = OnetokenPipe<TS, L>;
        e = cudaFuncSetAttribute(ssu_onetoken_kernel<TS, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, PS::kBytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ssu_onetoken_kernel<TS, L>, PS::kThreads, PS::kBytes);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    *ctas = n;
    return cudaSuccess;
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, int64_t batch, cudaStream_t stream) {
    using PS = OnetokenPipe<TS, L>;
    int per_sm = 0;
    cudaError_t e = resident_ctas<TS, L>(&per_sm);
    if (e != cudaSuccess) return e;
    const int64_t units = batch * p.H * p.ptiles;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t slots_on_gpu = static_cast<int64_t>(sms) * per_sm;
    const int64_t grid = units < slots_on_gpu ? units : slots_on_gpu;
    ssu_onetoken_kernel<TS, L><<<static_cast<unsigned>(grid), PS::kThreads, PS::kBytes, stream>>>(p, units);
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
    if (e != cudaSuccess) return e;
    if (sm_count() <= 0) return cudaErrorInvalidDevice;
    int per_sm = 0;
    return resident_ctas<TS, L>(&per_sm);
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
