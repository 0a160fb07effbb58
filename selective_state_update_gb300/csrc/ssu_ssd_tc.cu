// ssu_ssd_tc.cu -- the chunk scan of the packed SSD prefill on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// MATE documentation, page "Mamba / SSU", section "SSD packed prefill": the
// C . B^T products and the chunk scan.  For chunk c (tokens t, s < L <= Q),
// head h of group g, with cs the inclusive cumulative sum of a = A dt' over
// the chunk and S_in the state entering the chunk:
//     y_t = exp(cs_t) C_t . S_in + sum_{s<t} (C_t . B_s) exp(cs_t - cs_s) dt'_s x_s
//           + ((C_t . B_t) dt'_t + D) x_t,   gated by silu(z_t).
//
// A persistent grid (one CTA per SM) splits the (chunk, group, head) units
// into equal contiguous ranges; a CTA walks its range one (chunk, group)
// segment at a time.  C . B^T is the same for every head of the group, so
// it is computed once per segment, by tcgen05.mma into
// tensor memory (the row tiles of 128 tokens side by side, causal: tile m
// holds columns s < 128 (m + 1)).  Per head and row tile:
//   Y1 = C . S_in^T         tcgen05.mma, S_in as bf16 high and low parts
//                           (the state pass stores them in the operand layout);
//   W  = (C . B^T) exp(cs_t - cs_s) dt'_s for s < t, formed from tensor
//        memory (tcgen05.ld) 32 columns at a time into one of three
//        shared-memory buffers, in fp16 (11 significant bits; x is staged in
//        fp16 too, exactly for bf16 inputs in fp16's normal range, since both
//        operands of one MMA share a type).  For a block that
//        lies wholly before row t the decay factors through the block's last
//        token r, exp(cs_t - cs_r) exp(cs_r - cs_s), both at most 1 (cs only
//        decreases), the second with dt'_s kept per column for the head (E):
//        two products per weight; the diagonal block takes one exponential
//        per weight, the blocks after it are zero;
//   Y2 += W . X             tcgen05.mma per 32-column block (fp16 operands);
//   y  = exp(cs_t) Y1 + Y2 + ((C_t . B_t) dt'_t + D) x_t   (the diagonal in
//        fp32, from the same tensor-memory row), gated, stored.
// Warp roles: warps 0-7 form the weights and read the results out (warps w
// and w + 4 share tensor-memory lanes 32 (w % 4) ..., i.e. token rows, and
// split each block's columns and each row's outputs); warp 8 owns tensor
// memory and issues every MMA from one thread; warps 9 and 10 stage the next
// head's x rows, entering state and cumulative sums while the current head
// computes (into the shared memory of B once C . B^T is done, where it fits).
// Completion is tracked on mbarriers: tcgen05.commit arrives when an MMA
// group is done; every wait is bounded.
//
// Operand layouts are the canonical ones without swizzle: a matrix is cut
// into core matrices of 8 rows x 16 bytes stored as 128 contiguous bytes; the
// matrix descriptor gives the byte distance between core matrices that are
// neighbours along K (LBO) and along M or N (SBO).
#include <cstdint>

#include "ssu_device.cuh"
#include "ssu_ssd_params.h"

namespace ssu {

namespace {

// ---------------------------------------------------------------------------
// tcgen05 building blocks (inline PTX).
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, no swizzle: start address, LBO, SBO (all
// in 16-byte units), the fixed constant 0b001 at bits 46-48.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Instruction descriptor of kind::f16: A and B both bf16 (bf = 1) or both
// fp16 (bf = 0), fp32 D, dense, M x N; a_mn / b_mn select an MN-major A / B
// (0: K-major).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn, int bf = 1) {
    return (1u << 4) | (static_cast<uint32_t>(bf) << 7) | (static_cast<uint32_t>(bf) << 10) |
           (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] B[smem]; issued by one thread.
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_alloc512(uint32_t *dst_smem) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(dst_smem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc512(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(taddr) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's tensor-memory lane (lanes
// 32 (warp % 4) + lane); warp-collective.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Expect `bytes` more transaction bytes on the current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// 16 bytes global -> shared by cp.async; `valid` false fills zeros.
__device__ __forceinline__ void cp16(void *smem, const void *gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(smem)), "l"(gmem),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
// 2^x by the special-function unit (relative error below 2^-22); x <= 0 here.
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The power of two 2^k that brings a non-negative bound m into [2^13, 2^14)
// (k in [-126, 126]; 1 for m zero or not finite): the scale of an fp16
// operand whose magnitudes are at most m.
__device__ __forceinline__ int fp16_scale_exp(float m) {
    if (!(m > 0.f) || !(m <= 3.0e38f)) return 0;
    const int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xffu) - 126;  // m = f 2^e, f in [0.5, 1)
    const int k = 14 - e;
    return k < -126 ? -126 : (k > 126 ? 126 : k);
}
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }

// ---------------------------------------------------------------------------
// Layout of one CTA (P = 64 dim rows, N = dstate, Q = chunk size).
// ---------------------------------------------------------------------------
constexpr int kTcP = 64;
constexpr int kTcBlock = 32;      // weight columns per block
constexpr int kWBufs = 3;         // weight blocks in flight
constexpr int kEpi = 256;         // weight / readout threads (warps 0-7)
constexpr int kTcThreads = kEpi + 96;  // + warp 8 (MMA) and warps 9, 10 (loads)
constexpr int kTcCols = 512;      // tensor-memory columns

template <int Q, int N>
struct TcLayout {
    // C, B: [Q][N] K-major (K = n): element (t, n) at (t/8)(16N) + (n/8)128 + (t%8)16 + (n%8)2.
    static constexpr int kCBytes = Q * N * 2;
    static constexpr int kBBytes = Q * N * 2;
    // X (fp16): MN-major (N = p, K = s): element (p, s) at (p/8)(16Q) + 16s + (p%8)2.
    static constexpr int kXBytes = Q * kTcP * 2;
    // S_in high then low part, each K-major (N = p, K = n), the state pass's layout.
    static constexpr int kSBytes = 2 * kTcP * N * 2;
    static constexpr int kXSBytes = kXBytes + kSBytes;
    // Weights (fp16), per buffer K-major (M = t, K = s of the block):
    // element (t, sl) at (t/8)(kTcBlock/8)128 + (sl/8)128 + (t%8)16 + (sl%8)2.
    static constexpr int kWBuf = 128 * kTcBlock * 2;
    static constexpr int kWBytes = kWBufs * kWBuf;
    // Per head buffer: cs, dt' (loaded), E, cs log2(e) (formed) -- Q floats
    // each; then 2^-kx (the x scale) and the largest dt', 2 unused.
    static constexpr int kAuxBytes = 4 * Q * 4 + 16;
    static constexpr bool kAlias = kBBytes >= kXSBytes;  // the second head buffer lives in B's place
    static constexpr int kC = 0;
    static constexpr int kB = kC + kCBytes;
    static constexpr int kBuf0 = kB + kBBytes;
    static constexpr int kBuf1 = kAlias ? kB : kBuf0 + kXSBytes;
    static constexpr int kW = (kAlias ? kBuf0 + kXSBytes : kBuf1 + kXSBytes);
    static constexpr int kAux0 = kW + kWBytes;
    static constexpr int kAux1 = kAux0 + kAuxBytes;
    static constexpr int kCbd = kAux1 + kAuxBytes;  // the diagonal C_t . B_t of the rows, by tile parity
    static constexpr int kWmax = kCbd + 2 * 128 * 4; // per segment parity and warp: the largest |C . B^T|
    static constexpr int kBars = kWmax + 2 * 8 * 4;  // 16 mbarriers
    static constexpr int kTaddr = kBars + 16 * 8;
    static constexpr int kBytes = kTaddr + 16;
    // tensor-memory columns: C . B^T of tile 0 at 0, of tile 1 at 128; Y1, Y2
    static constexpr int kNcols0 = Q < 128 ? Q : 128;
    static constexpr int kCB1 = 128;
    static constexpr int kY1 = 384;
    static constexpr int kY2 = 448;
    static_assert(kBytes <= 227 * 1024, "chunk scan layout exceeds shared memory");
    static_assert(Q == 64 || Q == 128 || Q == 256, "chunk size");
    static_assert(N == 64 || N == 128, "dstate");
    static_assert(kY2 + kTcP <= kTcCols, "tensor-memory columns");
};

enum : int { kBarFull0 = 0, kBarFull1, kBarXFree0, kBarXFree1, kBarCB, kBarYFull, kBarYFree, kBarFinal, kBarEpi,
             kBarWFull0, kBarWFree0 = kBarWFull0 + kWBufs };
static_assert(kBarWFree0 + kWBufs <= 16, "barrier slots");

// A barrier of the weight / readout threads whose wait is bounded (a plain
// bar.sync would wait forever for a thread that left after a wait gave up):
// every thread arrives, then waits for the phase; `phase` counts the uses.
__device__ __forceinline__ bool epi_sync(uint64_t *bar, int &phase, long long lim) {
    mbar_arrive(bar);
    const bool ok = mbar_wait_bounded(bar, phase & 1, lim);
    ++phase;
    return ok;
}

__device__ __forceinline__ int64_t tc_ws_unit(const SsdParams &p, int64_t c, int h) {
    return static_cast<int64_t>(h) * p.nchunks + c;
}

// Stage head h's x rows (plain loads by the two loader warps), entering state
// and cumulative sums (bulk copies, their bytes registered on `full` by
// loader thread 0 first) into a head buffer; every loader thread arrives on
// `full` afterwards.
template <int Q, int N>
__device__ __forceinline__ void load_head(const SsdParams &p, unsigned char *smem, int buf, int h, int64_t c,
                                          int64_t t0, int L, uint64_t *full, int ld) {
    using TL = TcLayout<Q, N>;
    unsigned char *xs = smem + (buf ? TL::kBuf1 : TL::kBuf0);
    unsigned char *ss = xs + TL::kXBytes;
    float *aux = reinterpret_cast<float *>(smem + (buf ? TL::kAux1 : TL::kAux0));
    const int64_t ch = tc_ws_unit(p, c, h);
    if (ld == 0) {
        mbar_expect_tx(full, TL::kSBytes + 2 * Q * 4);  // the state parts, cs and dt
        bulk_load(ss, reinterpret_cast<const unsigned char *>(p.ws_state + ch * kTcP * N), TL::kSBytes, full);
        bulk_load(aux, p.ws_acs + ch * Q, Q * 4, full);
        bulk_load(aux + Q, p.ws_dtp + ch * Q, Q * 4, full);
    }
    // x rows as fp16 (the weights' type) times 2^kx, which puts the head's
    // largest |x| in [2^13, 2^14): exact for every value down to 2^-11 of
    // that largest one.  One 16-byte piece = 8 dim rows j of token s.  Loader
    // warp wl takes the token octets wl, wl + 2, ...; in one store phase
    // (8 lanes k) lane k writes piece j = k of token 8 o + (k + q + 4 u) % 8,
    // so the 8 pieces land in 8 different bank groups (pieces of one token
    // are 16 Q bytes apart, a multiple of 128); 16 loads in flight per lane.
    const float4 scl = __ldg(reinterpret_cast<const float4 *>(p.ws_scl + ch * 4));
    const int kx = fp16_scale_exp(scl.x);
    const float sx = pow2i(kx);
    if (ld == 0) {
        aux[4 * Q] = pow2i(-kx);
        aux[4 * Q + 1] = scl.y;
    }
    const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(p.x) + static_cast<int64_t>(h) * kTcP;
    constexpr int kOct = Q / 8;
    const int wl = ld >> 5, q = (ld >> 3) & 3, k = ld & 7;
    for (int o0 = wl; o0 < kOct; o0 += 16) {
        uint4 v[16];
#pragma unroll
        for (int u2 = 0; u2 < 16; ++u2) {
            const int o = o0 + 2 * (u2 >> 1), s = 8 * o + ((k + q + 4 * (u2 & 1)) & 7);
            v[u2] = make_uint4(0u, 0u, 0u, 0u);
            if (o < kOct && s < L)
                v[u2] = __ldg(reinterpret_cast<const uint4 *>(xg + (t0 + s) * p.H * kTcP + 8 * k));
        }
#pragma unroll
        for (int u2 = 0; u2 < 16; ++u2) {
            const int o = o0 + 2 * (u2 >> 1), s = 8 * o + ((k + q + 4 * (u2 & 1)) & 7);
            if (o >= kOct) continue;
            const uint32_t w[4] = {v[u2].x, v[u2].y, v[u2].z, v[u2].w};
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 hv =
                    __floats2half2_rn(__uint_as_float(w[e] << 16) * sx, __uint_as_float(w[e] & 0xffff0000u) * sx);
                out[e] = *reinterpret_cast<const uint32_t *>(&hv);
            }
            *reinterpret_cast<uint4 *>(xs + k * (16 * Q) + 16 * s) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

// The CTA's share of the units u = (chunk c, group g, head i of the group),
// numbered u = (c G + g) hpg + i: a contiguous range, equal in count for
// every CTA.  A segment is the part of the range within one (chunk, group):
// it shares C . B^T.  Every role walks the same segments in the same order.
struct TcSegment {
    int64_t c, t0;
    int g, ia, nh, L;
};
struct TcWalk {
    int64_t u, ue;
    __device__ TcWalk(const SsdParams &p) {
        const int64_t units = p.nchunks * p.G * p.hpg;
        u = units * blockIdx.x / gridDim.x;
        ue = units * (blockIdx.x + 1) / gridDim.x;
    }
    // The next segment holding work (chunks that are malformed -- flagged
    // by chunk_state -- or empty are passed over); false at the end.
    __device__ bool next(const SsdParams &p, int Q, TcSegment &sg) {
        while (u < ue) {
            const int64_t cg = u / p.hpg;
            sg.ia = static_cast<int>(u - cg * p.hpg);
            sg.nh = static_cast<int>(min(static_cast<int64_t>(p.hpg - sg.ia), ue - u));
            u += sg.nh;
            sg.c = cg / p.G;
            sg.g = static_cast<int>(cg - sg.c * p.G);
            const int64_t t0 = load_index(p.cu_chunk, sg.c, p.meta_i64), t1 = load_index(p.cu_chunk, sg.c + 1, p.meta_i64);
            if (t0 < 0 || t1 <= t0 || t1 - t0 > Q || t1 > p.tokens) continue;
            sg.t0 = t0;
            sg.L = static_cast<int>(t1 - t0);
            return true;
        }
        return false;
    }
};

template <int Q, int N>
__global__ void __launch_bounds__(kTcThreads, 1) ssd_scan_tc_kernel(const SsdParams p) {
    using TL = TcLayout<Q, N>;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + TL::kBars);
    uint32_t *taddr_slot = reinterpret_cast<uint32_t *>(smem + TL::kTaddr);
    float *wmax = reinterpret_cast<float *>(smem + TL::kWmax);  // [2][8]: per segment parity, per warp
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long lim = kWaitCycles;
    constexpr float kLog2e = 1.4426950408889634f;

    if (tid == 0) {
        mbar_init(&bars[kBarFull0], 64);
        mbar_init(&bars[kBarFull1], 64);
        mbar_init(&bars[kBarXFree0], 1 + kEpi);
        mbar_init(&bars[kBarXFree1], 1 + kEpi);
        mbar_init(&bars[kBarCB], 1);
        mbar_init(&bars[kBarYFull], 1);
        mbar_init(&bars[kBarYFree], kEpi);
        mbar_init(&bars[kBarFinal], 1);
        mbar_init(&bars[kBarEpi], kEpi);
        for (int i = 0; i < kWBufs; ++i) {
            mbar_init(&bars[kBarWFull0 + i], kEpi);
            mbar_init(&bars[kBarWFree0 + i], 1);
        }
    }
    if (warp == 8) tmem_alloc512(taddr_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *taddr_slot;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(taddr_slot + 1);
    if (tid == 0) *abort_flag = 0;
    __syncthreads();

    // Per head buffer b: its uses so far (the k-th use completes phase k of
    // Full[b] and XFree[b]); the head of a segment's j-th unit uses buffer
    // j % 2, so a segment's first head (loaded with C and B) uses buffer 0.
    int uses0 = 0, uses1 = 0;
    int seg = 0;  // segments begun (phase of CB)
    TcWalk walk(p);
    TcSegment sg;

    if (warp >= 9) {
        // ---------------- loads (two warps) ----------------
        const int ld = tid - 9 * 32;  // 0..63
        const __nv_bfloat16 *Cg = static_cast<const __nv_bfloat16 *>(p.C);
        const __nv_bfloat16 *Bg = static_cast<const __nv_bfloat16 *>(p.B);
        bool ok = true;
        while (ok && walk.next(p, Q, sg)) {
            // both head buffers and C, B free: the previous segment is done
            // (its last MMAs have read C and B, its weights are formed)
            if (uses0 > 0) ok = mbar_wait_bounded(&bars[kBarXFree0], (uses0 - 1) & 1, lim);
            if (ok && uses1 > 0) ok = mbar_wait_bounded(&bars[kBarXFree1], (uses1 - 1) & 1, lim);
            if (ok && *abort_flag) ok = false;
            if (!ok) break;
            for (int i = ld; i < Q * (N / 8); i += 64) {
                const int t = i / (N / 8), k = i % (N / 8);
                const bool in = t < sg.L;
                const int64_t src = ((sg.t0 + t) * p.G + sg.g) * N + 8 * k;
                const int dst = (t >> 3) * (16 * N) + k * 128 + (t & 7) * 16;
                cp16(smem + TL::kC + dst, in ? Cg + src : Cg, in);
                cp16(smem + TL::kB + dst, in ? Bg + src : Bg, in);
            }
            cp_wait_all();
            fence_proxy_async_smem();
            for (int j = 0; j < sg.nh; ++j) {
                const int buf = j & 1;
                if (j == 1 && TL::kAlias)
                    ok = mbar_wait_bounded(&bars[kBarCB], seg & 1, lim);  // B's place holds buffer 1
                else if (j >= 2)
                    ok = mbar_wait_bounded(&bars[buf ? kBarXFree1 : kBarXFree0], ((buf ? uses1 : uses0) - 1) & 1, lim);
                if (ok && *abort_flag) ok = false;
                if (!ok) break;
                load_head<Q, N>(p, smem, buf, sg.g * p.hpg + sg.ia + j, sg.c, sg.t0, sg.L,
                                &bars[buf ? kBarFull1 : kBarFull0], ld);
                fence_proxy_async_smem();
                mbar_arrive(&bars[buf ? kBarFull1 : kBarFull0]);
                (buf ? uses1 : uses0) += 1;
            }
            ++seg;
        }
        if (!ok && ld == 0) {
            flag(p.status, kDevTimeout);
            *abort_flag = 1;
        }
        // the bulk copies of the last heads loaded have landed before the CTA
        // retires (already so unless a wait gave up)
        if (ld == 0) {
            if (uses0 > 0) mbar_wait_bounded(&bars[kBarFull0], (uses0 - 1) & 1, lim);
            if (uses1 > 0) mbar_wait_bounded(&bars[kBarFull1], (uses1 - 1) & 1, lim);
        }
    } else if (warp == 8) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            const uint32_t sC = smem_addr(smem + TL::kC), sB = smem_addr(smem + TL::kB);
            const uint32_t sW = smem_addr(smem + TL::kW);
            constexpr uint32_t kSboNK = 16 * N;  // M/N-direction core-matrix stride of C, B, S_in
            bool ok = true;
            int blk = 0, tile = 0;  // running counts of weight blocks and (head, tile) results
            while (ok && walk.next(p, Q, sg)) {
                const int ntiles = sg.L > 128 ? 2 : 1;
                for (int j = 0; ok && j < sg.nh; ++j) {
                    const int buf = j & 1;
                    if (!(ok = mbar_wait_bounded(&bars[buf ? kBarFull1 : kBarFull0], (buf ? uses1 : uses0) & 1, lim))) break;
                    tc_fence_after();
                    if (j == 0) {
                        // C . B^T: tile 0 (columns s < 128), tile 1 (all Q columns)
                        for (int kk = 0; kk < N / 16; ++kk)
                            mma(tmem, smem_desc(sC + 256 * kk, 128, kSboNK), smem_desc(sB + 256 * kk, 128, kSboNK),
                                idesc_f16(128, TL::kNcols0, 0, 0), kk > 0);
                        if (ntiles > 1)
                            for (int kk = 0; kk < N / 16; ++kk)
                                mma(tmem + TL::kCB1, smem_desc(sC + 128 / 8 * kSboNK + 256 * kk, 128, kSboNK),
                                    smem_desc(sB + 256 * kk, 128, kSboNK), idesc_f16(128, 256, 0, 0), kk > 0);
                        mma_commit(&bars[kBarCB]);
                    }
                    const uint32_t sX = smem_addr(smem + (buf ? TL::kBuf1 : TL::kBuf0));
                    const uint32_t sS = sX + TL::kXBytes;
                    for (int m = 0; ok && m < ntiles; ++m, ++tile) {
                        if (tile > 0 && !(ok = mbar_wait_bounded(&bars[kBarYFree], (tile - 1) & 1, lim))) break;
                        tc_fence_after();
                        // Y1 = C_m . S_in^T, high part then low part
                        const uint32_t cm = sC + m * (128 / 8) * kSboNK;
                        for (int part = 0; part < 2; ++part)
                            for (int kk = 0; kk < N / 16; ++kk)
                                mma(tmem + TL::kY1, smem_desc(cm + 256 * kk, 128, kSboNK),
                                    smem_desc(sS + part * (kTcP * N * 2) + 256 * kk, 128, kSboNK),
                                    idesc_f16(128, kTcP, 0, 0), part > 0 || kk > 0);
                        // Y2 = sum over blocks W_b . X_b
                        const int nblk = (m == 0 ? TL::kNcols0 : Q) / kTcBlock;
                        for (int b = 0; b < nblk; ++b, ++blk) {
                            const int wb = blk % kWBufs;
                            if (!(ok = mbar_wait_bounded(&bars[kBarWFull0 + wb], (blk / kWBufs) & 1, lim))) break;
                            tc_fence_after();
                            for (int k2 = 0; k2 < kTcBlock / 16; ++k2)
                                mma(tmem + TL::kY2,
                                    smem_desc(sW + wb * TL::kWBuf + 256 * k2, 128, (kTcBlock / 8) * 128),
                                    smem_desc(sX + 16 * (kTcBlock * b + 16 * k2), 128, 16 * Q),
                                    idesc_f16(128, kTcP, 0, 1, 0), b > 0 || k2 > 0);
                            mma_commit(&bars[kBarWFree0 + wb]);
                        }
                        if (ok) mma_commit(&bars[kBarYFull]);
                    }
                    if (ok) mma_commit(&bars[buf ? kBarXFree1 : kBarXFree0]);
                    (buf ? uses1 : uses0) += 1;
                }
                ++seg;
            }
            if (!ok) {
                flag(p.status, kDevTimeout);
                *abort_flag = 1;
            }
            // every MMA issued has completed before tensor memory is freed
            mma_commit(&bars[kBarFinal]);
            mbar_wait_bounded(&bars[kBarFinal], 0, lim);
        }
        __syncwarp();
    } else {
        // ---------------- weights and readout ----------------
        // warps w and w + 4 own tensor-memory lanes 32 (w % 4) + lane, i.e.
        // row t of the tile; `half` picks their columns and outputs
        const int t = (warp & 3) * 32 + lane, half = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        unsigned char *wsm = smem + TL::kW;
        float *cbd_s = reinterpret_cast<float *>(smem + TL::kCbd);
        const __nv_bfloat16 *zg = static_cast<const __nv_bfloat16 *>(p.z);
        __nv_bfloat16 *yg = static_cast<__nv_bfloat16 *>(p.y);
        bool ok = true;
        int blk = 0, tile = 0, ephase = 0;
        float seg_cbmax = 0.f;
        while (ok && walk.next(p, Q, sg)) {
            const int ntiles = sg.L > 128 ? 2 : 1;
            const int L = sg.L;
            const int64_t t0 = sg.t0;
            for (int j = 0; ok && j < sg.nh; ++j) {
                const int buf = j & 1, h = sg.g * p.hpg + sg.ia + j;
                if (j == 0) {
                    if (!(ok = mbar_wait_bounded(&bars[kBarCB], seg & 1, lim))) break;
                    tc_fence_after();
                    // the largest |C_t . B_s| over the chunk's rows: with dt'
                    // it bounds every weight (the decays are at most 1), and
                    // so picks the power-of-two scale of each head's weights
                    float mcb = 0.f;
                    for (int m = 0; m < ntiles; ++m) {
                        const int ncol = m == 0 ? TL::kNcols0 : Q;
                        for (int s0 = half * (ncol / 2); s0 < (half + 1) * (ncol / 2); s0 += 16) {
                            uint32_t r[16];
                            tmem_ld16(tmem + lane_base + (m == 0 ? 0u : static_cast<uint32_t>(TL::kCB1)) + s0, r);
                            tmem_wait_ld();
                            if (128 * m + t < L) {
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj) mcb = fmaxf(mcb, fabsf(__uint_as_float(r[jj])));
                            }
                        }
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mcb = fmaxf(mcb, __shfl_xor_sync(0xffffffffu, mcb, off));
                    if (lane == 0) wmax[(seg & 1) * 8 + warp] = mcb;
                }
                if (!(ok = mbar_wait_bounded(&bars[buf ? kBarFull1 : kBarFull0], (buf ? uses1 : uses0) & 1, lim))) break;
                float *aux = reinterpret_cast<float *>(smem + (buf ? TL::kAux1 : TL::kAux0));
                const float *cs = aux, *dtp = aux + Q;
                float *E = aux + 2 * Q, *cs2 = aux + 3 * Q;
                // per column: cs log2(e), and E_s = 2^(cs2_r - cs2_s) dt'_s with r the last column of s's block
                for (int s = tid; s < Q; s += kEpi) {
                    const float c2 = cs[s] * kLog2e;
                    cs2[s] = c2;
                    E[s] = ex2(cs[s | (kTcBlock - 1)] * kLog2e - c2) * dtp[s];
                }
                if (!(ok = epi_sync(&bars[kBarEpi], ephase, lim))) break;
                if (j == 0) {
                    seg_cbmax = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) seg_cbmax = fmaxf(seg_cbmax, wmax[(seg & 1) * 8 + w]);
                }
                const unsigned char *xs = smem + (buf ? TL::kBuf1 : TL::kBuf0);
                const float Dh = p.D ? p.D[h] : 0.f;
                // the weights are formed times 2^kw, x was staged times 2^kx
                const int kw = fp16_scale_exp(seg_cbmax * aux[4 * Q + 1]);
                const float sw = pow2i(kw), xinv = aux[4 * Q], yinv = xinv * pow2i(-kw);
                for (int m = 0; ok && m < ntiles; ++m, ++tile) {
                    const int tg = 128 * m + t;  // token row within the chunk
                    const float cst = cs2[tg < Q ? tg : Q - 1];
                    // the gate's z row of this thread's outputs, in flight while the weights are formed
                    const int64_t row = ((t0 + tg) * p.H + h) * static_cast<int64_t>(kTcP);
                    uint4 zpre[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                                     make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                    if (zg && tg < L) {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            zpre[jj] = __ldg(reinterpret_cast<const uint4 *>(zg + row + 8 * (4 * half + jj)));
                    }
                    const uint32_t cbcol = m == 0 ? 0u : static_cast<uint32_t>(TL::kCB1);
                    const int nblk = (m == 0 ? TL::kNcols0 : Q) / kTcBlock;
                    for (int b = 0; b < nblk; ++b, ++blk) {
                        const int wb = blk % kWBufs;
                        if (blk >= kWBufs &&
                            !(ok = mbar_wait_bounded(&bars[kBarWFree0 + wb], ((blk - kWBufs) / kWBufs) & 1, lim)))
                            break;
                        const int s0 = kTcBlock * b + 16 * half;  // this thread's 16 columns
                        uint32_t r[16];
                        tmem_ld16(tmem + lane_base + cbcol + s0, r);
                        tmem_wait_ld();
                        float wv[16];
                        if (kTcBlock * b + kTcBlock <= tg) {
                            // the block lies wholly before row t
                            const float R = ex2(cst - cs2[kTcBlock * b + kTcBlock - 1]) * sw;
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) wv[jj] = __uint_as_float(r[jj]) * R * E[s0 + jj];
                        } else if (kTcBlock * b > tg) {
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) wv[jj] = 0.f;
                        } else {
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) {
                                const int s = s0 + jj;
                                const float cb = __uint_as_float(r[jj]);
                                if (s == tg) cbd_s[(tile & 1) * 128 + t] = cb;
                                wv[jj] = s < tg ? cb * ex2(cst - cs2[s]) * (dtp[s] * sw) : 0.f;
                            }
                        }
                        uint32_t hv[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const __half2 h2 = __floats2half2_rn(wv[2 * jj], wv[2 * jj + 1]);
                            hv[jj] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        const int off =
                            wb * TL::kWBuf + (t >> 3) * ((kTcBlock / 8) * 128) + 2 * half * 128 + (t & 7) * 16;
                        *reinterpret_cast<uint4 *>(wsm + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                        *reinterpret_cast<uint4 *>(wsm + off + 128) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
                        fence_proxy_async_smem();
                        mbar_arrive(&bars[kBarWFull0 + wb]);
                    }
                    if (!ok) break;
                    // the tile's results; the thread holding row t's diagonal has stored it
                    if (!(ok = mbar_wait_bounded(&bars[kBarYFull], tile & 1, lim))) break;
                    tc_fence_after();
                    if (!(ok = epi_sync(&bars[kBarEpi], ephase, lim))) break;
                    uint32_t y1[32], y2[32];
                    tmem_ld16(tmem + lane_base + TL::kY1 + 32 * half, y1);
                    tmem_ld16(tmem + lane_base + TL::kY1 + 32 * half + 16, y1 + 16);
                    tmem_ld16(tmem + lane_base + TL::kY2 + 32 * half, y2);
                    tmem_ld16(tmem + lane_base + TL::kY2 + 32 * half + 16, y2 + 16);
                    tmem_wait_ld();
                    const float cbd = cbd_s[(tile & 1) * 128 + t];
                    tc_fence_before();
                    mbar_arrive(&bars[kBarYFree]);
                    if (tg < L) {
                        const float e1 = ex2(cst);
                        const float wd = fmaf(cbd, dtp[tg], Dh) * xinv;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int jo = 4 * half + jj;  // p-octet
                            const uint4 xv = *reinterpret_cast<const uint4 *>(xs + jo * (16 * Q) + 16 * tg);
                            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};  // fp16 pairs
                            const uint32_t zw[4] = {zpre[jj].x, zpre[jj].y, zpre[jj].z, zpre[jj].w};
                            uint32_t out[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float v[2];
#pragma unroll
                                for (int k = 0; k < 2; ++k) {
                                    const int pp = 8 * jj + 2 * e + k;
                                    const float xv1 = __half2float(__ushort_as_half(
                                        static_cast<unsigned short>(k ? (xw[e] >> 16) : (xw[e] & 0xffffu))));
                                    v[k] = fmaf(wd, xv1,
                                                fmaf(e1, __uint_as_float(y1[pp]), __uint_as_float(y2[pp]) * yinv));
                                    if (zg) {
                                        const float zz = __uint_as_float(k ? (zw[e] & 0xffff0000u) : (zw[e] << 16));
                                        v[k] *= __fdividef(zz, 1.f + __expf(-zz));
                                    }
                                }
                                out[e] = pack_bf16x2(v[0], v[1]);
                            }
                            *reinterpret_cast<uint4 *>(yg + row + 8 * jo) = make_uint4(out[0], out[1], out[2], out[3]);
                        }
                    }
                }
                // this head's buffer (x rows, state, sums) may be refilled and,
                // after a segment's last head, C . B^T replaced
                if (!ok) break;
                tc_fence_before();
                mbar_arrive(&bars[buf ? kBarXFree1 : kBarXFree0]);
                (buf ? uses1 : uses0) += 1;
            }
            ++seg;
        }
        if (!ok) {
            if (tid == 0) flag(p.status, kDevTimeout);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8) tmem_dealloc512(tmem);
}

// Number of SMs of the current device (cached per device).
static int tc_sm_count() {
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = __atomic_load_n(&cache[dev], __ATOMIC_RELAXED);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        __atomic_store_n(&cache[dev], n, __ATOMIC_RELAXED);
    }
    return n;
}

// A persistent grid: one CTA per SM (the layout takes most of an SM's shared
// memory), or one per unit when there are fewer units.
template <int Q, int N>
cudaError_t launch_scan_tc_qn(const SsdParams &p, cudaStream_t stream) {
    using TL = TcLayout<Q, N>;
    cudaError_t e = cudaFuncSetAttribute(ssd_scan_tc_kernel<Q, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TL::kBytes);
    if (e != cudaSuccess) return e;
    const int sms = tc_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t units = p.nchunks * p.G * p.hpg;
    if (units == 0) return cudaSuccess;
    const int64_t grid = units < sms ? units : sms;
    ssd_scan_tc_kernel<Q, N><<<static_cast<unsigned>(grid), kTcThreads, TL::kBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_scan_tc(const SsdParams &p, cudaStream_t stream) {
    if (p.P != kTcP) return cudaErrorInvalidValue;
    switch (p.Q * 1000 + p.N) {
    case 64 * 1000 + 64: return launch_scan_tc_qn<64, 64>(p, stream);
    case 64 * 1000 + 128: return launch_scan_tc_qn<64, 128>(p, stream);
    case 128 * 1000 + 64: return launch_scan_tc_qn<128, 64>(p, stream);
    case 128 * 1000 + 128: return launch_scan_tc_qn<128, 128>(p, stream);
    case 256 * 1000 + 64: return launch_scan_tc_qn<256, 64>(p, stream);
    case 256 * 1000 + 128: return launch_scan_tc_qn<256, 128>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
