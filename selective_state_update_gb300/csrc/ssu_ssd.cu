// ssu_ssd.cu -- packed variable-length SSD prefill (Mamba-2).
//
// MATE documentation, page "Mamba / SSU", section "SSD packed prefill" and
// the API reference of ssd_combined_fwd_varlen: the recurrence of the decode
// step applied to every token of a packed batch of sequences, evaluated
// chunk by chunk in the five stages the page names -- chunk-local dt / decay
// cumulative sums, the states the chunks produce on their own, the passing
// of states from chunk to chunk, the C . B^T products and the chunk scan.
// For chunk c of tokens t (length Lc <= Q), head h, g = h / (heads/groups):
//     a_t   = A[h] dt'_t,  dt'_t = clamp(softplus(dt + bias), lo, hi)
//     Sc    = sum_t exp(sum_{s>t} a_s) dt'_t x_t B_t^T             (P x N)
//     S_end = exp(sum_t a_t) S_in + Sc
//     y_t   = exp(cs_t) C_t . S_in + sum_{s<=t} (C_t . B_s) exp(cs_t - cs_s) dt'_s x_s + D x_t
// with cs the inclusive cumulative sum of a over the chunk, y gated by
// silu(z).  A chunk opens a sequence when seq_idx changes (the page: seq_idx
// is the authority); its S_in is then the initial state (or zero).
//
// Four kernels over a caller-owned workspace; every contraction runs on the
// tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulation), with
// operands staged in shared memory in the inputs' own row layout by 16-byte
// cp.async and read as fragments with ldmatrix:
//   chunk_state  one CTA per (head, chunk): dt', the prefix and suffix sums
//                of a, and Sc = (w x)^T B with w_t = exp(sum_{s>t} a) dt'_t;
//                w x is split into a bf16 high and low part so that Sc keeps
//                ~2^-17 relative precision (the returned states need it);
//   state_pass   one CTA per (run of a sequence's chunks, head): replaces
//                each Sc in the workspace by the chunk's entering state (as
//                bf16 high and low parts) and writes the returned states;
//   chunk_cb     one CTA per (group, chunk): the causal 16 x 16 tiles of
//                C . B^T in fp32, stored in mma fragment order so that the
//                heads of the group read them back with coalesced loads, and
//                the diagonal C_t . B_t on its own;
//   chunk_scan   one CTA per (head, chunk): y from the entering state
//                (C . S_in^T scaled by exp(cs_t)) and from the strictly causal
//                weights (C . B^T) exp(cs_t - cs_s) dt'_s times x, the state
//                and the weights as bf16 high + low parts (one-part bf16
//                operands measured errors of up to 2.4 % of a token's row);
//                the diagonal weight (C_t . B_t) dt'_t and D are applied in
//                fp32, since the two can cancel for every dim row of a token
//                (both multiply x_t).
#include <cstdint>
#include <mutex>

#include "ssu_device.cuh"
#include "ssu_ssd_params.h"

namespace ssu {

// ---------------------------------------------------------------------------
// Tensor-core and staging helpers.  mma m16n8k16: A row-major (16 x 16), B
// "column-major" (16 x 8), fp32 accumulators.  Fragment of lane l (g = l/4,
// q = l%4): A {A[g][2q..2q+1]}, {A[g+8][2q..]}, {A[g][2q+8..]}, {A[g+8][2q+8..]};
// B {B[2q..2q+1][g]}, {B[2q+8..2q+9][g]}; D {D[g][2q..2q+1]}, {D[g+8][2q..2q+1]}.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8 x 8 b16 matrices from shared memory; lanes 8i..8i+7 give the row
// addresses of matrix i.  Lane l receives (row l/4, columns 2(l%4), 2(l%4)+1)
// of each matrix, or with .trans (rows 2(l%4), 2(l%4)+1, column l/4).
__device__ __forceinline__ void ldsm_x4(uint32_t *r, const void *smem_row) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_row));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t *r, const void *smem_row) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem_row));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

// 16 bytes global -> shared, asynchronously; `valid` false fills zeros and
// reads nothing.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(a), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Two floats as bf16x2 (x0 in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float x0, float x1) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(x0, x1);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// The bf16 high part of two floats and the bf16 low part of what is left.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t *hi, uint32_t *lo) {
    *hi = pack_bf16(x0, x1);
    const float h0 = __uint_as_float(*hi << 16), h1 = __uint_as_float(*hi & 0xffff0000u);
    *lo = pack_bf16(x0 - h0, x1 - h1);
}

// 2^x by the special-function unit (PTX ex2.approx.ftz: relative error
// below 2^-22, results below 2^-126 flushed to zero); x <= 0 here.
__device__ __forceinline__ float ex2_fast(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ int64_t meta_at(const void *p, int64_t i, int is_i64) { return load_index(p, i, is_i64); }

// Element (p, n) of a P x N state in the order the tensor cores read a
// K-major operand without swizzle: 8 x 8 core matrices (8 rows p of 8
// consecutive n), stored one after another along n, then along p.  The
// chunk states are kept in this order in the workspace (fp32), and the
// entering states as its bf16 high and low parts.
template <int N>
__host__ __device__ constexpr int canon(int p, int n) {
    return (p >> 3) * (N * 8) + (n >> 3) * 64 + (p & 7) * 8 + (n & 7);
}

// The causal 16 x 16 tiles (row tile m, column tile j <= m) of a chunk of Q
// tokens, numbered row tile by row tile.
__host__ __device__ constexpr int cb_tiles(int Q) { return (Q / 16) * (Q / 16 + 1) / 2; }
__device__ __forceinline__ int cb_tile(int m, int j) { return m * (m + 1) / 2 + j; }

// Index of (chunk c, head h) in the per-(chunk, head) workspace arrays:
// head-major, so that the chunks of one sequence and head are neighbours.
__device__ __forceinline__ int64_t ws_unit(const SsdParams &p, int64_t c, int h) {
    return static_cast<int64_t>(h) * p.nchunks + c;
}

// dt' of token t, head h: dt (+ bias), softplus, clamped to [lo, hi].
__device__ __forceinline__ float ssd_step(const SsdParams &p, int64_t t, int h) {
    const int64_t i = t * p.H + h;
    float v = p.dt_dtype == kF32 ? static_cast<const float *>(p.dt)[i]
                                 : bits_to_float(static_cast<const unsigned short *>(p.dt)[i], p.dt_dtype);
    v = processed_step(v, p.dt_bias ? p.dt_bias[h] : 0.f, p.softplus);
    return fminf(fmaxf(v, p.dt_lo), p.dt_hi);
}

// Inclusive prefix sums of v[0..n) in shared memory, one value per thread of
// a block of kThreads >= n threads, in place; `tmp` holds kThreads/32 floats.
template <int kThreads>
__device__ void block_scan(float *v, int n, float *tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float a = tid < n ? v[tid] : 0.f;
    float s = a;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    if (lane == 31) tmp[warp] = s;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; ++w) base += tmp[w];
    if (tid < n) v[tid] = base + s;
    __syncthreads();
}

// Rows [0, Q) of a bf16 tensor with row stride `stride` starting at row t0,
// `cols` columns from column c0, into shared-memory rows of `ld` elements;
// rows from L on are zero.  One 16-byte cp.async per 8 columns.
template <int kThreads>
__device__ __forceinline__ void stage_rows(__nv_bfloat16 *dst, int ld, const __nv_bfloat16 *src, int64_t t0,
                                           int64_t stride, int64_t c0, int Q, int L, int cols) {
    const int per_row = cols / 8;
    for (int i = threadIdx.x; i < Q * per_row; i += kThreads) {
        const int r = i / per_row, k = (i % per_row) * 8;
        const bool ok = r < L;
        const __nv_bfloat16 *s = ok ? src + (t0 + r) * stride + c0 + k : src;
        cp_async16(dst + r * ld + k, s, ok);
    }
}

// ---------------------------------------------------------------------------
// Stages 1-2: per (head, chunk) the cumulative sums and the chunk's own state.
// ---------------------------------------------------------------------------
template <int Q, int P, int N>
struct ChunkStateSmem {
    __nv_bfloat16 xs[Q][P + 8];  // x of the chunk, xs[t][p]
    __nv_bfloat16 bs[Q][N + 8];  // B of the chunk's group, bs[t][n]
    float cs[Q];                 // inclusive cumulative sums of a
    float rs[Q];                 // inclusive cumulative sums of a, reversed
    float w[Q];                  // dt', then exp(sum of the later a) dt'
    float tmp[8];
};

constexpr int kStateThreads = 256;

template <int Q, int P, int N>
__global__ void __launch_bounds__(kStateThreads, 2) ssd_chunk_state_kernel(const SsdParams p) {
    static_assert(P == 64 && N % 64 == 0 && Q <= kStateThreads, "tiling");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<ChunkStateSmem<Q, P, N> *>(smem_raw);
    const int h = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
    const int g = h / p.hpg;
    const int64_t t0 = meta_at(p.cu_chunk, c, p.meta_i64), t1 = meta_at(p.cu_chunk, c + 1, p.meta_i64);
    if (c == 0 && h == 0 && !p.intermediate) {  // every sequence's last chunk must name a chunk
        for (int64_t s = tid; s < p.nseq; s += kStateThreads) {
            const int64_t lc = meta_at(p.last_chunk, s, p.meta_i64);
            if (lc < 0 || lc >= p.nchunks) flag(p.status, kDevBadEntry);
        }
    }
    if (t0 < 0 || t1 < t0 || t1 - t0 > Q || t1 > p.tokens) {
        if (tid == 0) flag(p.status, kDevBadSeqlen);
        return;
    }
    const int L = static_cast<int>(t1 - t0);
    // the chunk's x and B rows, in flight while the decays are formed
    stage_rows<kStateThreads>(&sm.xs[0][0], P + 8, static_cast<const __nv_bfloat16 *>(p.x), t0,
                              static_cast<int64_t>(p.H) * P, static_cast<int64_t>(h) * P, Q, L, P);
    stage_rows<kStateThreads>(&sm.bs[0][0], N + 8, static_cast<const __nv_bfloat16 *>(p.B), t0,
                              static_cast<int64_t>(p.G) * N, static_cast<int64_t>(g) * N, Q, L, N);
    float *ws_acs = p.ws_acs + ws_unit(p, c, h) * Q;
    float *ws_dtp = p.ws_dtp + ws_unit(p, c, h) * Q;
    const float Ah = p.A[h];
    if (tid < Q) {
        const float d = tid < L ? ssd_step(p, t0 + tid, h) : 0.f;
        ws_dtp[tid] = d;
        sm.w[tid] = d;
        sm.cs[tid] = tid < L ? Ah * d : 0.f;
        sm.rs[tid] = 0.f;
    }
    __syncthreads();
    if (tid < L) sm.rs[tid] = sm.cs[L - 1 - tid];  // a reversed
    __syncthreads();
    block_scan<kStateThreads>(sm.cs, Q, sm.tmp);
    // rs[i] = sum of a over the last i + 1 tokens, summed from the end so the
    // weights of recent tokens carry no cancellation
    block_scan<kStateThreads>(sm.rs, Q, sm.tmp);
    if (tid < Q) {
        ws_acs[tid] = sm.cs[tid];
        const float later = tid + 1 < L ? sm.rs[L - 2 - tid] : 0.f;  // sum_{s>t} a_s
        sm.w[tid] = tid < L ? expf(later) * sm.w[tid] : 0.f;
    }
    if (tid == 0) p.ws_dec[ws_unit(p, c, h)] = L > 0 ? expf(sm.rs[L - 1]) : 1.f;
    cp_async_wait_all();
    __syncthreads();

    // Sc[p][n] = sum_t (w_t x[t][p]) B[t][n]: M = P, N, K = t.  Warp w: rows
    // p0 = 16 (w % 4), columns from n0 = (N / 2)(w / 4).
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, q = lane & 3, mi = lane >> 3;
    const int p0 = (warp & 3) * 16, n0 = (warp >> 2) * (N / 2);
    constexpr int NT = N / 16;  // n-tiles of 8 per warp
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    for (int k0 = 0; k0 < L; k0 += 16) {
        // A = (w x)^T: matrices (p 0-7 | 8-15) x (t 0-7 | 8-15) of xs, transposed
        uint32_t ax[4], ahi[4], alo[4];
        ldsm_x4_trans(ax, &sm.xs[k0 + (lane & 7) + (mi >> 1) * 8][p0 + (mi & 1) * 8]);
        const float w0 = sm.w[k0 + 2 * q], w1 = sm.w[k0 + 2 * q + 1];
        const float w8 = sm.w[k0 + 2 * q + 8], w9 = sm.w[k0 + 2 * q + 9];
        split_bf16(bf16_lo(ax[0]) * w0, bf16_hi(ax[0]) * w1, &ahi[0], &alo[0]);
        split_bf16(bf16_lo(ax[1]) * w0, bf16_hi(ax[1]) * w1, &ahi[1], &alo[1]);
        split_bf16(bf16_lo(ax[2]) * w8, bf16_hi(ax[2]) * w9, &ahi[2], &alo[2]);
        split_bf16(bf16_lo(ax[3]) * w8, bf16_hi(ax[3]) * w9, &ahi[3], &alo[3]);
        // the high part for every n-tile, then the low part: no accumulator is
        // used twice in a row
        uint32_t bb[NT / 2][4];
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
            // B[t][n]: matrices (t 0-7 | 8-15) x (n-tile j | j+1), transposed
            ldsm_x4_trans(bb[j / 2], &sm.bs[k0 + (lane & 7) + (mi & 1) * 8][n0 + 8 * j + (mi >> 1) * 8]);
            mma_bf16(acc[j], ahi, bb[j / 2][0], bb[j / 2][1]);
            mma_bf16(acc[j + 1], ahi, bb[j / 2][2], bb[j / 2][3]);
        }
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
            mma_bf16(acc[j], alo, bb[j / 2][0], bb[j / 2][1]);
            mma_bf16(acc[j + 1], alo, bb[j / 2][2], bb[j / 2][3]);
        }
    }
    float *out = p.ws_state + ws_unit(p, c, h) * P * N;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int n = n0 + 8 * j + 2 * q;
        *reinterpret_cast<float2 *>(out + canon<N>(p0 + gq, n)) = make_float2(acc[j][0], acc[j][1]);
        *reinterpret_cast<float2 *>(out + canon<N>(p0 + gq + 8, n)) = make_float2(acc[j][2], acc[j][3]);
    }
}

// ---------------------------------------------------------------------------
// Stage 3: states passed from chunk to chunk, one CTA per (run, head).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_state4(float *o, float4 v) { *reinterpret_cast<float4 *>(o) = v; }
__device__ __forceinline__ void store_state4(__half *o, float4 v) {
    o[0] = __float2half_rn(v.x), o[1] = __float2half_rn(v.y), o[2] = __float2half_rn(v.z), o[3] = __float2half_rn(v.w);
}
__device__ __forceinline__ void store_state4(__nv_bfloat16 *o, float4 v) {
    o[0] = __float2bfloat16_rn(v.x), o[1] = __float2bfloat16_rn(v.y), o[2] = __float2bfloat16_rn(v.z),
    o[3] = __float2bfloat16_rn(v.w);
}

template <typename TS>
__device__ __forceinline__ float4 load_state4(const void *base, int64_t i) {
    if constexpr (sizeof(TS) == 4) {
        return *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + i);
    } else {
        const TS *o = static_cast<const TS *>(base) + i;
        return make_float4(to_float(o[0]), to_float(o[1]), to_float(o[2]), to_float(o[3]));
    }
}

constexpr int kPassThreads = 256;
constexpr int kPassList = 256;  // returned states a run keeps in its list

// One CTA per (chunk c0, head); only a chunk that opens a run of its
// sequence's chunks works: it walks the run, the next chunk's Sc loaded
// while the current one is replaced.
template <int P, int N, typename TS>
__global__ void __launch_bounds__(kPassThreads) ssd_state_pass_kernel(const SsdParams p) {
    __shared__ int nlist;
    __shared__ int64_t list_chunk[kPassList];
    __shared__ int64_t list_seq[kPassList];
    const int c0 = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int64_t b = meta_at(p.seq_idx, c0, p.meta_i64);
    if (c0 > 0 && meta_at(p.seq_idx, c0 - 1, p.meta_i64) == b) return;  // not the first chunk of a run
    if (b < 0 || b >= p.nseq) {
        if (tid == 0) flag(p.status, kDevBadEntry);
        return;
    }
    // the sequences whose returned state is the end of a chunk of this
    // sequence from c0 on (chunks past the run's end are never reached)
    if (tid == 0) nlist = 0;
    __syncthreads();
    if (!p.intermediate) {
        for (int64_t s = tid; s < p.nseq; s += kPassThreads) {
            const int64_t lc = meta_at(p.last_chunk, s, p.meta_i64);
            if (lc >= c0 && lc < p.nchunks && meta_at(p.seq_idx, lc, p.meta_i64) == b) {
                const int k = atomicAdd(&nlist, 1);
                if (k < kPassList) list_chunk[k] = lc, list_seq[k] = s;
            }
        }
    }
    __syncthreads();
    const bool overflow = nlist > kPassList;
    const int nl = nlist < kPassList ? nlist : kPassList;

    // Thread tid holds the groups e = 4 (k kPassThreads + tid) of the canonical
    // order: four consecutive n of one row p.
    constexpr int kPer = P * N / (kPassThreads * 4);
    const int64_t PN = static_cast<int64_t>(P) * N;
    const int64_t hs = static_cast<int64_t>(h) * PN;
    float *ws0 = p.ws_state + ws_unit(p, 0, h) * PN;  // this head's chunks, contiguous
    int uoff[kPer];                                   // the groups in the [P][N] layout of the states
    float4 S[kPer], sc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int e = 4 * (k * kPassThreads + tid);
        const int pp = (e / (N * 8)) * 8 + (e % 64) / 8, nn = ((e / 64) % (N / 8)) * 8 + (e % 8);
        uoff[k] = pp * N + nn;
        S[k] = p.init ? load_state4<TS>(p.init, b * p.H * PN + hs + uoff[k]) : make_float4(0.f, 0.f, 0.f, 0.f);
        sc[k] = __ldcs(reinterpret_cast<const float4 *>(ws0 + c0 * PN + e));
    }
    for (int64_t c = c0;; ++c) {
        float *ws = ws0 + c * PN;
        const float dec = p.ws_dec[ws_unit(p, c, h)];
        const bool more = c + 1 < p.nchunks && meta_at(p.seq_idx, c + 1, p.meta_i64) == b;
        float4 nx[kPer];
        if (c + 1 < p.nchunks) {  // the next chunk's Sc (read one chunk ahead, also past the run's end)
#pragma unroll
            for (int k = 0; k < kPer; ++k)
                nx[k] = __ldcs(reinterpret_cast<const float4 *>(ws + PN + 4 * (k * kPassThreads + tid)));
        }
        __syncthreads();  // every thread has read chunk c's Sc before its slot is overwritten
        // the state entering chunk c, as bf16 high and low parts in canonical order
        unsigned char *slot = reinterpret_cast<unsigned char *>(ws);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int e = 4 * (k * kPassThreads + tid);
            uint2 hi, lo;
            split_bf16(S[k].x, S[k].y, &hi.x, &lo.x);
            split_bf16(S[k].z, S[k].w, &hi.y, &lo.y);
            *reinterpret_cast<uint2 *>(slot + 2 * e) = hi;
            *reinterpret_cast<uint2 *>(slot + 2 * PN + 2 * e) = lo;
            S[k] = make_float4(fmaf(dec, S[k].x, sc[k].x), fmaf(dec, S[k].y, sc[k].y), fmaf(dec, S[k].z, sc[k].z),
                               fmaf(dec, S[k].w, sc[k].w));
        }
        if (p.intermediate) {
#pragma unroll
            for (int k = 0; k < kPer; ++k) store_state4(static_cast<TS *>(p.states) + c * p.H * PN + hs + uoff[k], S[k]);
        } else {
            for (int i = 0; i < nl; ++i) {
                if (list_chunk[i] != c) continue;
#pragma unroll
                for (int k = 0; k < kPer; ++k)
                    store_state4(static_cast<TS *>(p.states) + list_seq[i] * p.H * PN + hs + uoff[k], S[k]);
            }
            if (overflow) {  // more such sequences than the list holds: find the rest
                for (int64_t s = 0; s < p.nseq; ++s) {
                    if (meta_at(p.last_chunk, s, p.meta_i64) != c) continue;
                    bool listed = false;
                    for (int i = 0; i < nl; ++i) listed |= list_seq[i] == s;
                    if (listed) continue;
#pragma unroll
                    for (int k = 0; k < kPer; ++k)
                        store_state4(static_cast<TS *>(p.states) + s * p.H * PN + hs + uoff[k], S[k]);
                }
            }
        }
        if (!more) break;
#pragma unroll
        for (int k = 0; k < kPer; ++k) sc[k] = nx[k];
    }
}

// ---------------------------------------------------------------------------
// Stage 4: C . B^T per (group, chunk), causal 16 x 16 tiles in fragment order.
// ---------------------------------------------------------------------------
template <int Q, int N>
struct ChunkCbSmem {
    __nv_bfloat16 cm[Q][N + 8];  // C rows, cm[t][n]
    __nv_bfloat16 bm[Q][N + 8];  // B rows, bm[s][n]
};

constexpr int kCbThreads = 256;

template <int Q, int N>
__global__ void __launch_bounds__(kCbThreads) ssd_chunk_cb_kernel(const SsdParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<ChunkCbSmem<Q, N> *>(smem_raw);
    const int g = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
    const int64_t t0 = meta_at(p.cu_chunk, c, p.meta_i64), t1 = meta_at(p.cu_chunk, c + 1, p.meta_i64);
    if (t0 < 0 || t1 < t0 || t1 - t0 > Q || t1 > p.tokens) return;  // flagged by chunk_state
    const int L = static_cast<int>(t1 - t0);
    const int64_t gs = static_cast<int64_t>(p.G) * N, g0 = static_cast<int64_t>(g) * N;
    stage_rows<kCbThreads>(&sm.cm[0][0], N + 8, static_cast<const __nv_bfloat16 *>(p.C), t0, gs, g0, Q, L, N);
    stage_rows<kCbThreads>(&sm.bm[0][0], N + 8, static_cast<const __nv_bfloat16 *>(p.B), t0, gs, g0, Q, L, N);
    cp_async_wait_all();
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, q = lane & 3, mi = lane >> 3;
    const int mt_end = (L + 15) / 16;  // row tiles holding tokens
    float *cb = p.ws_cb + (static_cast<int64_t>(c) * p.G + g) * cb_tiles(Q) * 256;
    float *cbd = p.ws_cbd + (static_cast<int64_t>(c) * p.G + g) * Q;
    for (int tile = warp; tile < mt_end * (mt_end + 1) / 2; tile += kCbThreads / 32) {
        int m = 0;
        while ((m + 1) * (m + 2) / 2 <= tile) ++m;
        const int j = tile - m * (m + 1) / 2;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int k0 = 0; k0 < N; k0 += 16) {
            uint32_t a[4], b[4];
            // C: matrices (t 0-7 | 8-15) x (n 0-7 | 8-15) of cm
            ldsm_x4(a, &sm.cm[16 * m + (lane & 7) + (mi & 1) * 8][k0 + (mi >> 1) * 8]);
            // B[k = n][col = s] = bm[s][n]: matrices (n 0-7 | 8-15) x (s 0-7 | 8-15)
            ldsm_x4(b, &sm.bm[16 * j + (lane & 7) + (mi >> 1) * 8][k0 + (mi & 1) * 8]);
            mma_bf16(acc[0], a, b[0], b[1]);
            mma_bf16(acc[1], a, b[2], b[3]);
        }
        float4 *o = reinterpret_cast<float4 *>(cb + static_cast<int64_t>(tile) * 256 + lane * 8);
        o[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        o[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
        if (j == m) {  // the diagonal: (row gq, col 2q + e) of columns 0-7, (row gq + 8, col 8 + 2q + e) of 8-15
            if (gq == 2 * q) cbd[16 * m + gq] = acc[0][0], cbd[16 * m + gq + 8] = acc[1][2];
            if (gq == 2 * q + 1) cbd[16 * m + gq] = acc[0][1], cbd[16 * m + gq + 8] = acc[1][3];
        }
    }
}

// ---------------------------------------------------------------------------
// Stage 5: the chunk scan, one CTA per (head, chunk); warp w takes the row
// tiles w and Q/16 - 1 - w (16 tokens each) so that the causal work is
// balanced.  Per row tile:
//   Y1 = C . S_in^T, scaled by exp(cs_t)   (S_in as bf16 high + low parts,
//                                           split once by the state pass)
//   Y2 = sum over column tiles j of W_j . x_j, W[t][s] = (C . B^T)
//        exp(cs_t - cs_s) dt'_s for s < t, as bf16 high + low parts; for a
//        tile that lies wholly before the rows the decay factors through the
//        tile's last token r, exp(cs_t - cs_r) exp(cs_r - cs_s), both at most
//        1 (cs only decreases), the second with dt'_s kept per column (E)
//   y = Y1 + Y2 + ((C_t . B_t) dt'_t + D) x_t   (the diagonal in fp32: it can
//        cancel D for every dim row of a token), gated by silu(z).
// ---------------------------------------------------------------------------
template <int Q, int P, int N>
struct ChunkScanSmem {
    __nv_bfloat16 xs[Q][P + 8];  // x rows, xs[s][p]
    __nv_bfloat16 zy[Q][P + 8];  // z rows, replaced row by row by y before its store
    __nv_bfloat16 ss[P][N + 8];  // entering state, bf16 high part, ss[p][n]
    __nv_bfloat16 sl[P][N + 8];  // and the bf16 low part of what is left
    float cs[Q];                 // inclusive cumulative sums of a, times log2(e)
    float dtp[Q];                // dt'
    float cbd[Q];                // C_t . B_t
    float E[Q];                  // exp(cs_r - cs_s) dt'_s, r the last token of s's 16-token tile
};

template <int Q, int P, int N>
__global__ void __launch_bounds__(Q, 2) ssd_chunk_scan_kernel(const SsdParams p) {
    static_assert(P == 64 && Q % 64 == 0, "tiling");
    constexpr int kThreads = Q;  // Q / 32 warps
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<ChunkScanSmem<Q, P, N> *>(smem_raw);
    const int h = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
    const int g = h / p.hpg;
    const int64_t t0 = meta_at(p.cu_chunk, c, p.meta_i64), t1 = meta_at(p.cu_chunk, c + 1, p.meta_i64);
    if (t0 < 0 || t1 < t0 || t1 - t0 > Q || t1 > p.tokens) return;  // flagged by chunk_state
    const int L = static_cast<int>(t1 - t0);
    if (L == 0) return;
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, q = lane & 3, mi = lane >> 3;
    const __nv_bfloat16 *Cg = static_cast<const __nv_bfloat16 *>(p.C);
    // C fragments (A of C . S_in^T) of row tile m, straight from global memory
    uint32_t cf[N / 16][4];
    auto load_cf = [&](int m) {
        const int ta = 16 * m + gq, tc = ta + 8;
        const unsigned int *ra = reinterpret_cast<const unsigned int *>(Cg + ((t0 + ta) * p.G + g) * N);
        const unsigned int *rc = reinterpret_cast<const unsigned int *>(Cg + ((t0 + tc) * p.G + g) * N);
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
            const int n2 = 8 * ks + q;  // (16 ks + 2 q) / 2
            cf[ks][0] = ta < L ? __ldg(ra + n2) : 0u;
            cf[ks][1] = tc < L ? __ldg(rc + n2) : 0u;
            cf[ks][2] = ta < L ? __ldg(ra + n2 + 4) : 0u;
            cf[ks][3] = tc < L ? __ldg(rc + n2 + 4) : 0u;
        }
    };
    load_cf(warp);  // the first row tile's, in flight during the staging below
    stage_rows<kThreads>(&sm.xs[0][0], P + 8, static_cast<const __nv_bfloat16 *>(p.x), t0,
                         static_cast<int64_t>(p.H) * P, static_cast<int64_t>(h) * P, Q, L, P);
    if (p.z)
        stage_rows<kThreads>(&sm.zy[0][0], P + 8, static_cast<const __nv_bfloat16 *>(p.z), t0,
                             static_cast<int64_t>(p.H) * P, static_cast<int64_t>(h) * P, Q, L, P);
    const int64_t ch = ws_unit(p, c, h);
    {  // the entering state's parts, from the canonical order into padded rows
        const unsigned char *slot = reinterpret_cast<const unsigned char *>(p.ws_state + ch * P * N);
        for (int i = tid; i < 2 * P * N / 8; i += kThreads) {
            const int part = i / (P * N / 8), b = (i % (P * N / 8)) * 16;
            const int pp = (b / (N * 16)) * 8 + (b % 128) / 16, n8 = ((b / 128) % (N / 8)) * 8;
            cp_async16(part ? &sm.sl[pp][n8] : &sm.ss[pp][n8], slot + part * (P * N * 2) + b, true);
        }
    }
    constexpr float kLog2e = 1.4426950408889634f;
    for (int t = tid; t < Q; t += kThreads) {
        sm.cs[t] = p.ws_acs[ch * Q + t] * kLog2e;
        sm.dtp[t] = p.ws_dtp[ch * Q + t];
        sm.cbd[t] = p.ws_cbd[(static_cast<int64_t>(c) * p.G + g) * Q + t];
    }
    __syncthreads();
    for (int t = tid; t < Q; t += kThreads) sm.E[t] = t < L ? ex2_fast(sm.cs[t | 15] - sm.cs[t]) * sm.dtp[t] : 0.f;
    cp_async_wait_all();
    __syncthreads();

    const float *cbg = p.ws_cb + (static_cast<int64_t>(c) * p.G + g) * cb_tiles(Q) * 256;
    const float Dh = p.D ? p.D[h] : 0.f;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        const int m = half ? Q / 16 - 1 - warp : warp;
        if (16 * m >= L) continue;
        const int ta = 16 * m + gq, tc = ta + 8;  // the two rows this lane holds
        float acc[P / 8][4];
#pragma unroll
        for (int j = 0; j < P / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        // y from the entering state, C . S_in^T (the high parts for every p-tile,
        // then the low parts: no accumulator is used twice in a row)
        if (half) load_cf(m);
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
                for (int j = 0; j < P / 8; j += 2) {
                    // S_in^T: B[k = n][col = p] = ss[p][n]: matrices (n 0-7 | 8-15) x (p-tile j | j+1)
                    uint32_t b[4];
                    ldsm_x4(b, part ? &sm.sl[8 * j + (lane & 7) + (mi >> 1) * 8][16 * ks + (mi & 1) * 8]
                                    : &sm.ss[8 * j + (lane & 7) + (mi >> 1) * 8][16 * ks + (mi & 1) * 8]);
                    mma_bf16(acc[j], cf[ks], b[0], b[1]);
                    mma_bf16(acc[j + 1], cf[ks], b[2], b[3]);
                }
            }
        }
        const float csa = sm.cs[ta], csc = sm.cs[tc];
        const float ea = exp2f(csa), ec = exp2f(csc);
#pragma unroll
        for (int j = 0; j < P / 8; ++j) acc[j][0] *= ea, acc[j][1] *= ea, acc[j][2] *= ec, acc[j][3] *= ec;
        // strictly causal part, 16 tokens s at a time; the next tile's C . B^T
        // is loaded while this one is used
        const float4 *row_tiles = reinterpret_cast<const float4 *>(cbg + static_cast<int64_t>(cb_tile(m, 0)) * 256) +
                                  lane * 2;
        float4 v0 = __ldg(row_tiles), v1 = __ldg(row_tiles + 1), w0 = v0, w1 = v1;
        if (m > 0) w0 = __ldg(row_tiles + 64), w1 = __ldg(row_tiles + 65);
        for (int js = 0; js <= m; ++js) {
            const float cb[2][4] = {{v0.x, v0.y, v0.z, v0.w}, {v1.x, v1.y, v1.z, v1.w}};
            v0 = w0, v1 = w1;  // two tiles ahead in flight
            if (js + 2 <= m) w0 = __ldg(row_tiles + (js + 2) * 64), w1 = __ldg(row_tiles + (js + 2) * 64 + 1);
            uint32_t mf[4], ml[4];
            if (js < m) {  // the tile lies wholly before the rows: decays through its last token
                const float r = sm.cs[16 * js + 15];
                const float Ra = ex2_fast(csa - r), Rc = ex2_fast(csc - r);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const float2 e = *reinterpret_cast<const float2 *>(&sm.E[16 * js + 8 * jj + 2 * q]);
                    split_bf16(cb[jj][0] * Ra * e.x, cb[jj][1] * Ra * e.y, &mf[2 * jj], &ml[2 * jj]);
                    split_bf16(cb[jj][2] * Rc * e.x, cb[jj][3] * Rc * e.y, &mf[2 * jj + 1], &ml[2 * jj + 1]);
                }
            } else {  // the diagonal tile: W[t][s] for s < t, one exponential each
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int s0 = 16 * js + 8 * jj + 2 * q, s1 = s0 + 1;
                    const float d0 = sm.dtp[s0], d1 = sm.dtp[s1], e0 = sm.cs[s0], e1 = sm.cs[s1];
                    const float m00 = s0 < ta ? cb[jj][0] * ex2_fast(csa - e0) * d0 : 0.f;
                    const float m01 = s1 < ta ? cb[jj][1] * ex2_fast(csa - e1) * d1 : 0.f;
                    const float m10 = s0 < tc ? cb[jj][2] * ex2_fast(csc - e0) * d0 : 0.f;
                    const float m11 = s1 < tc ? cb[jj][3] * ex2_fast(csc - e1) * d1 : 0.f;
                    split_bf16(m00, m01, &mf[2 * jj], &ml[2 * jj]);
                    split_bf16(m10, m11, &mf[2 * jj + 1], &ml[2 * jj + 1]);
                }
            }
            // (A operand order: {rows g, k 2q}, {rows g+8, k 2q}, {rows g, k 2q+8}, {rows g+8, k 2q+8})
            uint32_t bx[P / 16][4];
#pragma unroll
            for (int j = 0; j < P / 8; j += 2) {
                // X: B[k = s][col = p] = xs[s][p]: matrices (s 0-7 | 8-15) x (p-tile j | j+1), transposed
                ldsm_x4_trans(bx[j / 2], &sm.xs[16 * js + (lane & 7) + (mi & 1) * 8][8 * j + (mi >> 1) * 8]);
                mma_bf16(acc[j], mf, bx[j / 2][0], bx[j / 2][1]);
                mma_bf16(acc[j + 1], mf, bx[j / 2][2], bx[j / 2][3]);
            }
#pragma unroll
            for (int j = 0; j < P / 8; j += 2) {
                mma_bf16(acc[j], ml, bx[j / 2][0], bx[j / 2][1]);
                mma_bf16(acc[j + 1], ml, bx[j / 2][2], bx[j / 2][3]);
            }
        }
        // epilogue: + ((C_t . B_t) dt'_t + D) x_t in fp32, gate, store
        const float wa = fmaf(sm.cbd[ta], sm.dtp[ta], Dh), wc = fmaf(sm.cbd[tc], sm.dtp[tc], Dh);
#pragma unroll
        for (int j = 0; j < P / 8; ++j) {
            const int pp = 8 * j + 2 * q;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int t = r ? tc : ta;
                if (t >= L) continue;
                const uint32_t xb = *reinterpret_cast<const uint32_t *>(&sm.xs[t][pp]);
                const float wd = r ? wc : wa;
                float v0 = fmaf(wd, bf16_lo(xb), acc[j][2 * r]);
                float v1 = fmaf(wd, bf16_hi(xb), acc[j][2 * r + 1]);
                uint32_t *zy = reinterpret_cast<uint32_t *>(&sm.zy[t][pp]);
                if (p.z) {
                    const uint32_t zb = *zy;
                    const float z0 = bf16_lo(zb), z1 = bf16_hi(zb);
                    v0 *= __fdividef(z0, 1.f + __expf(-z0));
                    v1 *= __fdividef(z1, 1.f + __expf(-z1));
                }
                *zy = pack_bf16(v0, v1);  // this lane's z element becomes its y element
            }
        }
        // the warp's 16 rows of y, 16 bytes per lane and store
        __syncwarp();
        for (int i = lane; i < 16 * (P / 8); i += 32) {
            const int t = 16 * m + i / (P / 8), k = (i % (P / 8)) * 8;
            if (t < L)
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.y) + ((t0 + t) * p.H + h) * static_cast<int64_t>(P) + k) =
                    *reinterpret_cast<const uint4 *>(&sm.zy[t][k]);
        }
    }
}

// ---------------------------------------------------------------------------
// Launch.
// ---------------------------------------------------------------------------
template <typename K>
static cudaError_t allow_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int Q, int P, int N>
static cudaError_t launch_qpn(const SsdParams &p, cudaStream_t stream) {
    const size_t s1 = sizeof(ChunkStateSmem<Q, P, N>), s4 = sizeof(ChunkCbSmem<Q, N>),
                 s5 = sizeof(ChunkScanSmem<Q, P, N>);
    cudaError_t e;
    if ((e = allow_smem(ssd_chunk_state_kernel<Q, P, N>, s1)) != cudaSuccess) return e;
    if ((e = allow_smem(ssd_chunk_cb_kernel<Q, N>, s4)) != cudaSuccess) return e;
    if ((e = allow_smem(ssd_chunk_scan_kernel<Q, P, N>, s5)) != cudaSuccess) return e;
    const dim3 g1(static_cast<unsigned>(p.H), static_cast<unsigned>(p.nchunks));
    ssd_chunk_state_kernel<Q, P, N><<<g1, kStateThreads, s1, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 g3(static_cast<unsigned>(p.nchunks), static_cast<unsigned>(p.H));
    switch (p.state_dtype) {
    case kF32: ssd_state_pass_kernel<P, N, float><<<g3, kPassThreads, 0, stream>>>(p); break;
    case kF16: ssd_state_pass_kernel<P, N, __half><<<g3, kPassThreads, 0, stream>>>(p); break;
    case kBF16: ssd_state_pass_kernel<P, N, __nv_bfloat16><<<g3, kPassThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 g4(static_cast<unsigned>(p.G), static_cast<unsigned>(p.nchunks));
    ssd_chunk_cb_kernel<Q, N><<<g4, kCbThreads, s4, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ssd_chunk_scan_kernel<Q, P, N><<<g1, Q, s5, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_ssd(const SsdParams &p, cudaStream_t stream) {
    if (p.P != 64) return cudaErrorInvalidValue;
    const int key = p.Q * 1000 + p.N;
    switch (key) {
    case 64 * 1000 + 64: return launch_qpn<64, 64, 64>(p, stream);
    case 64 * 1000 + 128: return launch_qpn<64, 64, 128>(p, stream);
    case 128 * 1000 + 64: return launch_qpn<128, 64, 64>(p, stream);
    case 128 * 1000 + 128: return launch_qpn<128, 64, 128>(p, stream);
    case 256 * 1000 + 64: return launch_qpn<256, 64, 64>(p, stream);
    case 256 * 1000 + 128: return launch_qpn<256, 64, 128>(p, stream);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Library-owned scratch for ssu_ssd_prefill_static: the workspace of one call
// (at most kSsdStaticScratchBytes), a file-scope device array, so that such a
// call allocates nothing.  Nothing in it needs to start at zero: the kernels
// write every part of the workspace before they read it.  Calls that overlap
// in time share it and corrupt each other's results.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_ssd_scratch[kSsdStaticScratchBytes];

cudaError_t ssd_static_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    static std::mutex lock;
    static void *addr[kMaxDevices] = {};
    std::lock_guard<std::mutex> guard(lock);
    if (addr[dev] == nullptr) {  // once per device, with that device current
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ssd_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

}  // namespace ssu
