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
// Three kernels over a caller-owned workspace:
//   chunk_state  one CTA per (head, chunk), on the tensor cores (mma.sync
//                m16n8k16, bf16 operands, fp32 accumulation; operands staged
//                in shared memory in the inputs' own row layout by 16-byte
//                cp.async and read as fragments with ldmatrix): dt', the
//                prefix and suffix sums of a, and Sc = (w x)^T B with
//                w_t = exp(sum_{s>t} a) dt'_t; w x is split into a bf16 high
//                and low part so that Sc keeps ~2^-17 relative precision (the
//                returned states need it);
//   state_pass   one CTA per (run of a sequence's chunks, head): replaces
//                each Sc in the workspace by the chunk's entering state (as
//                bf16 high and low parts, in the operand order of the scan's
//                MMA) and writes the returned states;
//   scan         one CTA per (group, chunk), on the 5th-generation tensor
//                cores with C . B^T kept in tensor memory (ssu_ssd_tc.cu).
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

// Four 8 x 8 b16 matrices from shared memory, transposed; lanes 8i..8i+7
// give the row addresses of matrix i.  Lane l receives rows 2(l%4),
// 2(l%4)+1 of column l/4 of each matrix.
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
// The chunk is staged in parts of QH tokens (128 at most), so that three
// CTAs share an SM.
template <int Q>
__host__ __device__ constexpr int chunk_part() { return Q < 128 ? Q : 128; }

template <int Q, int P, int N>
struct ChunkStateSmem {
    static constexpr int QH = chunk_part<Q>();
    __nv_bfloat16 xs[QH][P + 8];  // x of one part of the chunk, xs[t][p]
    __nv_bfloat16 bs[QH][N + 8];  // B of the chunk's group for the part, bs[t][n]
    float cs[Q];                 // inclusive cumulative sums of a
    float rs[Q];                 // inclusive cumulative sums of a, reversed
    float w[Q];                  // dt', then exp(sum of the later a) dt'
    float tmp[8];
    float mx[2][8];              // per warp: largest |x| and largest dt'
};

constexpr int kStateThreads = 256;

template <int Q, int P, int N>
__global__ void __launch_bounds__(kStateThreads, 3) ssd_chunk_state_kernel(const SsdParams p) {
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
    constexpr int QH = chunk_part<Q>();
    // x and B rows of part pt (tokens pt QH ...), zero from L on
    auto stage_part = [&](int pt) {
        const int Lp = L - pt * QH;
        stage_rows<kStateThreads>(&sm.xs[0][0], P + 8, static_cast<const __nv_bfloat16 *>(p.x), t0 + pt * QH,
                                  static_cast<int64_t>(p.H) * P, static_cast<int64_t>(h) * P, QH, Lp, P);
        stage_rows<kStateThreads>(&sm.bs[0][0], N + 8, static_cast<const __nv_bfloat16 *>(p.B), t0 + pt * QH,
                                  static_cast<int64_t>(p.G) * N, static_cast<int64_t>(g) * N, QH, Lp, N);
    };
    // the first part's x and B rows, in flight while the decays are formed
    stage_part(0);
    float *ws_acs = p.ws_acs + ws_unit(p, c, h) * Q;
    float *ws_dtp = p.ws_dtp + ws_unit(p, c, h) * Q;
    const float Ah = p.A[h];
    float dmax = 0.f;  // largest dt' of this thread's token
    if (tid < Q) {
        const float d = tid < L ? ssd_step(p, t0 + tid, h) : 0.f;
        dmax = d;
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
    uint32_t xm = 0;  // the largest |x| bits, over the parts
    for (int pt = 0; pt < Q / QH; ++pt) {
        if (pt > 0) {
            if (pt * QH >= L) break;  // the rest of the chunk is empty
            __syncthreads();          // every warp is done with the previous part
            stage_part(pt);
            cp_async_wait_all();
            __syncthreads();
        }
        const int kend = min(L, (pt + 1) * QH);
        for (int k0 = pt * QH; k0 < kend; k0 += 16) {
            const int kr = k0 - pt * QH;  // row of the part in shared memory
            // A = (w x)^T: matrices (p 0-7 | 8-15) x (t 0-7 | 8-15) of xs, transposed
            uint32_t ax[4], ahi[4], alo[4];
            ldsm_x4_trans(ax, &sm.xs[kr + (lane & 7) + (mi >> 1) * 8][p0 + (mi & 1) * 8]);
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
                ldsm_x4_trans(bb[j / 2], &sm.bs[kr + (lane & 7) + (mi & 1) * 8][n0 + 8 * j + (mi >> 1) * 8]);
                mma_bf16(acc[j], ahi, bb[j / 2][0], bb[j / 2][1]);
                mma_bf16(acc[j + 1], ahi, bb[j / 2][2], bb[j / 2][3]);
            }
#pragma unroll
            for (int j = 0; j < NT; j += 2) {
                mma_bf16(acc[j], alo, bb[j / 2][0], bb[j / 2][1]);
                mma_bf16(acc[j + 1], alo, bb[j / 2][2], bb[j / 2][3]);
            }
        }
        // the part's largest |x| (rows from L on are zero); bf16 magnitudes
        // compare as unsigned integers
        for (int i = tid; i < QH * (P / 8); i += kStateThreads) {
            const uint4 v = *reinterpret_cast<const uint4 *>(&sm.xs[i / (P / 8)][(i % (P / 8)) * 8]);
            xm = __vmaxu2(xm, __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                       __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
        }
    }
    float *out = p.ws_state + ws_unit(p, c, h) * P * N;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int n = n0 + 8 * j + 2 * q;
        *reinterpret_cast<float2 *>(out + canon<N>(p0 + gq, n)) = make_float2(acc[j][0], acc[j][1]);
        *reinterpret_cast<float2 *>(out + canon<N>(p0 + gq + 8, n)) = make_float2(acc[j][2], acc[j][3]);
    }
    // the largest |x| and dt' of the chunk and head, from which the scan
    // picks the power-of-two scales of its fp16 operands
    float xmax = fmaxf(__uint_as_float(xm << 16), __uint_as_float(xm & 0xffff0000u));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        xmax = fmaxf(xmax, __shfl_xor_sync(0xffffffffu, xmax, off));
        dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, off));
    }
    if (lane == 0) sm.mx[0][warp] = xmax, sm.mx[1][warp] = dmax;
    __syncthreads();
    if (tid == 0) {
        float a = 0.f, b = 0.f;
        for (int i = 0; i < kStateThreads / 32; ++i) a = fmaxf(a, sm.mx[0][i]), b = fmaxf(b, sm.mx[1][i]);
        *reinterpret_cast<float4 *>(p.ws_scl + ws_unit(p, c, h) * 4) = make_float4(a, b, 0.f, 0.f);
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
// Launch.
// ---------------------------------------------------------------------------
template <typename K>
static cudaError_t allow_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int Q, int P, int N>
static cudaError_t launch_qpn(const SsdParams &p, cudaStream_t stream) {
    const size_t s1 = sizeof(ChunkStateSmem<Q, P, N>);
    cudaError_t e;
    if ((e = allow_smem(ssd_chunk_state_kernel<Q, P, N>, s1)) != cudaSuccess) return e;
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
    return launch_ssd_scan_tc(p, stream);
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
