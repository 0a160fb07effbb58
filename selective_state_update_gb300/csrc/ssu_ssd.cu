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
//   chunk_state  one CTA per (chunk, head): dt', the cumulative sums, and
//                Sc as a tensor-core product (mma.sync bf16, fp32
//                accumulation) of the decay-weighted x -- split into a bf16
//                high and low part so the state keeps ~2^-17 relative
//                precision -- with B; Sc goes to the workspace;
//   state_pass   one CTA per (sequence run, head): walks the run's chunks,
//                replaces each Sc in the workspace by the chunk's entering
//                state and writes the states the call returns;
//   chunk_scan   one CTA per (chunk, head, 64-token block): y from the
//                entering state (C . S_in^T) and the causal C . B^T products
//                times the decays and dt' x, on the tensor cores (bf16
//                operands, fp32 accumulation; the entering state and the
//                decayed C . B^T weights as bf16 high + low parts).
#include <cstdint>

#include "ssu_device.cuh"

namespace ssu {

// ---------------------------------------------------------------------------
// Tensor-core helpers: m16n8k16, A row-major (16 x 16), B column-major
// (16 x 8), fp32 accumulators.  Fragment of lane l (g = l / 4, q = l % 4):
// A regs {A[g][2q..2q+1]}, {A[g+8][2q..]}, {A[g][2q+8..]}, {A[g+8][2q+8..]};
// B regs {B[2q..2q+1][g]}, {B[2q+8..2q+9][g]}; D {D[g][2q..2q+1]},
// {D[g+8][2q..2q+1]}.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// dt' of token t, head h: dt (+ bias), softplus, clamped to [lo, hi].
__device__ __forceinline__ float ssd_step(const SsdParams &p, int64_t t, int h) {
    const int64_t i = t * p.H + h;
    float v = p.dt_dtype == kF32 ? static_cast<const float *>(p.dt)[i]
                                 : bits_to_float(static_cast<const unsigned short *>(p.dt)[i], p.dt_dtype);
    v = processed_step(v, p.dt_bias ? p.dt_bias[h] : 0.f, p.softplus);
    return fminf(fmaxf(v, p.dt_lo), p.dt_hi);
}

// Inclusive prefix sums of v[0..n) in shared memory by a 128-thread block
// (n <= 256), in place; `tmp` holds 8 floats.
__device__ void block_scan_256(float *v, int n, float *tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // each thread two consecutive values
    float a = 2 * tid < n ? v[2 * tid] : 0.f;
    float b = 2 * tid + 1 < n ? v[2 * tid + 1] : 0.f;
    b += a;
    float s = b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    if (lane == 31) tmp[warp] = s;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; ++w) base += tmp[w];
    const float excl = base + s - b;  // sum of everything before this thread's pair
    if (2 * tid < n) v[2 * tid] = excl + a;
    if (2 * tid + 1 < n) v[2 * tid + 1] = excl + b;
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Stage 1-2: per (chunk, head) the cumulative sums and the chunk's own state.
// ---------------------------------------------------------------------------
template <int Q, int P, int N>
struct ChunkStateSmem {
    static constexpr int kPad = 8;  // bf16 elements of padding per transposed row
    static constexpr int kT = Q + kPad;
    __nv_bfloat16 xt[P][kT];  // x of the chunk, transposed: xt[p][t]
    __nv_bfloat16 bt[N][kT];  // B of the chunk's group, transposed: bt[n][t]
    float a[Q];               // A dt'
    float cs[Q];              // inclusive cumulative sums of a
    float rs[Q];              // inclusive cumulative sums of a reversed
    float w[Q];               // dt', then exp(sum of the later a) dt'
    float tmp[8];
};

template <int Q, int P, int N>
__global__ void __launch_bounds__(128) ssd_chunk_state_kernel(const SsdParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<ChunkStateSmem<Q, P, N> *>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int g = h / p.hpg;
    const int64_t t0 = meta_at(p.cu_chunk, c, p.meta_i64), t1 = meta_at(p.cu_chunk, c + 1, p.meta_i64);
    const int L = static_cast<int>(t1 - t0);
    if (c == 0 && h == 0 && !p.intermediate) {  // every sequence's last chunk must name a chunk
        for (int64_t s = tid; s < p.nseq; s += 128) {
            const int64_t lc = meta_at(p.last_chunk, s, p.meta_i64);
            if (lc < 0 || lc >= p.nchunks) flag(p.status, kDevBadEntry);
        }
    }
    if (t0 < 0 || t1 < t0 || t1 - t0 > Q || t1 > p.tokens) {
        if (tid == 0) flag(p.status, kDevBadSeqlen);
        return;
    }
    float *ws_acs = p.ws_acs + (static_cast<int64_t>(c) * p.H + h) * Q;
    float *ws_dtp = p.ws_dtp + (static_cast<int64_t>(c) * p.H + h) * Q;
    // dt', a = A dt'
    const float Ah = p.A[h];
    for (int t = tid; t < Q; t += 128) {
        const float d = t < L ? ssd_step(p, t0 + t, h) : 0.f;
        ws_dtp[t] = d;
        sm.w[t] = d;
        sm.a[t] = t < L ? Ah * d : 0.f;
        sm.cs[t] = sm.a[t];
    }
    __syncthreads();
    for (int t = tid; t < Q; t += 128) sm.rs[t] = t < L ? sm.a[L - 1 - t] : 0.f;  // a reversed
    __syncthreads();
    block_scan_256(sm.cs, Q, sm.tmp);
    // rs[i] = sum of a over the last i + 1 tokens, summed from the end so the
    // decays of recent tokens carry no cancellation
    block_scan_256(sm.rs, Q, sm.tmp);
    for (int t = tid; t < Q; t += 128) {
        ws_acs[t] = sm.cs[t];
        const float later = t + 1 < L ? sm.rs[L - 2 - t] : 0.f;  // sum_{s>t} a_s
        sm.w[t] = t < L ? expf(later) * sm.w[t] : 0.f;
    }
    if (tid == 0) p.ws_dec[static_cast<int64_t>(c) * p.H + h] = L > 0 ? expf(sm.rs[L - 1]) : 1.f;
    // x (transposed) and B (transposed) of the chunk, zero beyond L
    for (int i = tid; i < Q * (P / 8); i += 128) {
        const int t = i / (P / 8), p8 = (i % (P / 8)) * 8;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (t < L) u = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.x) +
                                                         ((t0 + t) * p.H + h) * static_cast<int64_t>(P) + p8);
        const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
        for (int k = 0; k < 8; ++k) sm.xt[p8 + k][t] = e[k];
    }
    for (int i = tid; i < Q * (N / 8); i += 128) {
        const int t = i / (N / 8), n8 = (i % (N / 8)) * 8;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (t < L) u = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.B) +
                                                         ((t0 + t) * p.G + g) * static_cast<int64_t>(N) + n8);
        const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
        for (int k = 0; k < 8; ++k) sm.bt[n8 + k][t] = e[k];
    }
    __syncthreads();
    // Sc[p][n] = sum_t (w_t x[t][p]) B[t][n]: M = P rows, N columns, K = t.
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, q = lane & 3;
    for (int pb = warp * 16; pb < P; pb += 64) {
        float acc[N / 8][4];
#pragma unroll
        for (int j = 0; j < N / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        for (int k0 = 0; k0 < L; k0 += 16) {
            uint32_t ahi[4], alo[4];
            const int r0 = pb + gq, r1 = pb + gq + 8, c0 = k0 + 2 * q, c1 = k0 + 2 * q + 8;
            const float w00 = sm.w[c0], w01 = sm.w[c0 + 1], w10 = sm.w[c1], w11 = sm.w[c1 + 1];
            split_bf16(__bfloat162float(sm.xt[r0][c0]) * w00, __bfloat162float(sm.xt[r0][c0 + 1]) * w01, &ahi[0], &alo[0]);
            split_bf16(__bfloat162float(sm.xt[r1][c0]) * w00, __bfloat162float(sm.xt[r1][c0 + 1]) * w01, &ahi[1], &alo[1]);
            split_bf16(__bfloat162float(sm.xt[r0][c1]) * w10, __bfloat162float(sm.xt[r0][c1 + 1]) * w11, &ahi[2], &alo[2]);
            split_bf16(__bfloat162float(sm.xt[r1][c1]) * w10, __bfloat162float(sm.xt[r1][c1 + 1]) * w11, &ahi[3], &alo[3]);
#pragma unroll
            for (int j = 0; j < N / 8; ++j) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sm.bt[8 * j + gq][c0]);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sm.bt[8 * j + gq][c1]);
                mma_bf16(acc[j], ahi, b0, b1);
                mma_bf16(acc[j], alo, b0, b1);
            }
        }
        float *out = p.ws_state + ((static_cast<int64_t>(c) * p.H + h) * P) * N;
#pragma unroll
        for (int j = 0; j < N / 8; ++j) {
            const int n = 8 * j + 2 * q;
            *reinterpret_cast<float2 *>(out + (pb + gq) * N + n) = make_float2(acc[j][0], acc[j][1]);
            *reinterpret_cast<float2 *>(out + (pb + gq + 8) * N + n) = make_float2(acc[j][2], acc[j][3]);
        }
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

template <int P, int N, typename TS>
__global__ void __launch_bounds__(256) ssd_state_pass_kernel(const SsdParams p) {
    const int c0 = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int64_t b = meta_at(p.seq_idx, c0, p.meta_i64);
    if (c0 > 0 && meta_at(p.seq_idx, c0 - 1, p.meta_i64) == b) return;  // not the first chunk of a run
    if (b < 0 || b >= p.nseq) {
        if (tid == 0) flag(p.status, kDevBadEntry);
        return;
    }
    constexpr int kPer = P * N / (256 * 4);  // float4 per thread
    float4 S[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int64_t e = (static_cast<int64_t>(k) * 256 + tid) * 4;
        S[k] = p.init ? load_state4<TS>(p.init, ((b * p.H + h) * P) * static_cast<int64_t>(N) + e)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int c = c0; c < p.nchunks; ++c) {
        if (c > c0 && meta_at(p.seq_idx, c, p.meta_i64) != b) break;
        float *ws = p.ws_state + ((static_cast<int64_t>(c) * p.H + h) * P) * N;
        const float dec = p.ws_dec[static_cast<int64_t>(c) * p.H + h];
        float4 sc[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) sc[k] = *reinterpret_cast<const float4 *>(ws + (k * 256 + tid) * 4);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            *reinterpret_cast<float4 *>(ws + (k * 256 + tid) * 4) = S[k];  // the state entering chunk c
            S[k] = make_float4(fmaf(dec, S[k].x, sc[k].x), fmaf(dec, S[k].y, sc[k].y), fmaf(dec, S[k].z, sc[k].z),
                               fmaf(dec, S[k].w, sc[k].w));
        }
        if (p.intermediate) {
#pragma unroll
            for (int k = 0; k < kPer; ++k)
                store_state4(static_cast<TS *>(p.states) + ((static_cast<int64_t>(c) * p.H + h) * P) * N +
                                 (k * 256 + tid) * 4, S[k]);
        } else {
            for (int64_t s = 0; s < p.nseq; ++s) {
                if (meta_at(p.last_chunk, s, p.meta_i64) != c) continue;
#pragma unroll
                for (int k = 0; k < kPer; ++k)
                    store_state4(static_cast<TS *>(p.states) + ((s * p.H + h) * P) * static_cast<int64_t>(N) +
                                     (k * 256 + tid) * 4, S[k]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Stages 4-5: the chunk scan, one CTA per (chunk, head, 64-token block).
// ---------------------------------------------------------------------------
template <int Q, int P, int N>
struct ChunkScanSmem {
    static constexpr int kPadN = 8, kPadT = 8;
    __nv_bfloat16 cm[64][N + kPadN];  // C of the block's tokens, cm[t][n]
    __nv_bfloat16 bm[Q][N + kPadN];   // B of the chunk's tokens up to the block's end, bm[s][n]
    __nv_bfloat16 xt[P][Q + kPadT];   // x transposed, xt[p][s]
    __nv_bfloat16 sin[P][N + kPadN];  // entering state, bf16 high part, sin[p][n]
    __nv_bfloat16 slo[P][N + kPadN];  // and the bf16 low part of what is left
    float cs[Q], dtp[Q];
};

template <int Q, int P, int N>
__global__ void __launch_bounds__(128) ssd_chunk_scan_kernel(const SsdParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    auto &sm = *reinterpret_cast<ChunkScanSmem<Q, P, N> *>(smem_raw);
    const int c = blockIdx.x, h = blockIdx.y, blk = blockIdx.z, tid = threadIdx.x;
    const int g = h / p.hpg;
    const int64_t t0 = meta_at(p.cu_chunk, c, p.meta_i64), t1 = meta_at(p.cu_chunk, c + 1, p.meta_i64);
    if (t0 < 0 || t1 < t0 || t1 - t0 > Q || t1 > p.tokens) return;  // flagged by chunk_state
    const int L = static_cast<int>(t1 - t0);
    const int tb0 = blk * 64;
    if (tb0 >= L) return;
    const int send = min(L, tb0 + 64);  // tokens s < send can reach this block
    const float *wcs = p.ws_acs + (static_cast<int64_t>(c) * p.H + h) * Q;
    const float *wdt = p.ws_dtp + (static_cast<int64_t>(c) * p.H + h) * Q;
    for (int t = tid; t < Q; t += 128) {
        sm.cs[t] = wcs[t];
        sm.dtp[t] = wdt[t];
    }
    for (int i = tid; i < 64 * (N / 8); i += 128) {
        const int t = i / (N / 8), n8 = (i % (N / 8)) * 8;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (tb0 + t < L)
            u = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.C) +
                                                 ((t0 + tb0 + t) * p.G + g) * static_cast<int64_t>(N) + n8);
        *reinterpret_cast<uint4 *>(&sm.cm[t][n8]) = u;
    }
    for (int i = tid; i < send * (N / 8); i += 128) {
        const int s = i / (N / 8), n8 = (i % (N / 8)) * 8;
        *reinterpret_cast<uint4 *>(&sm.bm[s][n8]) = *reinterpret_cast<const uint4 *>(
            static_cast<const __nv_bfloat16 *>(p.B) + ((t0 + s) * p.G + g) * static_cast<int64_t>(N) + n8);
    }
    for (int i = tid; i < Q * (P / 8); i += 128) {
        const int s = i / (P / 8), p8 = (i % (P / 8)) * 8;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (s < send)
            u = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.x) +
                                                 ((t0 + s) * p.H + h) * static_cast<int64_t>(P) + p8);
        const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
        for (int k = 0; k < 8; ++k) sm.xt[p8 + k][s] = e[k];
    }
    {
        const float *ws = p.ws_state + ((static_cast<int64_t>(c) * p.H + h) * P) * N;
        for (int i = tid; i < P * N / 4; i += 128) {
            const float4 v = *reinterpret_cast<const float4 *>(ws + i * 4);
            const int pp = (i * 4) / N, n = (i * 4) % N;
            uint2 hi, lo;
            split_bf16(v.x, v.y, &hi.x, &lo.x);
            split_bf16(v.z, v.w, &hi.y, &lo.y);
            *reinterpret_cast<uint2 *>(&sm.sin[pp][n]) = hi;
            *reinterpret_cast<uint2 *>(&sm.slo[pp][n]) = lo;
        }
    }
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, q = lane & 3;
    const int tb = tb0 + warp * 16;  // this warp's 16 tokens
    if (tb >= L) return;
    // C fragments of the warp's rows for every k-step over n
    uint32_t cf[N / 16][4];
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks) {
        const int r0 = warp * 16 + gq, n0 = ks * 16 + 2 * q;
        cf[ks][0] = *reinterpret_cast<const uint32_t *>(&sm.cm[r0][n0]);
        cf[ks][1] = *reinterpret_cast<const uint32_t *>(&sm.cm[r0 + 8][n0]);
        cf[ks][2] = *reinterpret_cast<const uint32_t *>(&sm.cm[r0][n0 + 8]);
        cf[ks][3] = *reinterpret_cast<const uint32_t *>(&sm.cm[r0 + 8][n0 + 8]);
    }
    // y from the entering state: (C . S_in^T) scaled by exp(cs_t), S_in as
    // the sum of its bf16 high and low parts
    float yacc[P / 8][4];
#pragma unroll
    for (int j = 0; j < P / 8; ++j) yacc[j][0] = yacc[j][1] = yacc[j][2] = yacc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < N / 16; ++ks) {
#pragma unroll
        for (int j = 0; j < P / 8; ++j) {
            const int r = 8 * j + gq, n0 = ks * 16 + 2 * q;
            mma_bf16(yacc[j], cf[ks], *reinterpret_cast<const uint32_t *>(&sm.sin[r][n0]),
                     *reinterpret_cast<const uint32_t *>(&sm.sin[r][n0 + 8]));
            mma_bf16(yacc[j], cf[ks], *reinterpret_cast<const uint32_t *>(&sm.slo[r][n0]),
                     *reinterpret_cast<const uint32_t *>(&sm.slo[r][n0 + 8]));
        }
    }
    const int ta = tb + gq, tc = tb + gq + 8;  // the two rows this lane holds
    const float ea = expf(sm.cs[min(ta, Q - 1)]), ec = expf(sm.cs[min(tc, Q - 1)]);
#pragma unroll
    for (int j = 0; j < P / 8; ++j) {
        yacc[j][0] *= ea;
        yacc[j][1] *= ea;
        yacc[j][2] *= ec;
        yacc[j][3] *= ec;
    }
    // causal part, 16 tokens s at a time
    for (int sb = 0; sb <= tb; sb += 16) {
        float cb[2][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) cb[jj][0] = cb[jj][1] = cb[jj][2] = cb[jj][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int s = sb + 8 * jj + gq;
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sm.bm[s][ks * 16 + 2 * q]);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sm.bm[s][ks * 16 + 2 * q + 8]);
                mma_bf16(cb[jj], cf[ks], b0, b1);
            }
        }
        // M[t][s] = CB exp(cs_t - cs_s) dt'_s for s <= t (and s < L), else 0,
        // as a bf16 high and low part: the diagonal term alone can nearly
        // cancel D x_t, so M keeps ~2^-17 relative precision
        uint32_t mf[4], ml[4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int s0 = sb + 8 * jj + 2 * q, s1 = s0 + 1;
            const float ws0 = s0 < send ? sm.dtp[s0] : 0.f, ws1 = s1 < send ? sm.dtp[s1] : 0.f;
            const float csa = sm.cs[min(ta, Q - 1)], csc = sm.cs[min(tc, Q - 1)];
            const float m00 = s0 <= ta ? cb[jj][0] * expf(csa - sm.cs[s0]) * ws0 : 0.f;
            const float m01 = s1 <= ta ? cb[jj][1] * expf(csa - sm.cs[s1]) * ws1 : 0.f;
            const float m10 = s0 <= tc ? cb[jj][2] * expf(csc - sm.cs[s0]) * ws0 : 0.f;
            const float m11 = s1 <= tc ? cb[jj][3] * expf(csc - sm.cs[s1]) * ws1 : 0.f;
            split_bf16(m00, m01, &mf[2 * jj], &ml[2 * jj]);
            split_bf16(m10, m11, &mf[2 * jj + 1], &ml[2 * jj + 1]);
        }
        // A operand order: {rows g, k 2q}, {rows g+8, k 2q}, {rows g, k 2q+8},
        // {rows g+8, k 2q+8} -- the order mf and ml are filled in
#pragma unroll
        for (int j = 0; j < P / 8; ++j) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&sm.xt[8 * j + gq][sb + 2 * q]);
            const uint32_t b1 = *reinterpret_cast<const uint32_t *>(&sm.xt[8 * j + gq][sb + 2 * q + 8]);
            mma_bf16(yacc[j], mf, b0, b1);
            mma_bf16(yacc[j], ml, b0, b1);
        }
    }
    // epilogue: + D x, gate, store
    const float Dh = p.D ? p.D[h] : 0.f;
#pragma unroll
    for (int j = 0; j < P / 8; ++j) {
        const int pp = 8 * j + 2 * q;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int t = half ? tc : ta;
            if (t >= L) continue;
            const int64_t o = ((t0 + t) * p.H + h) * static_cast<int64_t>(P) + pp;
            const uint32_t xb = *reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(p.x) + o);
            float v0 = fmaf(Dh, bf16_lo(xb), yacc[j][2 * half]);
            float v1 = fmaf(Dh, bf16_hi(xb), yacc[j][2 * half + 1]);
            if (p.z) {
                const uint32_t zb = *reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(p.z) + o);
                v0 *= silu_gate(bf16_lo(zb), 1);
                v1 *= silu_gate(bf16_hi(zb), 1);
            }
            *reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(p.y) + o) = pack_bf16(v0, v1);
        }
    }
}

// ---------------------------------------------------------------------------
// Launch.
// ---------------------------------------------------------------------------
template <int Q, int P, int N>
static cudaError_t launch_qpn(const SsdParams &p, cudaStream_t stream) {
    const size_t s1 = sizeof(ChunkStateSmem<Q, P, N>), s3 = sizeof(ChunkScanSmem<Q, P, N>);
    cudaError_t e = cudaFuncSetAttribute(ssd_chunk_state_kernel<Q, P, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(s1));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(ssd_chunk_scan_kernel<Q, P, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(s3));
    if (e != cudaSuccess) return e;
    const dim3 g1(static_cast<unsigned>(p.nchunks), static_cast<unsigned>(p.H));
    ssd_chunk_state_kernel<Q, P, N><<<g1, 128, s1, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    switch (p.state_dtype) {
    case kF32: ssd_state_pass_kernel<P, N, float><<<g1, 256, 0, stream>>>(p); break;
    case kF16: ssd_state_pass_kernel<P, N, __half><<<g1, 256, 0, stream>>>(p); break;
    case kBF16: ssd_state_pass_kernel<P, N, __nv_bfloat16><<<g1, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 g3(static_cast<unsigned>(p.nchunks), static_cast<unsigned>(p.H), Q / 64);
    ssd_chunk_scan_kernel<Q, P, N><<<g3, 128, s3, stream>>>(p);
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

}  // namespace ssu
