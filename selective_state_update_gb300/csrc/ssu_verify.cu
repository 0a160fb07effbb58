// ssu_verify.cu -- speculative decoding on the checkpoint + buffer form.
//
// Article "ReplaySSM: Cache SSM Inputs, Not State", section 投机解码回滚:
// the T draft tokens of a sequence are appended to its input buffer after
// the c committed entries, every draft is verified against the same
// checkpoint and buffer under a causal mask, and committing the accepted
// prefix is moving the buffer's count -- there is no per-draft state
// snapshot and no state restore.  The flush fires one window early, when
// c + 2T >= L, so that the next step always finds T free entries.
//
// Two launches:
//   fold     one CTA per (sequence, head, 64 dim rows), only for sequences
//            whose flush fires: the committed entries are applied to the
//            checkpoint in order (fp32) and the checkpoint is written once.
//            It runs on its own launch because the drafts' B, which a group
//            of heads shares, takes the place of entries that the group's
//            other heads fold.
//   verify   one CTA per (sequence, head, 64 dim rows): every draft is read
//            out against the checkpoint (as stored) and the window, without
//            forming a state; the drafts are appended as entries c .. c+T-1
//            and count_out = c (nothing committed).
// Readout of draft k, with M = c + k the last step it sees (steps m < c are
// the committed entries, m >= c the drafts), a_m = exp(A dt'_m) and
// g_{i:M} = a_i ... a_M (g_{M+1:M} = 1):
//     y_k = g_{0:M} (S_ckpt . C_k) + sum_{m <= M} g_{m+1:M} dt'_m x_m (B_m . C_k) + D x_k
// (the unrolled recurrence of section 核心做法; the causal mask is m <= M).
// The page forms the two sums as masked GEMMs over the window; at a few
// drafts per sequence they are T dot products per state row (S_ckpt . C_k)
// and (c + T) x T dot products per CTA (B_m . C_k), then a walk over the
// window per (row, draft) -- no tensor cores, and no state kept in registers
// once the dots are taken.  Four threads share a state row (dstate / 4
// columns each, in interleaved groups of four); the entries' and drafts'
// operands are staged in shared memory once per CTA.
#include <cstdint>
#include <type_traits>

#include "ssu_device.cuh"
#include "ssu_verify.h"

namespace ssu {

constexpr int kVerifyRows = 64;             // dim rows per CTA
constexpr int kVerifyThreads = 4 * kVerifyRows;

// Element i of an array of dtype IO: its stored bits (16-bit types
// zero-extended), its value, and a store of stored bits.  IO is a template
// argument: the staging code is compiled once per operand dtype and chosen
// once per CTA.
template <int IO>
__device__ __forceinline__ uint32_t io_bits(const void *base, int64_t i) {
    if constexpr (IO == kF32)
        return __float_as_uint(static_cast<const float *>(base)[i]);
    else
        return static_cast<const unsigned short *>(base)[i];
}
template <int IO>
__device__ __forceinline__ float io_value(uint32_t bits) {
    if constexpr (IO == kF32)
        return __uint_as_float(bits);
    else if constexpr (IO == kBF16)
        return __uint_as_float(bits << 16);
    else
        return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}
template <int IO>
__device__ __forceinline__ float io_load(const void *base, int64_t i) { return io_value<IO>(io_bits<IO>(base, i)); }
template <int IO>
__device__ __forceinline__ void io_store_bits(void *base, int64_t i, uint32_t v) {
    if constexpr (IO == kF32)
        static_cast<uint32_t *>(base)[i] = v;
    else
        static_cast<unsigned short *>(base)[i] = static_cast<unsigned short>(v);
}
// A run-time dtype of the operands as a template argument.
template <typename F>
__device__ __forceinline__ void with_io(int dtype, F &&f) {
    if (dtype == kF32)
        f(std::integral_constant<int, kF32>{});
    else if (dtype == kBF16)
        f(std::integral_constant<int, kBF16>{});
    else
        f(std::integral_constant<int, kF16>{});
}

__device__ __forceinline__ void store_ts(float *o, float v) { *o = v; }
__device__ __forceinline__ void store_ts(__half *o, float v) { *o = __float2half_rn(v); }
__device__ __forceinline__ void store_ts(__nv_bfloat16 *o, float v) { *o = __float2bfloat16_rn(v); }

// The sequence's slot, its committed count, and whether it is a pad slot;
// false (flagged) for a bad table entry, slot or count.
__device__ __forceinline__ bool verify_sequence(const KParams &p, int64_t b, int64_t *slot, int *c, bool *pad) {
    const int cb = p.cnt_in[b];  // in flight beside the table lookup (count_in holds one entry per sequence)
    if (!table_slot(p, p.rd, b, 0, b, b, slot)) return false;
    if (!slot_ok(p, *slot)) return false;
    *pad = *slot == p.pad;
    *c = *pad ? 0 : cb;
    if (*c < 0 || *c >= p.rlen) {
        flag(p.status, kDevBadCount);
        return false;
    }
    return true;
}

// Shared-memory staging of one CTA: the buffered entries' B (fp32, per
// entry) and their x, dt' for the CTA's 64 rows; the drafts' B, C and x, dt,
// z for the rows.  Everything is loaded once, cooperatively and coalesced,
// before the state walks through it.
struct VerifyStage {
    float *eB;   // [L][N]
    float *ex;   // [L][64]
    float *ed;   // [L][64]
    float *dB;   // [T][N]
    float *dC;   // [T][N]
    float *dx;   // [T][64]
    float *dd;   // [T][64] processed steps
    float *dz;   // [T][64]
    uint32_t *rB;  // [T][N] the drafts' B as stored bits, for the append
    uint32_t *rx;  // [T][64] the drafts' x as stored bits
    float *bc;   // [c + T][T] B_m . C_k (entry m < c, else draft m - c)
    float *us;   // [T][64] S_ckpt row . C_k
    float *ga;   // [c + T][64] decay exp(A dt'_m) of each step and row
    float *te;   // [c + T][64] input term dt'_m x_m of each step and row
};

__host__ __device__ inline size_t verify_smem_bytes(int L, int T, int N) {
    return sizeof(float) * (static_cast<size_t>(L) * N + 2 * L * kVerifyRows + 3 * static_cast<size_t>(T) * N +
                            5 * T * kVerifyRows + static_cast<size_t>(L + T) * T +
                            2 * static_cast<size_t>(L + T) * kVerifyRows);
}

__device__ __forceinline__ VerifyStage verify_stage(float *smem, int L, int T, int N) {
    VerifyStage st;
    st.eB = smem;
    st.ex = st.eB + L * N;
    st.ed = st.ex + L * kVerifyRows;
    st.dB = st.ed + L * kVerifyRows;
    st.dC = st.dB + T * N;
    st.dx = st.dC + T * N;
    st.dd = st.dx + T * kVerifyRows;
    st.dz = st.dd + T * kVerifyRows;
    st.rB = reinterpret_cast<uint32_t *>(st.dz + T * kVerifyRows);
    st.rx = st.rB + T * N;
    st.us = reinterpret_cast<float *>(st.rx + T * kVerifyRows);
    st.bc = st.us + T * kVerifyRows;
    st.ga = st.bc + (L + T) * T;
    st.te = st.ga + (L + T) * kVerifyRows;
    return st;
}

// Entries 0 .. c-1 of (slot, group g): their B.
template <int IO, int N>
__device__ __forceinline__ void stage_entry_B(const KParams &p, const VerifyStage &st, int64_t slot, int c, int g) {
    const int64_t eb0 = (slot * p.rlen * p.G + g) * static_cast<int64_t>(N);  // entry 0's B
    for (int i = threadIdx.x; i < c * N; i += kVerifyThreads) {
        const int j = i / N, n = i % N;
        st.eB[i] = io_load<IO>(p.Bbuf, eb0 + static_cast<int64_t>(j) * p.G * N + n);
    }
}

// Entries 0 .. c-1 of (slot, head h): their x and dt' rows row0 .. row0+63.
template <int IO>
__device__ __forceinline__ void stage_entry_rows(const KParams &p, const VerifyStage &st, int64_t slot, int c, int h,
                                                 int row0) {
    const int64_t e0 = (slot * p.rlen * p.H + h) * static_cast<int64_t>(p.P) + row0;  // entry 0's row row0
    for (int i = threadIdx.x; i < c * kVerifyRows; i += kVerifyThreads) {
        const int j = i / kVerifyRows, r = i % kVerifyRows;
        if (row0 + r >= p.P) continue;
        const int64_t e = e0 + static_cast<int64_t>(j) * p.H * p.P + r;
        st.ed[i] = p.dtbuf[e];
        st.ex[i] = io_load<IO>(p.xbuf, e);
    }
}

// Columns of a row: thread q of the row's four owns the groups of four
// columns 16 i + 4 q .. + 3 (i < NPT / 4), so that the four threads read
// neighbouring 16-byte pieces.
__device__ __forceinline__ int col_of(int i4, int q) { return 16 * i4 + 4 * q; }

// The committed entries applied to this thread's columns of its row.
template <int NPT>
__device__ __forceinline__ void apply_entries(const KParams &p, const VerifyStage &st, int c, int r, int q, float Ah,
                                              float *s) {
    for (int j = 0; j < c; ++j) {
        const float dj = st.ed[j * kVerifyRows + r];
        const float dA = decay_inline(Ah, dj);
        const float dx = dj * st.ex[j * kVerifyRows + r];
        const float *Bj = st.eB + j * p.N;
#pragma unroll
        for (int i4 = 0; i4 < NPT / 4; ++i4) {
            const float4 bv = *reinterpret_cast<const float4 *>(Bj + col_of(i4, q));
            s[4 * i4] = fmaf(s[4 * i4], dA, dx * bv.x);
            s[4 * i4 + 1] = fmaf(s[4 * i4 + 1], dA, dx * bv.y);
            s[4 * i4 + 2] = fmaf(s[4 * i4 + 2], dA, dx * bv.z);
            s[4 * i4 + 3] = fmaf(s[4 * i4 + 3], dA, dx * bv.w);
        }
    }
}

// This thread's columns of a state row (`row` points at the row's start).
template <typename TS, int NPT>
__device__ __forceinline__ void load_state_part(const TS *row, int q, float *s) {
#pragma unroll
    for (int i4 = 0; i4 < NPT / 4; ++i4) {
        const TS *src = row + col_of(i4, q);
        if constexpr (sizeof(TS) == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src);
            s[4 * i4] = v.x, s[4 * i4 + 1] = v.y, s[4 * i4 + 2] = v.z, s[4 * i4 + 3] = v.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[4 * i4 + e] = to_float(src[e]);
        }
    }
}

template <typename TS, int NPT>
__device__ __forceinline__ void store_state_part(TS *row, int q, const float *s) {
#pragma unroll
    for (int i4 = 0; i4 < NPT / 4; ++i4) {
        TS *dst = row + col_of(i4, q);
        if constexpr (sizeof(TS) == 4) {
            *reinterpret_cast<float4 *>(dst) = make_float4(s[4 * i4], s[4 * i4 + 1], s[4 * i4 + 2], s[4 * i4 + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) store_ts(dst + e, s[4 * i4 + e]);
        }
    }
}

template <typename TS, int NPT>
__global__ void __launch_bounds__(kVerifyThreads, 2) ssu_verify_fold_kernel(const KParams p, int T) {
    extern __shared__ __align__(16) float vsmem[];
    const int64_t b = blockIdx.x;
    const int h = blockIdx.y, g = h / p.heads_per_group, row0 = blockIdx.z * kVerifyRows;
    const int r = threadIdx.x / 4, row = row0 + r, q = threadIdx.x & 3;
    int64_t slot;
    int c;
    bool pad;
    if (!verify_sequence(p, b, &slot, &c, &pad)) return;  // flagged (again) by the verify launch
    if (pad || c + 2 * T < p.rlen) return;                 // no flush here
    const VerifyStage st = verify_stage(vsmem, p.rlen, T, p.N);
    with_io(p.io_dtype, [&](auto io) {
        stage_entry_B<decltype(io)::value, 4 * NPT>(p, st, slot, c, g);
        stage_entry_rows<decltype(io)::value>(p, st, slot, c, h, row0);
    });
    __syncthreads();
    if (row >= p.P) return;
    TS *srow = static_cast<TS *>(p.state) + ((slot * p.H + h) * static_cast<int64_t>(p.P) + row) * p.N;
    float s[NPT];
    load_state_part<TS, NPT>(srow, q, s);
    apply_entries<NPT>(p, st, c, r, q, p.A[h], s);
    store_state_part<TS, NPT>(srow, q, s);
}

// One CTA per (sequence, group, 64 dim rows) walks the group's heads: the
// group's entries' B, the drafts' B and C and the (c + T) T dots B_m . C_k are
// staged and formed once; per head, the entries' and drafts' rows, the
// appends, the step terms, S_ckpt . C_k and the walks, the head's state row
// part loaded while its rows are staged.  Four CTAs per SM (measured: 0.517
// ms per call against 0.558 ms at three and 0.680 ms at two with the next
// head's state prefetched into registers): the warps, not the registers,
// hide each head's chain.
template <typename TS, int NPT>
__global__ void __launch_bounds__(kVerifyThreads, 4) ssu_verify_kernel(const KParams p, int T, int fold_here) {
    extern __shared__ __align__(16) float vsmem[];
    constexpr int N = 4 * NPT;
    const int64_t b = blockIdx.x;
    const int g = blockIdx.y, row0 = blockIdx.z * kVerifyRows;
    const int hpg = p.heads_per_group, h0 = g * hpg;
    const int r = threadIdx.x / 4, row = row0 + r, q = threadIdx.x & 3;
    const bool active = row < p.P;  // the four threads of a row agree
    int64_t slot;
    int c;
    bool pad;
    if (!verify_sequence(p, b, &slot, &c, &pad)) return;
    const bool fold = !pad && c + 2 * T >= p.rlen;
    // With fold_here (dim within one 64-row block, so this CTA owns every row
    // of the group's heads) a flush folds the c committed entries here, head
    // by head, before the readout; otherwise the fold launch has done it.
    const int cf = fold && fold_here ? c : 0;  // committed entries folded here
    if (fold) c = 0;
    if (g == 0 && blockIdx.z == 0 && threadIdx.x == 0) p.cnt_out[b] = c;
    const VerifyStage st = verify_stage(vsmem, p.rlen, T, N);
    const bool live = !pad && active;
    auto state_row = [&](int h) {
        return static_cast<const TS *>(p.state) + ((slot * p.H + h) * static_cast<int64_t>(p.P) + row) * N;
    };
    // the first head's state row part in flight while the group's operands are staged
    float s[NPT];
    if (live) {
        load_state_part<TS, NPT>(state_row(h0), q, s);
    } else {
#pragma unroll
        for (int i = 0; i < NPT; ++i) s[i] = 0.f;
    }
    with_io(p.io_dtype, [&](auto io) {
        constexpr int IO = decltype(io)::value;
        stage_entry_B<IO, N>(p, st, slot, c + cf, g);  // (one of c and cf is 0)
        for (int i = threadIdx.x; i < T * N; i += kVerifyThreads) {
            const int k = i / N, n = i % N;
            const int64_t rr = b * T + k;
            const uint32_t bb = io_bits<IO>(p.B, rr * p.Bs[0] + g * p.Bs[1] + n * p.Bs[2]);
            st.dC[i] = io_load<IO>(p.C, rr * p.Cs[0] + g * p.Cs[1] + n * p.Cs[2]);
            st.dB[i] = io_value<IO>(bb);
            st.rB[i] = bb;
        }
        __syncthreads();
        // the drafts' B become entries c .. c+T-1 of the group (once: the
        // group's first 64-row block)
        if (!pad && blockIdx.z == 0) {
            const int64_t eb = ((slot * p.rlen + c) * p.G + g) * static_cast<int64_t>(N);
            for (int i = threadIdx.x; i < T * N; i += kVerifyThreads) {
                const int k = i / N, n = i % N;
                io_store_bits<IO>(p.Bbuf, eb + static_cast<int64_t>(k) * p.G * N + n, st.rB[i]);
            }
        }
    });
    // B_m . C_k for every step m <= c + k that draft k sees, one warp per dot
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < (c + T) * T; i += kVerifyThreads / 32) {
        const int m = i / T, k = i % T;
        if (m > c + k) continue;  // masked: the same for the whole warp
        const float *Bm = m < c ? st.eB + m * N : st.dB + (m - c) * N;
        const float *Ck = st.dC + k * N;
        float v = 0.f;
#pragma unroll
        for (int n = lane; n < N; n += 32) v = fmaf(Bm[n], Ck[n], v);
        v = row_sum<32>(v);
        if (lane == 0) st.bc[i] = v;
    }
    for (int j = 0; j < hpg; ++j) {
        const int h = h0 + j;
        // this head's rows of the entries and the drafts
        const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
        with_io(p.io_dtype, [&](auto io) {
            constexpr int IO = decltype(io)::value;
            stage_entry_rows<IO>(p, st, slot, c + cf, h, row0);
            for (int i = threadIdx.x; i < T * kVerifyRows; i += kVerifyThreads) {
                const int k = i / kVerifyRows, rw = i % kVerifyRows, rrow = row0 + rw;
                if (rrow >= p.P) continue;
                const int64_t rr = b * T + k;
                const int64_t di = rr * p.dts[0] + h * p.dts[1] + rrow * p.dts[2];
                const float dtv = p.dt_dtype == kF32 ? static_cast<const float *>(p.dt)[di]
                                                     : bits_to_float(static_cast<const unsigned short *>(p.dt)[di], p.dt_dtype);
                st.dd[i] = processed_step(dtv, bias, p.softplus);
                const uint32_t xb = io_bits<IO>(p.x, rr * p.xs[0] + h * p.xs[1] + rrow * p.xs[2]);
                st.dx[i] = io_value<IO>(xb);
                st.rx[i] = xb;
                st.dz[i] = p.z ? io_load<IO>(p.z, rr * p.zs[0] + h * p.zs[1] + rrow * p.zs[2]) : 0.f;
            }
            __syncthreads();
            // the drafts' x and dt' become entries c .. c+T-1 of this head
            if (!pad) {
                const int64_t e0 = ((slot * p.rlen + c) * p.H + h) * static_cast<int64_t>(p.P) + row0;
                for (int i = threadIdx.x; i < T * kVerifyRows; i += kVerifyThreads) {
                    const int k = i / kVerifyRows, rw = i % kVerifyRows;
                    if (row0 + rw >= p.P) continue;
                    const int64_t e = e0 + static_cast<int64_t>(k) * p.H * p.P + rw;
                    io_store_bits<IO>(p.xbuf, e, st.rx[i]);
                    p.dtbuf[e] = st.dd[i];
                }
            }
        });
        const float Ah = p.A[h];
        if (cf > 0 && live) {
            // the flush: the committed entries into this head's checkpoint rows
            // (the fold launch's arithmetic), written back as stored; the
            // drafts then read the new checkpoint
            apply_entries<NPT>(p, st, cf, r, q, Ah, s);
            TS *srow = const_cast<TS *>(state_row(h));
            store_state_part<TS, NPT>(srow, q, s);
            if constexpr (sizeof(TS) != 4) {
#pragma unroll
                for (int i = 0; i < NPT; ++i) s[i] = to_float(static_cast<TS>(s[i]));
            }
        }
        // each step's decay and input term per row, shared by the drafts' walks
        for (int i = threadIdx.x; i < (c + T) * kVerifyRows; i += kVerifyThreads) {
            const int m = i / kVerifyRows;
            const bool entry = m < c;
            const float d = entry ? st.ed[i] : st.dd[i - c * kVerifyRows];
            const float xv = entry ? st.ex[i] : st.dx[i - c * kVerifyRows];
            st.ga[i] = decay_inline(Ah, d);
            st.te[i] = d * xv;
        }
        // S_ckpt . C_k of this row, over the row's four threads
        for (int k = 0; k < T; ++k) {
            const float *Ck = st.dC + k * N;
            float part = 0.f;
#pragma unroll
            for (int i4 = 0; i4 < NPT / 4; ++i4) {
                const float4 cv = *reinterpret_cast<const float4 *>(Ck + col_of(i4, q));
                part = fmaf(s[4 * i4], cv.x, part);
                part = fmaf(s[4 * i4 + 1], cv.y, part);
                part = fmaf(s[4 * i4 + 2], cv.z, part);
                part = fmaf(s[4 * i4 + 3], cv.w, part);
            }
            part = row_sum<4>(part);
            if (q == 0) st.us[k * kVerifyRows + r] = part;
        }
        __syncthreads();
        // draft k (thread q of the row takes k = q, q + 4, ...): the walk
        // from step c + k down to step 0 gathers the decayed window sum and
        // g_{0:M}
        if (active) {
            const float Dh = p.D ? p.D[h] : 0.f;
            for (int k = q; k < T; k += 4) {
                float acc = 0.f, gam = 1.f;
                for (int m = c + k; m >= 0; --m) {
                    acc = fmaf(gam, st.te[m * kVerifyRows + r] * st.bc[m * T + k], acc);
                    gam *= st.ga[m * kVerifyRows + r];
                }
                const float sum = fmaf(gam, st.us[k * kVerifyRows + r], acc);
                const int64_t rr = b * T + k;
                store_small(p.y, rr * p.ys[0] + h * p.ys[1] + row * p.ys[2], p.io_dtype,
                            output(sum, Dh, st.dx[k * kVerifyRows + r],
                                   silu_gate(st.dz[k * kVerifyRows + r], p.z != nullptr)));
            }
        }
        __syncthreads();  // the head's stage is read out before the next head's is written
        if (live && j + 1 < hpg) load_state_part<TS, NPT>(state_row(h + 1), q, s);
    }
}

template <typename TS, int NPT>
static cudaError_t launch_verify_t(const KParams &p, int64_t batch, int T, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(batch), static_cast<unsigned>(p.H),
                    static_cast<unsigned>((p.P + kVerifyRows - 1) / kVerifyRows));
    const size_t smem = verify_smem_bytes(p.rlen, T, p.N);
    cudaError_t e;
    if (smem > 48 * 1024) {
        if ((e = cudaFuncSetAttribute(ssu_verify_fold_kernel<TS, NPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem))) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(ssu_verify_kernel<TS, NPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem))) != cudaSuccess)
            return e;
    }
    // One 64-row block: the verify CTAs fold the flushing sequences themselves.
    // More: a separate fold launch first, because the drafts' B, which a
    // group's first block appends, takes the place of entries that the
    // group's other blocks still fold.
    const int fold_here = p.P <= kVerifyRows ? 1 : 0;
    if (!fold_here) {
        ssu_verify_fold_kernel<TS, NPT><<<grid, kVerifyThreads, smem, stream>>>(p, T);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const dim3 ggrid(static_cast<unsigned>(batch), static_cast<unsigned>(p.G),
                     static_cast<unsigned>((p.P + kVerifyRows - 1) / kVerifyRows));
    ssu_verify_kernel<TS, NPT><<<ggrid, kVerifyThreads, smem, stream>>>(p, T, fold_here);
    return cudaGetLastError();
}

template <typename TS>
static cudaError_t launch_verify_n(const KParams &p, int64_t batch, int T, cudaStream_t stream) {
    switch (p.N) {
    case 16: return launch_verify_t<TS, 4>(p, batch, T, stream);
    case 32: return launch_verify_t<TS, 8>(p, batch, T, stream);
    case 64: return launch_verify_t<TS, 16>(p, batch, T, stream);
    case 128: return launch_verify_t<TS, 32>(p, batch, T, stream);
    case 256: return launch_verify_t<TS, 64>(p, batch, T, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_verify(int state_dtype, const KParams &p, int64_t batch, int T, cudaStream_t stream) {
    switch (state_dtype) {
    case kF32: return launch_verify_n<float>(p, batch, T, stream);
    case kF16: return launch_verify_n<__half>(p, batch, T, stream);
    case kBF16: return launch_verify_n<__nv_bfloat16>(p, batch, T, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
