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
//   verify   one CTA per (sequence, head, 64 dim rows): the state is carried
//            in registers from the checkpoint (as stored) through the
//            committed entries and then the drafts, each draft's y read
//            after its own step; the drafts are appended as entries
//            c .. c+T-1 and count_out = c (nothing committed).
// The page evaluates the drafts as two masked GEMMs over the window; the
// state carried through the window in registers reads the same bytes (the
// checkpoint once, each entry once) and gives the drafts' outputs in order,
// which at a few drafts per sequence needs no tensor cores.  Four threads
// share a state row (dstate / 4 columns each).
#include <cstdint>

#include "ssu_device.cuh"
#include "ssu_verify.h"

namespace ssu {

constexpr int kVerifyRows = 64;             // dim rows per CTA
constexpr int kVerifyThreads = 4 * kVerifyRows;

__device__ __forceinline__ float load_small(const void *base, int64_t i, int dtype) {
    return dtype == kF32 ? static_cast<const float *>(base)[i]
                         : bits_to_float(static_cast<const unsigned short *>(base)[i], dtype);
}

__device__ __forceinline__ void store_ts(float *o, float v) { *o = v; }
__device__ __forceinline__ void store_ts(__half *o, float v) { *o = __float2half_rn(v); }
__device__ __forceinline__ void store_ts(__nv_bfloat16 *o, float v) { *o = __float2bfloat16_rn(v); }

// The sequence's slot, its committed count, and whether it is a pad slot;
// false (flagged) for a bad table entry, slot or count.
__device__ __forceinline__ bool verify_sequence(const KParams &p, int64_t b, int64_t *slot, int *c, bool *pad) {
    if (!table_slot(p, p.rd, b, 0, b, b, slot)) return false;
    if (!slot_ok(p, *slot)) return false;
    *pad = *slot == p.pad;
    *c = *pad ? 0 : p.cnt_in[b];
    if (*c < 0 || *c >= p.rlen) {
        flag(p.status, kDevBadCount);
        return false;
    }
    return true;
}

// One buffered entry j applied to this thread's NPT columns of row `row`.
template <int NPT>
__device__ __forceinline__ void apply_entry(const KParams &p, int64_t slot, int j, int h, int g, int row, int q,
                                            float Ah, float *s) {
    const int64_t e = ((slot * p.rlen + j) * p.H + h) * static_cast<int64_t>(p.P) + row;
    const float dj = p.dtbuf[e];
    const float dA = decay(Ah, dj);
    const float dx = dj * load_small(p.xbuf, e, p.io_dtype);
    const int64_t be = ((slot * p.rlen + j) * p.G + g) * static_cast<int64_t>(p.N) + q * NPT;
#pragma unroll
    for (int i = 0; i < NPT; ++i) s[i] = fmaf(s[i], dA, dx * load_small(p.Bbuf, be + i, p.io_dtype));
}

template <typename TS, int NPT>
__global__ void __launch_bounds__(kVerifyThreads) ssu_verify_fold_kernel(const KParams p, int T) {
    const int64_t b = blockIdx.x;
    const int h = blockIdx.y, g = h / p.heads_per_group;
    const int row = blockIdx.z * kVerifyRows + threadIdx.x / 4, q = threadIdx.x & 3;
    int64_t slot;
    int c;
    bool pad;
    if (!verify_sequence(p, b, &slot, &c, &pad)) return;  // flagged (again) by the verify launch
    if (pad || c + 2 * T < p.rlen || row >= p.P) return;   // no flush here
    TS *srow = static_cast<TS *>(p.state) + ((slot * p.H + h) * static_cast<int64_t>(p.P) + row) * p.N + q * NPT;
    float s[NPT];
#pragma unroll
    for (int i = 0; i < NPT; ++i) s[i] = to_float(srow[i]);
    const float Ah = p.A[h];
    for (int j = 0; j < c; ++j) apply_entry<NPT>(p, slot, j, h, g, row, q, Ah, s);
#pragma unroll
    for (int i = 0; i < NPT; ++i) store_ts(srow + i, s[i]);
}

template <typename TS, int NPT>
__global__ void __launch_bounds__(kVerifyThreads) ssu_verify_kernel(const KParams p, int T) {
    const int64_t b = blockIdx.x;
    const int h = blockIdx.y, g = h / p.heads_per_group;
    const int row = blockIdx.z * kVerifyRows + threadIdx.x / 4, q = threadIdx.x & 3;
    const bool active = row < p.P;  // the four threads of a row agree
    int64_t slot;
    int c;
    bool pad;
    if (!verify_sequence(p, b, &slot, &c, &pad)) return;
    const bool fold = !pad && c + 2 * T >= p.rlen;
    if (fold) c = 0;
    if (h == 0 && blockIdx.z == 0 && threadIdx.x == 0) p.cnt_out[b] = c;
    // the checkpoint as stored (after the fold launch), then the committed entries
    float s[NPT];
    const TS *srow =
        static_cast<const TS *>(p.state) + ((slot * p.H + h) * static_cast<int64_t>(p.P) + row) * p.N + q * NPT;
#pragma unroll
    for (int i = 0; i < NPT; ++i) s[i] = (pad || !active) ? 0.f : to_float(srow[i]);
    const float Ah = p.A[h];
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
    const float Dh = p.D ? p.D[h] : 0.f;
    if (active)
        for (int j = 0; j < c; ++j) apply_entry<NPT>(p, slot, j, h, g, row, q, Ah, s);
    // the drafts in order, each read out after its own step and appended
    for (int k = 0; k < T; ++k) {
        const int64_t r = b * T + k;
        float part = 0.f, d = 0.f, xv = 0.f;
        if (active) {
            d = processed_step(load_small(p.dt, r * p.dts[0] + h * p.dts[1] + row * p.dts[2], p.dt_dtype), bias,
                               p.softplus);
            xv = load_small(p.x, r * p.xs[0] + h * p.xs[1] + row * p.xs[2], p.io_dtype);
            const float dA = decay(Ah, d), dx = d * xv;
            const int64_t bo = r * p.Bs[0] + g * p.Bs[1], co = r * p.Cs[0] + g * p.Cs[1];
#pragma unroll
            for (int i = 0; i < NPT; ++i) {
                const int n = q * NPT + i;
                s[i] = fmaf(s[i], dA, dx * load_small(p.B, bo + n * p.Bs[2], p.io_dtype));
                part = fmaf(s[i], load_small(p.C, co + n * p.Cs[2], p.io_dtype), part);
            }
        }
        const float sum = row_sum<4>(part);
        if (!active) continue;
        if (q == 0) {
            const float z = p.z ? load_small(p.z, r * p.zs[0] + h * p.zs[1] + row * p.zs[2], p.io_dtype) : 0.f;
            store_small(p.y, r * p.ys[0] + h * p.ys[1] + row * p.ys[2], p.io_dtype,
                        output(sum, Dh, xv, silu_gate(z, p.z != nullptr)));
        }
        if (pad) continue;
        const int64_t e = ((slot * p.rlen + c + k) * p.H + h) * static_cast<int64_t>(p.P) + row;
        if (q == 0) {  // x keeps its bits, the processed step is stored in fp32
            if (p.io_dtype == kF32)
                static_cast<float *>(p.xbuf)[e] = xv;
            else
                static_cast<unsigned short *>(p.xbuf)[e] =
                    static_cast<const unsigned short *>(p.x)[r * p.xs[0] + h * p.xs[1] + row * p.xs[2]];
            p.dtbuf[e] = d;
        }
        if (h % p.heads_per_group == 0 && row == 0) {  // B once per group: the first head's first row
            const int64_t be = ((slot * p.rlen + c + k) * p.G + g) * static_cast<int64_t>(p.N) + q * NPT;
            const int64_t bo = r * p.Bs[0] + g * p.Bs[1];
#pragma unroll
            for (int i = 0; i < NPT; ++i) {
                const int64_t src = bo + (q * NPT + i) * p.Bs[2];
                if (p.io_dtype == kF32)
                    static_cast<float *>(p.Bbuf)[be + i] = static_cast<const float *>(p.B)[src];
                else
                    static_cast<unsigned short *>(p.Bbuf)[be + i] = static_cast<const unsigned short *>(p.B)[src];
            }
        }
    }
}

template <typename TS, int NPT>
static cudaError_t launch_verify_t(const KParams &p, int64_t batch, int T, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(batch), static_cast<unsigned>(p.H),
                    static_cast<unsigned>((p.P + kVerifyRows - 1) / kVerifyRows));
    ssu_verify_fold_kernel<TS, NPT><<<grid, kVerifyThreads, 0, stream>>>(p, T);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ssu_verify_kernel<TS, NPT><<<grid, kVerifyThreads, 0, stream>>>(p, T);
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
