// ssu_shadow.cu -- the low-precision read copy of state rows.
//
// Article "ReplaySSM: Cache SSM Inputs, Not State", section 低精度读写分离:
// the steps that do not fold read the checkpoint only to form the output, so
// they can read a low-precision copy of it while the recurrence keeps the
// full-precision checkpoint; the copy never feeds the recurrence.  This
// kernel builds the copy of rows written by other means; a fold of the
// replay kernel rewrites the copy of the rows it folds with the same
// arithmetic (shadow_scale / e4m3_code in ssu_device.cuh).
//
// One warp per state row: the row's largest magnitude (an exact maximum),
// its scale amax / 448 and factor 448 / amax in fp32, then each element's
// code (E4M3); or the row scale, each block's scale code and the elements'
// E2M1 codes (NVFP4, dstate a multiple of 32).
#include "ssu_device.cuh"

namespace ssu {

template <typename TS>
__global__ void __launch_bounds__(256)
    ssu_shadow_refresh_kernel(const TS *state, int64_t rows, int dstate, int format, void *shadow, float *scale) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
        const TS *row = state + r * dstate;
        if (format == kShadowF16) {
            __half *out = static_cast<__half *>(shadow) + r * dstate;
            for (int n = lane; n < dstate; n += 32) out[n] = __float2half_rn(to_float(row[n]));
            continue;
        }
        if (format == kShadowNVFP4) {
            // lane l takes elements 32 j + l: a block of 16 is half a warp
            float amax = 0.f;
            for (int n = lane; n < dstate; n += 32) amax = fmaxf(amax, fabsf(to_float(row[n])));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float sr = nvfp4_row_scale(amax);
            float *rec = scale + r * nvfp4_scale_words(dstate);
            unsigned char *bcodes = reinterpret_cast<unsigned char *>(rec + 1);
            if (lane == 0) rec[0] = sr;
            unsigned char *out = static_cast<unsigned char *>(shadow) + r * (dstate / 2);
            for (int n0 = 0; n0 < dstate; n0 += 32) {
                const float v = to_float(row[n0 + lane]);
                float bmax = fabsf(v);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
                const unsigned int bc = nvfp4_block_code(bmax, sr);
                const float den = __fmul_rn(e4m3_value(bc), sr);
                const float q = den > 0.f ? __fdiv_rn(v, den) : 0.f;
                const float q1 = __shfl_down_sync(0xffffffffu, q, 1);
                if ((lane & 1) == 0) out[(n0 + lane) / 2] = static_cast<unsigned char>(e2m1x2_code(q, q1));
                if ((lane & 15) == 0) bcodes[(n0 + lane) / 16] = static_cast<unsigned char>(bc);
            }
            continue;
        }
        float amax = 0.f;
        for (int n = lane; n < dstate; n += 32) amax = fmaxf(amax, fabsf(to_float(row[n])));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float f = shadow_factor_of(amax);
        if (lane == 0) scale[r] = shadow_scale_of(amax);
        unsigned char *out = static_cast<unsigned char *>(shadow) + r * dstate;
        for (int n = lane; n < dstate; n += 32) out[n] = e4m3_code(__fmul_rn(to_float(row[n]), f));
    }
}

cudaError_t launch_shadow_refresh(const void *state, int state_dtype, int64_t rows, int dstate, int format,
                                  void *shadow, float *scale, cudaStream_t stream) {
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    const unsigned g = static_cast<unsigned>(blocks);
    switch (state_dtype) {
    case kF32:
        ssu_shadow_refresh_kernel<float><<<g, 256, 0, stream>>>(static_cast<const float *>(state), rows, dstate,
                                                                format, shadow, scale);
        break;
    case kF16:
        ssu_shadow_refresh_kernel<__half><<<g, 256, 0, stream>>>(static_cast<const __half *>(state), rows, dstate,
                                                                 format, shadow, scale);
        break;
    case kBF16:
        ssu_shadow_refresh_kernel<__nv_bfloat16><<<g, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(state), rows, dstate, format, shadow, scale);
        break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace ssu
