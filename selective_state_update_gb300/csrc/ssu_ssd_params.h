// ssu_ssd_params.h -- parameters of the packed SSD prefill kernels
// (ssu_ssd_prefill), shared by the C ABI and the kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace ssu {

// Packed variable-length SSD prefill (ssu_ssd_prefill).
struct SsdParams {
    int64_t tokens, nchunks, nseq;
    int32_t H, G, hpg, P, N, Q;
    int32_t dt_dtype, state_dtype, softplus, intermediate, meta_i64;
    float dt_lo, dt_hi;
    const void *x, *dt, *B, *C, *z;  // x, z [tokens, H, P] bf16; dt [tokens, H]; B, C [tokens, G, N] bf16
    const float *A, *D, *dt_bias;
    const void *cu_chunk, *seq_idx, *last_chunk;
    const void *init;                // [nseq, H, P, N] state dtype or NULL
    void *y;                         // [tokens, H, P] bf16
    void *states;                    // [nchunks or nseq, H, P, N] state dtype
    float *ws_state;                 // [H, nchunks, P*N]: chunk states (fp32), then entering states (bf16 hi | lo)
    float *ws_acs, *ws_dtp;          // [H, nchunks, Q]
    float *ws_dec;                   // [H, nchunks]
    float *ws_scl;                   // [H, nchunks, 4]: largest |x| and dt' of the chunk, 2 unused
    int32_t *status;
};
cudaError_t launch_ssd(const SsdParams &p, cudaStream_t stream);
// The chunk scan on the 5th-generation tensor cores (ssu_ssd_tc.cu).
cudaError_t launch_ssd_scan_tc(const SsdParams &p, cudaStream_t stream);

// The library-owned workspace of ssu_ssd_prefill_static on the current
// device: kSsdStaticScratchBytes at *ptr (looked up once per device).
constexpr size_t kSsdStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;
cudaError_t ssd_static_scratch(void **ptr);

}  // namespace ssu
