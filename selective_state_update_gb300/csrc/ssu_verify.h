// ssu_verify.h -- launcher of the speculative-decoding kernels on the
// checkpoint + buffer form (ssu_replay_verify).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "ssu_internal.h"

namespace ssu {

// `batch` sequences of `T` draft tokens each (rows b * T + k of the row
// operands); the fold launch, then the verify launch, on `stream`.
cudaError_t launch_verify(int state_dtype, const KParams &p, int64_t batch, int T, cudaStream_t stream);

}  // namespace ssu
