// ssu_replay_bf16.cu -- the checkpoint + buffer kernels (ssu_replay.cuh) for
// bf16 operands.
#include "ssu_replay.cuh"

namespace ssu {
template cudaError_t launch_replay_io<kBF16>(int, int, const KParams &, int64_t, cudaStream_t);
}  // namespace ssu
