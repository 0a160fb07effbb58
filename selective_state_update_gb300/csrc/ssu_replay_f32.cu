// ssu_replay_f32.cu -- the checkpoint + buffer kernels (ssu_replay.cuh) for
// fp32 operands, and the launcher that picks the operand dtype.
#include "ssu_replay.cuh"

namespace ssu {

template cudaError_t launch_replay_io<kF32>(int, int, const KParams &, int64_t, cudaStream_t);

cudaError_t launch_replay(int state_dtype, int lanes, const KParams &p, int64_t batch, cudaStream_t stream) {
    switch (p.io_dtype) {
    case kF32: return launch_replay_io<kF32>(state_dtype, lanes, p, batch, stream);
    case kF16: return launch_replay_io<kF16>(state_dtype, lanes, p, batch, stream);
    case kBF16: return launch_replay_io<kBF16>(state_dtype, lanes, p, batch, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
