// fa_bwd.cu -- backward kernels (placeholder until the recompute kernels land).
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
cudaError_t launch_backward(const BwdLaunch&, bool, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa
