// Forward kernels with float32 I/O.
#include "ssm_fwd_impl.cuh"

namespace ssm {
cudaError_t launch_fwd_f32(const FwdLaunch& L, int mode, cudaStream_t stream) {
    return launch_fwd_io<float>(L, mode, stream);
}
}  // namespace ssm
