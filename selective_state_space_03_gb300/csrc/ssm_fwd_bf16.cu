// Forward kernels with bf16 I/O (float32 state and arithmetic).
#include "ssm_fwd_impl.cuh"

namespace ssm {
cudaError_t launch_fwd_bf16(const FwdLaunch& L, int mode, cudaStream_t stream) {
    return launch_fwd_io<__nv_bfloat16>(L, mode, stream);
}
}  // namespace ssm
