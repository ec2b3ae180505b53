// Backward kernel with bf16 I/O (float32 state, arithmetic and gradients).
#include "ssm_bwd_impl.cuh"

namespace ssm {
cudaError_t launch_bwd_bf16(const BwdLaunch& L, cudaStream_t stream) {
    return launch_bwd_io<__nv_bfloat16>(L, stream);
}
}  // namespace ssm
