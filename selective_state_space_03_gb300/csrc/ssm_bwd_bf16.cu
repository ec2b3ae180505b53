// Backward kernel with bf16 I/O (float32 state, arithmetic and gradients).
#include "ssm_bwd2_impl.cuh"

namespace ssm {
cudaError_t launch_bwd_bf16(const BwdLaunch& L, cudaStream_t stream) {
    return L.kd == 2 ? launch_bwd2_io<__nv_bfloat16>(L, stream) : launch_bwd_io<__nv_bfloat16>(L, stream);
}
cudaError_t launch_bwd_carry_bf16(const BwdLaunch& L, cudaStream_t stream) {
    return launch_bwd_carry_io<__nv_bfloat16>(L, stream);
}
}  // namespace ssm
