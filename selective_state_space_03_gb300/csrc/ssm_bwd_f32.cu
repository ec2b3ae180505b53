// Backward kernel with float32 I/O.
#include "ssm_bwd2_impl.cuh"

namespace ssm {
cudaError_t launch_bwd_f32(const BwdLaunch& L, cudaStream_t stream) {
    return L.kd == 2 ? launch_bwd2_io<float>(L, stream) : launch_bwd_io<float>(L, stream);
}
cudaError_t launch_bwd_carry_f32(const BwdLaunch& L, cudaStream_t stream) {
    return launch_bwd_carry_io<float>(L, stream);
}
}  // namespace ssm
