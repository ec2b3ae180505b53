// Middle pass of the chunked forward when it has many chunks: the start state of
// every chunk in one sweep over the chunk carries, linear in their number.
//
// Pass 1 leaves, per chain and chunk j < nchunk - 1, the chunk's end state from a
// zero start S_j and its delta sum. The chunk maps compose as
//   H_j = exp(A * sum of delta over chunk j) * H_{j-1} + S_j,   H_{-1} = h0,
// the chunk-boundary state carried forward as the ruDNN page's `chunk_kda` carries
// its state from chunk to chunk. Pass 2 of chunk k needs H_{k-1}; folding it
// there costs k carries per chunk, O(nchunk^2) in all, which dominates shapes
// with hundreds or thousands of chunks. This kernel folds them once per chain
// and overwrites S_j with H_j, so pass 2 loads one state.
//
// One thread per (chain, group of 4 states); the loads of NB chunks are issued
// together, ahead of the dependent updates.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kNB = 8;      // chunks whose carries are loaded together

__global__ void __launch_bounds__(128) fwd_carry_scan_kernel(const FwdLaunch p) {
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t chain = gid >> 2;                 // b * D + d
    if (chain >= p.B * p.D) return;
    const int s0 = int(gid & 3) * 4;
    const int64_t b = chain / p.D, d = chain - b * p.D;
    const int64_t nprev = p.nchunk - 1;
    const float4 a = *reinterpret_cast<const float4*>(p.A + d * kDS + s0);
    const float A2[4] = {a.x * kLog2e, a.y * kLog2e, a.z * kLog2e, a.w * kLog2e};
    float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.h0 != nullptr) h = *reinterpret_cast<const float4*>(p.h0 + chain * kDS + s0);
    for (int64_t j0 = 0; j0 < nprev; j0 += kNB) {
        float sd[kNB];
        float4 S[kNB];
#pragma unroll
        for (int u = 0; u < kNB; ++u) {
            sd[u] = 0.f;
            S[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j0 + u < nprev) {
                const int64_t row = (b * nprev + j0 + u) * p.D + d;
                sd[u] = p.ws_Sd[row];
                S[u] = *reinterpret_cast<const float4*>(p.ws_S + row * kDS + s0);
            }
        }
#pragma unroll
        for (int u = 0; u < kNB; ++u) {
            if (j0 + u >= nprev) break;
            h.x = fmaf(ex2(A2[0] * sd[u]), h.x, S[u].x);
            h.y = fmaf(ex2(A2[1] * sd[u]), h.y, S[u].y);
            h.z = fmaf(ex2(A2[2] * sd[u]), h.z, S[u].z);
            h.w = fmaf(ex2(A2[3] * sd[u]), h.w, S[u].w);
            const int64_t row = (b * nprev + j0 + u) * p.D + d;
            *reinterpret_cast<float4*>(p.ws_S + row * kDS + s0) = h;      // start state of chunk j + 1
        }
    }
}

}  // namespace

cudaError_t launch_fwd_carry_scan(const FwdLaunch& L, cudaStream_t stream) {
    const int64_t threads = L.B * L.D * 4;
    const int64_t blocks = (threads + 127) / 128;
    if (blocks > int64_t(0x7fffffff)) return cudaErrorInvalidValue;
    fwd_carry_scan_kernel<<<unsigned(blocks), 128, 0, stream>>>(L);
    return cudaGetLastError();
}

}  // namespace ssm
