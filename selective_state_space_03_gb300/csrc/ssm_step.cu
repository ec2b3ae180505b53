// ssm_scan_step: one recurrence step for every (b, d) chain, state updated in place.
//
// Decoding generates one token at a time, so the scan advances by a single step
// per call with the state carried between calls (the ruDNN page's fused
// recurrent decode advances its state the same way, one token per call):
//   h[b,d,s] <- exp(delta[b,d] A[d,s]) h[b,d,s] + delta[b,d] b[b,s] x[b,d]
//   y[b,d]   <- sum_s h[b,d,s] c[b,s]
// It is ssm_scan_fwd with T = 1 and hT written over h0.
//
// The step moves 128 bytes of state per chain in and out and does 16 exp per
// chain, so it is bound by HBM (or by launch latency for small B*D). Layout: 4
// lanes per chain, 4 states per lane in one 16-byte load and store, the readout
// finished with two shuffles; 32 chains per 128-thread CTA. Steps are launched
// with programmatic stream serialization: a step's loads of its own inputs
// overlap the end of the previous step, and only the state load waits for it.
#include "ssm_common.cuh"
#include "ssm_internal.h"
#include "ssm_scan.h"

namespace ssm {
namespace {

struct StepLaunch {
    const void* x;       // (B, D) io
    const void* delta;   // (B, D) io
    const float* A;      // (D, 16)
    const void* b;       // (B, 16) io
    const void* c;       // (B, 16) io
    float* h;            // (B, D, 16), read and written
    void* y;             // (B, D) io
    int64_t B, D;
    bool softplus;       // delta holds raw values
};

template <typename TIO>
__global__ void __launch_bounds__(128) step_kernel(const StepLaunch p) {
    const int64_t gid = int64_t(blockIdx.x) * 128 + threadIdx.x;
    const int64_t chain = gid >> 2;
    const int sg = int(gid & 3), s0 = sg * 4;
    const bool valid = chain < p.B * p.D;       // whole 4-lane groups are valid or not
    // Consecutive steps on a stream are launched as programmatic dependents: let the next
    // step's CTAs start now; they run up to their wait below while this grid finishes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float acc = 0.f;
    float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
    float dl = 0.f, dx = 0.f, bv[4] = {0.f, 0.f, 0.f, 0.f}, cv[4] = {0.f, 0.f, 0.f, 0.f};
    float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {      // this step's inputs, which no earlier step writes
        const int64_t bb = chain / p.D, d = chain - bb * p.D;
        dl = to_f32(static_cast<const TIO*>(p.delta)[chain]);
        if (p.softplus) dl = softplus_f32(dl);
        dx = dl * to_f32(static_cast<const TIO*>(p.x)[chain]);
        load_vals<TIO, 4>(static_cast<const TIO*>(p.b) + bb * kDS + s0, bv);
        load_vals<TIO, 4>(static_cast<const TIO*>(p.c) + bb * kDS + s0, cv);
        a4 = *reinterpret_cast<const float4*>(p.A + d * kDS + s0);
    }
    // the state (and y) belong to the previous step: wait until the grid before this one has
    // completed and its writes are visible (returns at once without such a grid)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (valid) {
        hv = *reinterpret_cast<const float4*>(p.h + chain * kDS + s0);
        hv.x = fmaf(ex2(dl * (a4.x * kLog2e)), hv.x, dx * bv[0]);
        hv.y = fmaf(ex2(dl * (a4.y * kLog2e)), hv.y, dx * bv[1]);
        hv.z = fmaf(ex2(dl * (a4.z * kLog2e)), hv.z, dx * bv[2]);
        hv.w = fmaf(ex2(dl * (a4.w * kLog2e)), hv.w, dx * bv[3]);
        acc = fmaf(hv.x, cv[0], fmaf(hv.y, cv[1], fmaf(hv.z, cv[2], hv.w * cv[3])));
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (!valid) return;
    *reinterpret_cast<float4*>(p.h + chain * kDS + s0) = hv;
    if (sg == 0) static_cast<TIO*>(p.y)[chain] = from_f32<TIO>(acc);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" ssm_status ssm_scan_step(const ssm_scan_desc* desc, const void* x, const void* delta, const float* A,
                                    const void* b, const void* c, float* h, void* y, void* stream) {
    if (desc == nullptr) return SSM_ERR_INVALID_ARG;
    const ssm_scan_desc& d = *desc;
    if (d.B < 0 || d.D < 0 || d.DS < 0 || d.T != 1) return SSM_ERR_INVALID_ARG;
    if (d.io != SSM_IO_F32 && d.io != SSM_IO_BF16) return SSM_ERR_INVALID_ARG;
    if (d.ckpt_interval < 0 || (d.flags & ~(SSM_SCAN_DETERMINISTIC | SSM_SCAN_DELTA_SOFTPLUS | SSM_SCAN_LOOKBACK)) != 0 || d.B > 65535) return SSM_ERR_INVALID_ARG;
    if (d.DS != kDS || d.D > kMaxD) return SSM_ERR_UNSUPPORTED;
    if (d.B == 0 || d.D == 0) return SSM_OK;
    if (!x || !delta || !A || !b || !c || !h || !y) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, delta, A, b, c, h, y};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SSM_ERR_MISALIGNED;
    const int64_t threads = d.B * d.D * 4;
    const int64_t blocks = (threads + 127) / 128;
    if (blocks > int64_t(0x7fffffff)) return SSM_ERR_UNSUPPORTED;
    StepLaunch L{x, delta, A, b, c, h, y, d.B, d.D, (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(128);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap with the previous step
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = d.io == SSM_IO_BF16 ? cudaLaunchKernelEx(&cfg, step_kernel<__nv_bfloat16>, L)
                                              : cudaLaunchKernelEx(&cfg, step_kernel<float>, L);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
