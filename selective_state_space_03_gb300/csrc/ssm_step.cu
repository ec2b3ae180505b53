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
// chain, so it is bound by HBM (or by launch latency for small B*D). Layout: 2
// lanes per chain, 8 states per lane in two 16-byte loads and stores, the
// readout finished with one shuffle; 64 chains per 128-thread CTA (with 4 lanes
// per chain workload 5's 81920 chains took 2560 CTAs, 1.05 waves at 16 per SM;
// with 2, 1280 CTAs fit in one). Steps are launched with programmatic stream
// serialization: a step's CTAs are scheduled while the previous kernel on the
// stream finishes, and every load waits (griddepcontrol.wait) until that
// kernel has completed and its writes are visible, whatever kernel it was.
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
    bool inputs_ready;   // the preceding kernel writes none of x, delta, A, b, c
};

// 8 consecutive I/O values as float32 (16-byte aligned)
template <typename TIO>
__device__ __forceinline__ void load8(const TIO* p, float (&v)[8]) {
    if constexpr (std::is_same<TIO, float>::value) {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

// This step's x, delta (through softplus when asked), b, c and A.
template <typename TIO>
__device__ __forceinline__ void load_step_inputs(const StepLaunch& p, int64_t chain, int s0, float& dl, float& dx,
                                                 float (&bv)[8], float (&cv)[8], float (&av)[8]) {
    const int64_t bb = chain / p.D, d = chain - bb * p.D;
    dl = to_f32(static_cast<const TIO*>(p.delta)[chain]);
    if (p.softplus) dl = softplus_f32(dl);
    dx = dl * to_f32(static_cast<const TIO*>(p.x)[chain]);
    load8<TIO>(static_cast<const TIO*>(p.b) + bb * kDS + s0, bv);
    load8<TIO>(static_cast<const TIO*>(p.c) + bb * kDS + s0, cv);
    load8<float>(p.A + d * kDS + s0, av);
}

template <typename TIO>
__global__ void __launch_bounds__(128) step_kernel(const StepLaunch p) {
    const int64_t gid = int64_t(blockIdx.x) * 128 + threadIdx.x;
    const int64_t chain = gid >> 1;
    const int sg = int(gid & 1), s0 = sg * 8;
    const bool valid = chain < p.B * p.D;       // whole lane pairs are valid or not
    // Consecutive steps on a stream are launched as programmatic dependents: let the next
    // step's CTAs be scheduled now; they run up to their wait below while this grid finishes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float acc = 0.f;
    float hv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float dl = 0.f, dx = 0.f, bv[8], cv[8], av[8];
    // Inputs the caller declared untouched by the preceding kernel load while it finishes.
    if (p.inputs_ready && valid) load_step_inputs<TIO>(p, chain, s0, dl, dx, bv, cv, av);
    // Otherwise every input may have been written by the kernel before this one on the stream
    // (the previous step writes h and y; a projection kernel may write x, delta, b, c, even one
    // that lets its dependents launch before its own stores): wait until that grid has
    // completed and its writes are visible (returns at once when there is no such grid).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (valid) {
        if (!p.inputs_ready) load_step_inputs<TIO>(p, chain, s0, dl, dx, bv, cv, av);
        load8<float>(p.h + chain * kDS + s0, hv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            hv[i] = fmaf(ex2(dl * (av[i] * kLog2e)), hv[i], dx * bv[i]);
            acc = fmaf(hv[i], cv[i], acc);
        }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (!valid) return;
    float4* hd = reinterpret_cast<float4*>(p.h + chain * kDS + s0);
    hd[0] = make_float4(hv[0], hv[1], hv[2], hv[3]);
    hd[1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
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
    if (d.ckpt_interval < 0 || (d.flags & ~(SSM_SCAN_DETERMINISTIC | SSM_SCAN_DELTA_SOFTPLUS | SSM_SCAN_LOOKBACK | SSM_SCAN_STEP_INPUTS_READY)) != 0 || d.B > 65535) return SSM_ERR_INVALID_ARG;
    if (d.DS != kDS || d.D > kMaxD) return SSM_ERR_UNSUPPORTED;
    if (d.B == 0 || d.D == 0) return SSM_OK;
    if (!x || !delta || !A || !b || !c || !h || !y) return SSM_ERR_INVALID_ARG;
    // A, b, c and h are read with 16-byte loads; x, delta and y one element per chain, so a
    // row of a (B, T, D) tensor (x[:, t] with B = 1) can be passed as it is
    const void* vec_ptrs[] = {A, b, c, h};
    for (const void* q : vec_ptrs)
        if (!aligned16(q)) return SSM_ERR_MISALIGNED;
    const uintptr_t esz = d.io == SSM_IO_BF16 ? 2 : 4;
    const void* elem_ptrs[] = {x, delta, y};
    for (const void* q : elem_ptrs)
        if (reinterpret_cast<uintptr_t>(q) % esz != 0) return SSM_ERR_MISALIGNED;
    const int64_t threads = d.B * d.D * 2;
    const int64_t blocks = (threads + 127) / 128;
    if (blocks > int64_t(0x7fffffff)) return SSM_ERR_UNSUPPORTED;
    StepLaunch L{x, delta, A, b, c, h, y, d.B, d.D, (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0,
                 (d.flags & SSM_SCAN_STEP_INPUTS_READY) != 0};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(128);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // scheduled while the previous kernel ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = d.io == SSM_IO_BF16 ? cudaLaunchKernelEx(&cfg, step_kernel<__nv_bfloat16>, L)
                                              : cudaLaunchKernelEx(&cfg, step_kernel<float>, L);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
