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
// One warp per (chain, group of 4 states), the carries split into 32 consecutive segments, one
// per lane, so the dependent L2 round trips per chain drop from nchunk / 8 to about
// nchunk / 128:
//   1. each lane composes the maps of its segment (from a zero start: the segment's own delta
//      sum and end state);
//   2. an exclusive scan of the 32 segment maps over the warp's lanes (five shuffle rounds;
//      composing map (s1, S1) then (s2, S2) gives (s1 + s2, exp(A s2) S1 + S2));
//   3. each lane applies the maps of its segment again from its segment's start state
//      exp(A s_before) h0 + S_before and writes every chunk's start state.
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kNB = 8;      // chunks whose carries are loaded together

__global__ void __launch_bounds__(128) fwd_carry_scan_kernel(const FwdLaunch p) {
    const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;   // warp: (chain, group)
    const int lane = threadIdx.x & 31;
    const int64_t chain = gw >> 2;                  // b * D + d
    if (chain >= p.B * p.D) return;                 // whole warps leave together
    const int s0 = int(gw & 3) * 4;
    const int64_t b = chain / p.D, d = chain - b * p.D;
    const int64_t nprev = p.nchunk - 1;
    const int64_t seg = (nprev + 31) / 32;
    const int64_t j_begin = min(nprev, lane * seg), j_end = min(nprev, j_begin + seg);
    const float4 a = *reinterpret_cast<const float4*>(p.A + d * kDS + s0);
    const float A2[4] = {a.x * kLog2e, a.y * kLog2e, a.z * kLog2e, a.w * kLog2e};
    auto row_of = [&](int64_t j) { return (b * nprev + j) * p.D + d; };

    // apply the maps of chunks [j0, j1) to h (and accumulate their delta sums); with `store`,
    // write the state after each chunk (the start state of the next one)
    auto sweep = [&](int64_t j0, int64_t j1, float4& h, float& sig, bool store) {
        for (int64_t jb = j0; jb < j1; jb += kNB) {
            float sd[kNB];
            float4 S[kNB];
#pragma unroll
            for (int u = 0; u < kNB; ++u) {
                sd[u] = 0.f;
                S[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (jb + u < j1) {
                    const int64_t row = row_of(jb + u);
                    sd[u] = p.ws_Sd[row];
                    S[u] = *reinterpret_cast<const float4*>(p.ws_S + row * kDS + s0);
                }
            }
#pragma unroll
            for (int u = 0; u < kNB; ++u) {
                if (jb + u >= j1) break;
                h.x = fmaf(ex2(A2[0] * sd[u]), h.x, S[u].x);
                h.y = fmaf(ex2(A2[1] * sd[u]), h.y, S[u].y);
                h.z = fmaf(ex2(A2[2] * sd[u]), h.z, S[u].z);
                h.w = fmaf(ex2(A2[3] * sd[u]), h.w, S[u].w);
                sig += sd[u];
                if (store) *reinterpret_cast<float4*>(p.ws_S + row_of(jb + u) * kDS + s0) = h;
            }
        }
    };
    // 1. this lane's segment as one map (delta sum sig, end state S from a zero start)
    float sig = 0.f;
    float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
    sweep(j_begin, j_end, S, sig, false);
    // 2. inclusive scan of the maps over the lanes, then shifted by one lane (exclusive)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float ps = __shfl_up_sync(0xffffffffu, sig, off);
        const float px = __shfl_up_sync(0xffffffffu, S.x, off), py = __shfl_up_sync(0xffffffffu, S.y, off);
        const float pz = __shfl_up_sync(0xffffffffu, S.z, off), pw = __shfl_up_sync(0xffffffffu, S.w, off);
        if (lane >= off) {      // the earlier lanes' map first, then this lane's
            S.x = fmaf(ex2(A2[0] * sig), px, S.x);
            S.y = fmaf(ex2(A2[1] * sig), py, S.y);
            S.z = fmaf(ex2(A2[2] * sig), pz, S.z);
            S.w = fmaf(ex2(A2[3] * sig), pw, S.w);
            sig += ps;
        }
    }
    float sig_ex = __shfl_up_sync(0xffffffffu, sig, 1);
    float4 S_ex = make_float4(__shfl_up_sync(0xffffffffu, S.x, 1), __shfl_up_sync(0xffffffffu, S.y, 1),
                              __shfl_up_sync(0xffffffffu, S.z, 1), __shfl_up_sync(0xffffffffu, S.w, 1));
    if (lane == 0) {
        sig_ex = 0.f;
        S_ex = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // 3. the state entering this lane's segment, then its chunks again, storing each start state
    float4 h = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.h0 != nullptr) h = *reinterpret_cast<const float4*>(p.h0 + chain * kDS + s0);
    h.x = fmaf(ex2(A2[0] * sig_ex), h.x, S_ex.x);
    h.y = fmaf(ex2(A2[1] * sig_ex), h.y, S_ex.y);
    h.z = fmaf(ex2(A2[2] * sig_ex), h.z, S_ex.z);
    h.w = fmaf(ex2(A2[3] * sig_ex), h.w, S_ex.w);
    float unused = 0.f;
    sweep(j_begin, j_end, h, unused, true);
}

}  // namespace

cudaError_t launch_fwd_carry_scan(const FwdLaunch& L, cudaStream_t stream) {
    const int64_t threads = L.B * L.D * 4 * 32;       // one warp per (chain, group of 4 states)
    const int64_t blocks = (threads + 127) / 128;
    if (blocks > int64_t(0x7fffffff)) return cudaErrorInvalidValue;
    fwd_carry_scan_kernel<<<unsigned(blocks), 128, 0, stream>>>(L);
    return cudaGetLastError();
}

}  // namespace ssm
