// Backward scan kernel: reverse sweep with recomputation from checkpoints.
//
// Gradients (page "pssa_kernels.py", `scan_bwd`, re-derived for the loss
// L = sum dy*y + sum ghT*hT): with g_t = dL/dh_t,
//   g_t     = dy_t c_t + a_{t+1} g_{t+1}         (g_{T-1} = dy_{T-1} c_{T-1} + ghT)
//   p_t     = g_t a_t h_{t-1}   (= (a_t g_t) h_{t-1}: the carried adjoint times h_{t-1})
//   gdelta  = sum_s p_t A + x_t sum_s g_t b_t       gx = delta_t sum_s g_t b_t
//   gb      = sum_d g_t delta_t x_t                 gc = sum_d dy_t h_t
//   gA      = sum_{b,t} p_t delta_t                 gh0 = a_0 g_0.
//
// Only the states at chunk boundaries survive the forward (every K <= 256
// steps, as the ruDNN page's `chunk_kda_backward` rematerialises each chunk
// from its retained boundary state). Per chunk, in reverse chunk order:
//   level 2: scan the chunk forward from its checkpoint and keep the state at
//            the start of every LS-step sub-chunk in shared memory;
//   level 3: per sub-chunk, in reverse order, rescan it from its sub-checkpoint
//            into registers (h_t for LS steps);
//   reverse: walk the sub-chunk backwards, recomputing a_t, carrying a_t g_t.
// Thread layout: CTA of 256 threads = 64 channels of one batch, each channel's
// 16 states on 4 neighbouring lanes (4 states per lane). Sums over s (gx,
// gdelta) are reduce-scatters over the 4 lanes and 4 steps. Sums over d (gb,
// gc) are reduce-scatters over the 8 channels of a warp, then shared-memory
// atomics across the CTA's 8 warps, then one vector atomic add per 4 states
// per CTA into global memory. gA is accumulated in registers over all steps of
// the CTA and added atomically once.
#pragma once

#include <type_traits>

#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

template <typename TIO>
struct BwdCfg {
    static constexpr int NT = 256;
    static constexpr int G = 4;
    static constexpr int KS = kDS / G;
    static constexpr int DT = NT / G;
    static constexpr int LS = 16;                       // sub-chunk length
    static constexpr int NSUB = int(kMaxBwdK) / LS;     // sub-checkpoints per chunk
    static constexpr bool BF = std::is_same<TIO, __nv_bfloat16>::value;
    static constexpr size_t X_BYTES = size_t(2) * LS * DT * sizeof(TIO);   // one tensor, 2 buffers
    static constexpr size_t BC_RAW = size_t(2) * LS * kDS * sizeof(TIO);
    static constexpr size_t BC_F32 = BF ? size_t(LS) * kDS * 4 : 0;
    static constexpr size_t SUB_BYTES = size_t(NSUB) * NT * KS * 4;
    static constexpr size_t GX_BYTES = size_t(LS) * DT * 4;
    static constexpr size_t RED_BYTES = size_t(LS) * 2 * kDS * 4;
    static constexpr size_t SMEM = 3 * X_BYTES + 2 * BC_RAW + 2 * BC_F32 + SUB_BYTES + 2 * GX_BYTES + RED_BYTES;
};

// Sum of v[k] over the 8 lanes of a warp that share (lane & 3); lane returns
// the total of entry (lane >> 2).
__device__ __forceinline__ float warp_reduce_scatter8(const float (&v)[8], int lane) {
    const int cw = lane >> 2;
    float a[4];
    const bool b2 = cw & 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = b2 ? v[k] : v[k + 4];
        const float keep = b2 ? v[k + 4] : v[k];
        a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float c2[2];
    const bool b1 = cw & 2;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = b1 ? a[k] : a[k + 2];
        const float keep = b1 ? a[k + 2] : a[k];
        c2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const bool b0 = cw & 1;
    const float send = b0 ? c2[0] : c2[1];
    const float keep = b0 ? c2[1] : c2[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 4);
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <typename TIO, bool VEC>
__global__ void __launch_bounds__(256, 2) bwd_kernel(const BwdLaunch p) {
    using C = BwdCfg<TIO>;
    constexpr int NT = C::NT, KS = C::KS, DT = C::DT, LS = C::LS;

    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* ptr = smem;
    TIO* xs = reinterpret_cast<TIO*>(ptr);  ptr += C::X_BYTES;
    TIO* ds = reinterpret_cast<TIO*>(ptr);  ptr += C::X_BYTES;
    TIO* dys = reinterpret_cast<TIO*>(ptr); ptr += C::X_BYTES;
    TIO* bsr = reinterpret_cast<TIO*>(ptr); ptr += C::BC_RAW;
    TIO* csr = reinterpret_cast<TIO*>(ptr); ptr += C::BC_RAW;
    float* bsf = reinterpret_cast<float*>(ptr); ptr += C::BC_F32;
    float* csf = reinterpret_cast<float*>(ptr); ptr += C::BC_F32;
    float4* sub = reinterpret_cast<float4*>(ptr); ptr += C::SUB_BYTES;   // [NSUB][NT]
    float* gxs = reinterpret_cast<float*>(ptr); ptr += C::GX_BYTES;      // [LS][DT]
    float* gds = reinterpret_cast<float*>(ptr); ptr += C::GX_BYTES;      // [LS][DT]
    float* red = reinterpret_cast<float*>(ptr);                          // [LS][2][16]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int cg = tid >> 2;
    const int gl = tid & 3;
    const int s0 = gl * KS;
    const int64_t T = p.T, D = p.D, K = p.K;
    const int64_t b = blockIdx.y;
    const int64_t d0 = int64_t(blockIdx.x) * DT;
    const int64_t d = d0 + cg;
    const bool valid = d < D;

    const TIO* xg = static_cast<const TIO*>(p.x) + b * T * D;
    const TIO* dg = static_cast<const TIO*>(p.delta) + b * T * D;
    const TIO* dyg = static_cast<const TIO*>(p.dy) + b * T * D;
    const TIO* bg = static_cast<const TIO*>(p.b) + b * T * kDS;
    const TIO* cgl = static_cast<const TIO*>(p.c) + b * T * kDS;

    float A2[KS], Af[KS], gcarry[KS], gAacc[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        Af[s] = valid ? p.A[d * kDS + s0 + s] : 0.f;
        A2[s] = Af[s] * kLog2e;
        gcarry[s] = (valid && p.ghT != nullptr) ? p.ghT[(b * D + d) * kDS + s0 + s] : 0.f;
        gAacc[s] = 0.f;
    }
    for (int i = tid; i < LS * 2 * kDS; i += NT) red[i] = 0.f;

    const int64_t nck = (T + K - 1) / K;
    for (int64_t j = nck - 1; j >= 0; --j) {
        const int64_t cs = j * K;
        const int64_t ce = min(T, cs + K);
        const int nsub = int((ce - cs + LS - 1) / LS);

        auto stage = [&](int i, int buf, bool rev) {
            const int64_t t0 = cs + int64_t(i) * LS;
            stage_tile<TIO, LS, DT, NT, VEC>(xs + buf * LS * DT, xg, D, t0, ce, d0);
            stage_tile<TIO, LS, DT, NT, VEC>(ds + buf * LS * DT, dg, D, t0, ce, d0);
            stage_tile<TIO, LS, kDS, NT, true>(bsr + buf * LS * kDS, bg, kDS, t0, ce, 0);
            if (rev) {
                stage_tile<TIO, LS, DT, NT, VEC>(dys + buf * LS * DT, dyg, D, t0, ce, d0);
                stage_tile<TIO, LS, kDS, NT, true>(csr + buf * LS * kDS, cgl, kDS, t0, ce, 0);
            }
        };

        // ---- level 2: forward over the chunk, keeping sub-chunk start states
        float h[KS];
        {
            const float* src = p.ckpt + ((j * p.B + b) * D + (valid ? d : 0)) * kDS + s0;
#pragma unroll
            for (int s = 0; s < KS; ++s) h[s] = valid ? src[s] : 0.f;
        }
        stage(0, 0, false);
        cp_async_commit();
        for (int i = 0; i < nsub; ++i) {
            const int buf = i & 1;
            if (i + 1 < nsub) {
                stage(i + 1, buf ^ 1, false);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float* bt;
            if constexpr (C::BF) {
                widen_bf16<NT>(bsf, reinterpret_cast<const __nv_bfloat16*>(bsr + buf * LS * kDS), LS * kDS);
                __syncthreads();
                bt = bsf;
            } else {
                bt = reinterpret_cast<const float*>(bsr + buf * LS * kDS);
            }
            sub[i * NT + tid] = make_float4(h[0], h[1], h[2], h[3]);
            const TIO* xt = xs + buf * LS * DT;
            const TIO* dt = ds + buf * LS * DT;
#pragma unroll 4
            for (int r = 0; r < LS; ++r) {
                const float dl = to_f32(dt[r * DT + cg]);
                const float dx = dl * to_f32(xt[r * DT + cg]);
#pragma unroll
                for (int s = 0; s < KS; ++s) h[s] = fmaf(ex2(dl * A2[s]), h[s], dx * bt[r * kDS + s0 + s]);
            }
            __syncthreads();
        }

        // ---- reverse over the sub-chunks
        stage(nsub - 1, 0, true);
        cp_async_commit();
        for (int ii = 0; ii < nsub; ++ii) {
            const int i = nsub - 1 - ii;
            const int buf = ii & 1;
            if (ii + 1 < nsub) {
                stage(i - 1, buf ^ 1, true);
                cp_async_commit();
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float* bt;
            const float* ct;
            if constexpr (C::BF) {
                widen_bf16<NT>(bsf, reinterpret_cast<const __nv_bfloat16*>(bsr + buf * LS * kDS), LS * kDS);
                widen_bf16<NT>(csf, reinterpret_cast<const __nv_bfloat16*>(csr + buf * LS * kDS), LS * kDS);
                __syncthreads();
                bt = bsf;
                ct = csf;
            } else {
                bt = reinterpret_cast<const float*>(bsr + buf * LS * kDS);
                ct = reinterpret_cast<const float*>(csr + buf * LS * kDS);
            }
            const TIO* xt = xs + buf * LS * DT;
            const TIO* dt = ds + buf * LS * DT;
            const TIO* dyt = dys + buf * LS * DT;
            const int64_t t0 = cs + int64_t(i) * LS;

            // level 3: states of this sub-chunk into registers
            float hs[KS], hw[LS][KS];
            {
                const float4 v = sub[i * NT + tid];
                hs[0] = v.x; hs[1] = v.y; hs[2] = v.z; hs[3] = v.w;
            }
#pragma unroll
            for (int r = 0; r < LS; ++r) {
                const float dl = to_f32(dt[r * DT + cg]);
                const float dx = dl * to_f32(xt[r * DT + cg]);
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    const float prev = (r == 0) ? hs[s] : hw[r - 1][s];
                    hw[r][s] = fmaf(ex2(dl * A2[s]), prev, dx * bt[r * kDS + s0 + s]);
                }
            }

            // reverse sweep over the sub-chunk, 4 steps at a time
#pragma unroll
            for (int rg = LS - 4; rg >= 0; rg -= 4) {
                float rr[4], qq[4];
#pragma unroll
                for (int jj = 3; jj >= 0; --jj) {
                    const int r = rg + jj;
                    const float dl = to_f32(dt[r * DT + cg]);
                    const float dx = dl * to_f32(xt[r * DT + cg]);
                    const float dyv = to_f32(dyt[r * DT + cg]);
                    float racc = 0.f, qacc = 0.f, part[8];
#pragma unroll
                    for (int s = 0; s < KS; ++s) {
                        const float a = ex2(dl * A2[s]);
                        const float g = fmaf(dyv, ct[r * kDS + s0 + s], gcarry[s]);
                        gcarry[s] = a * g;
                        const float hp = (r == 0) ? hs[s] : hw[r - 1][s];
                        const float pp = gcarry[s] * hp;
                        gAacc[s] = fmaf(pp, dl, gAacc[s]);
                        racc = fmaf(pp, Af[s], racc);
                        qacc = fmaf(g, bt[r * kDS + s0 + s], qacc);
                        part[s] = g * dx;               // gb partial (this channel)
                        part[4 + s] = dyv * hw[r][s];   // gc partial (this channel)
                    }
                    rr[jj] = racc;
                    qq[jj] = qacc;
                    const float v = warp_reduce_scatter8(part, lane);
                    const int cw = lane >> 2;           // entry this lane now holds
                    atomicAdd(&red[r * 2 * kDS + (cw >> 2) * kDS + s0 + (cw & 3)], v);
                }
                const float rs = reduce_scatter_steps<4>(rr, gl);
                const float qs = reduce_scatter_steps<4>(qq, gl);
                const int r = rg + gl;
                const float dl = to_f32(dt[r * DT + cg]);
                const float xv = to_f32(xt[r * DT + cg]);
                gxs[r * DT + cg] = dl * qs;
                gds[r * DT + cg] = rs + xv * qs;
            }
            __syncthreads();

            // flush the sub-chunk: gx, gdelta tiles; gb, gc partial sums
            const int64_t rows = min(int64_t(LS), ce - t0);
            float* gxg = p.gx + b * T * D;
            float* gdg = p.gdelta + b * T * D;
            if constexpr (VEC) {
                constexpr int CPR = DT / 4;
                for (int k = tid; k < LS * CPR; k += NT) {
                    const int r = k / CPR, cc = k % CPR;
                    const int64_t col = d0 + int64_t(cc) * 4;
                    if (r < rows && col < D) {
                        *reinterpret_cast<float4*>(gxg + (t0 + r) * D + col) =
                            *reinterpret_cast<const float4*>(gxs + r * DT + cc * 4);
                        *reinterpret_cast<float4*>(gdg + (t0 + r) * D + col) =
                            *reinterpret_cast<const float4*>(gds + r * DT + cc * 4);
                    }
                }
            } else {
                for (int k = tid; k < LS * DT; k += NT) {
                    const int r = k / DT, cc = k % DT;
                    if (r < rows && d0 + cc < D) {
                        gxg[(t0 + r) * D + d0 + cc] = gxs[k];
                        gdg[(t0 + r) * D + d0 + cc] = gds[k];
                    }
                }
            }
            if (tid < LS * 8) {                         // LS rows x (gb, gc) x 4 quads of states
                const int r = tid >> 3, tensor = (tid >> 2) & 1, q = tid & 3;
                if (r < rows) {
                    const float* src = red + r * 2 * kDS + tensor * kDS + q * 4;
                    float* dst = (tensor == 0 ? p.gb : p.gc) + (b * T + t0 + r) * kDS + q * 4;
                    red_add_v4(dst, src[0], src[1], src[2], src[3]);
                }
            }
            __syncthreads();
            for (int k = tid; k < LS * 2 * kDS; k += NT) red[k] = 0.f;
            // the next sub-chunk's first barrier orders these zeros before its atomics
        }
    }

    if (!valid) return;
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        p.gh0[(b * D + d) * kDS + s0 + s] = gcarry[s];
        atomicAdd(&p.gA[d * kDS + s0 + s], gAacc[s]);
    }
}

template <typename TIO>
cudaError_t launch_bwd_io(const BwdLaunch& L, cudaStream_t stream) {
    using C = BwdCfg<TIO>;
    auto kern = L.vec ? bwd_kernel<TIO, true> : bwd_kernel<TIO, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
    if (e != cudaSuccess) return e;
    const dim3 grid(unsigned((L.D + C::DT - 1) / C::DT), unsigned(L.B));
    kern<<<grid, C::NT, C::SMEM, stream>>>(L);
    return cudaGetLastError();
}

}  // namespace ssm
