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
//            into a window of tensor memory (h_t for LS steps; TMEM keeps the
//            64 registers the window would take free for occupancy, and its
//            traffic bypasses the shared-memory pipe);
//   reverse: walk the sub-chunk backwards, recomputing a_t, carrying a_t g_t.
//
// Layout: a CTA of 128 threads covers 32 channels of one batch; each channel's
// 16 states are on 4 neighbouring lanes (4 states per lane), so a warp holds 8
// channels. Per tile of LS steps the raw inputs land in shared memory through
// cp.async and are converted once into one float4 (delta, delta*x, x, dy) per
// (step, channel) and float32 b, c rows, so the inner loop reads one 16-byte
// value per step for the channel and one per 4 states for b and c. The raw
// buffer is refilled with the next tile while the converted one is used.
// Sums over s (gx, gdelta) are reduce-scatters over the channel's 4 lanes and
// 4 steps; sums over d (gb, gc) are reduce-scatters over the warp's 8 channels
// into per-warp shared slots, summed over the CTA's warps once per tile and added
// to global memory with one red.global.add.v4.f32 per 4 states per CTA. (On
// sm_103a shuffles and shared loads share one pipe of ~1 warp-instruction per
// clock per SM, and a 16-byte broadcast load takes 4 of its cycles, so the
// reductions are built to spend as few of those cycles as possible.) gA is
// accumulated in registers over the CTA's whole sweep and added atomically once.
// The per-state arithmetic runs on pairs of neighbouring states as packed f32x2
// operations (FMUL2 / FFMA2: one issue slot for two operations), the MUFU
// exponentials and the reductions stay scalar.
//
// The same file holds the chunk-parallel pass (bwd_carry_kernel), and the
// kernels' deterministic (partials instead of atomics) and fused (softplus on
// delta, skip connection) variants.
#pragma once

#include <type_traits>

#include "ssm_common.cuh"
#include "ssm_internal.h"
#include "ssm_tmem.cuh"

namespace ssm {

template <typename TIO>
struct BwdCfg {
    static constexpr int NT = 128;
    static constexpr int NW = NT / 32;
    static constexpr int G = 4;
    static constexpr int KS = kDS / G;                  // states per lane
    static constexpr int DT = NT / G;                   // channels per CTA (32)
    static constexpr int LS = 16;                       // sub-chunk (tile) length
    static constexpr int NSUB = int(kMaxBwdK) / LS;     // sub-checkpoints per chunk
    static constexpr bool BF = std::is_same<TIO, __nv_bfloat16>::value;
    static constexpr int EPC = 16 / int(sizeof(TIO));
    static constexpr int X_CPR = DT / EPC;              // 16-byte chunks per raw tile row
    static constexpr int X_CH = LS * X_CPR;
    static constexpr int BC_CH = LS * kDS / EPC;
    // shared memory (bytes)
    static constexpr size_t RAW_X = size_t(LS) * DT * sizeof(TIO);          // one of x, delta, dy
    static constexpr size_t RAW_BC = size_t(LS) * kDS * sizeof(TIO);        // one of b, c
    // float4 per (step, channel); rows padded by one float4 so that the 4 lanes of a channel,
    // which read 4 different steps at once in the per-step sums, hit different banks
    static constexpr int CROW = DT + 1;
    static constexpr size_t CONV = size_t(LS) * CROW * 16;
    static constexpr size_t BCF = size_t(LS) * kDS * 4;                     // one of b, c as float32
    static constexpr size_t SUB = size_t(NSUB) * NT * 16;                   // float4 sub-checkpoints
    static constexpr size_t GBC = size_t(NW) * LS * 2 * kDS * 4;            // per-warp sums of gb, gc for a tile
    // level-3 window per lane: LS steps x 4 states of h, then the same of b (b_t kept from
    // level 3 so the reverse reads it from TMEM instead of shared memory)
    static constexpr uint32_t TMEM_B = LS * KS;
    static constexpr uint32_t TMEM_COLS = 2 * LS * KS;
    static constexpr size_t SMEM = 3 * RAW_X + 2 * RAW_BC + CONV + 2 * BCF + SUB + GBC + 16;
};

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}


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

// The first two stages of warp_reduce_scatter8: sums over the 4 lanes {cw, cw^2, cw^4, cw^6}
// (cw = lane >> 2); lane returns entries 2 (cw >> 1) and 2 (cw >> 1) + 1.
__device__ __forceinline__ float2 warp_reduce_scatter8_half(const float (&v)[8], int lane) {
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
    return make_float2(c2[0], c2[1]);
}

__device__ __forceinline__ float4 operator+(const float4 a, const float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <typename TIO, bool VEC, bool FUSE>
__global__ void __launch_bounds__(128, 4) bwd_kernel(const BwdLaunch p) {
    using C = BwdCfg<TIO>;
    constexpr int NT = C::NT, KS = C::KS, DT = C::DT, LS = C::LS, EPC = C::EPC;

    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* ptr = smem;
    TIO* xr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_X;
    TIO* dr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_X;
    TIO* yr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_X;
    TIO* br = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_BC;
    TIO* cr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_BC;
    float4* conv = reinterpret_cast<float4*>(ptr); ptr += C::CONV;     // [LS][CROW]
    float* bf = reinterpret_cast<float*>(ptr);     ptr += C::BCF;      // [LS][16]
    float* cf = reinterpret_cast<float*>(ptr);     ptr += C::BCF;
    float4* sub = reinterpret_cast<float4*>(ptr);  ptr += C::SUB;      // [NSUB][NT]
    float* gbc = reinterpret_cast<float*>(ptr);    ptr += C::GBC;      // [NW][LS][2][16]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ptr);

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int cw = lane >> 2;               // channel within the warp
    const int sg = lane & 3;                // state group within the channel
    const int c = warp * 8 + cw;            // channel within the CTA
    const int s0 = sg * KS;
    const int64_t T = p.T, D = p.D, K = p.K;
    const int64_t b = blockIdx.y;
    const int64_t d0 = int64_t(blockIdx.x) * DT;
    const int64_t d = d0 + c;
    const bool valid = d < D;
    const bool full_d = d0 + DT <= D;

    const TIO* xg = static_cast<const TIO*>(p.x) + b * T * D;
    const TIO* dg = static_cast<const TIO*>(p.delta) + b * T * D;
    const TIO* dyg = static_cast<const TIO*>(p.dy) + b * T * D;
    const TIO* bg = static_cast<const TIO*>(p.b) + b * T * kDS;
    const TIO* cgl = static_cast<const TIO*>(p.c) + b * T * kDS;
    float* gxg = p.gx + b * T * D;
    float* gdg = p.gdelta + b * T * D;

    const float Dk = (FUSE && valid && p.Dskip != nullptr) ? p.Dskip[d] : 0.f;   // skip weight
    float skip_acc = 0.f;                                                         // sum of dy x
    // per-state values as pairs of neighbouring states, for packed f32x2 arithmetic
    float2 A2[2], Af[2], gcarry[2], gAacc[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int s = s0 + 2 * q;
        Af[q] = valid ? make_float2(p.A[d * kDS + s], p.A[d * kDS + s + 1]) : make_float2(0.f, 0.f);
        A2[q] = make_float2(Af[q].x * kLog2e, Af[q].y * kLog2e);
        gcarry[q] = (valid && p.ghT != nullptr)
            ? make_float2(p.ghT[(b * D + d) * kDS + s], p.ghT[(b * D + d) * kDS + s + 1]) : make_float2(0.f, 0.f);
        gAacc[q] = make_float2(0.f, 0.f);
    }

    // level-3 window in tensor memory: this warp's 32 lanes x LS*4 columns
    if (warp == 0) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tw = tmem_base + (uint32_t((warp & 3) * 32) << 16);

    // this thread's 16-byte chunk of a full raw tile (x, delta, dy) and of b, c
    const int xr_r = tid / C::X_CPR, xr_c = (tid % C::X_CPR) * EPC;
    const int x_goff = xr_r * int(D) + xr_c, x_soff = xr_r * DT + xr_c;

    auto stage = [&](int64_t t0, int64_t tend, bool rev) {
        if (VEC && full_d && t0 + LS <= tend) {
            if (tid < C::X_CH) {
                const int64_t base = t0 * D + d0;
                cp_async16(xr + x_soff, xg + base + x_goff, 16);
                cp_async16(dr + x_soff, dg + base + x_goff, 16);
                if (rev) cp_async16(yr + x_soff, dyg + base + x_goff, 16);
            }
            if (tid < C::BC_CH) {
                cp_async16(br + tid * EPC, bg + t0 * kDS + tid * EPC, 16);
                if (rev) cp_async16(cr + tid * EPC, cgl + t0 * kDS + tid * EPC, 16);
            }
        } else {
            stage_tile<TIO, LS, DT, NT, VEC>(xr, xg, D, t0, tend, d0);
            stage_tile<TIO, LS, DT, NT, VEC>(dr, dg, D, t0, tend, d0);
            if (rev) stage_tile<TIO, LS, DT, NT, VEC>(yr, dyg, D, t0, tend, d0);
            stage_tile<TIO, LS, kDS, NT, true>(br, bg, kDS, t0, tend, 0);
            if (rev) stage_tile<TIO, LS, kDS, NT, true>(cr, cgl, kDS, t0, tend, 0);
        }
        cp_async_commit();
    };
    // raw tile -> (delta, delta*x, x, dy) per (step, channel) and float32 b, c rows
    // (rows >= rows_valid are padding: with softplus their delta must stay 0, not ln 2)
    auto convert = [&](bool rev, int64_t rows_valid) {
#pragma unroll
        for (int k = 0; k < LS * DT / NT; ++k) {
            const int i = tid + NT * k;
            float dl = to_f32(dr[i]);
            if (FUSE && p.softplus) dl = (i / DT < rows_valid) ? softplus_f32(dl) : 0.f;
            const float xv = to_f32(xr[i]);
            conv[(i / DT) * C::CROW + i % DT] = make_float4(dl, dl * xv, xv, rev ? to_f32(yr[i]) : 0.f);
        }
#pragma unroll
        for (int k = 0; k < LS * kDS / NT; ++k) {
            const int i = tid + NT * k;
            bf[i] = to_f32(br[i]);
            if (rev) cf[i] = to_f32(cr[i]);
        }
    };
    // gb, gc of the tile starting at t0: sum the warps' slots, add to global (rows below t_lim)
    auto flush_gbc = [&](int64_t t0, int64_t t_lim) {
        const int r = tid >> 3, tau = (tid >> 2) & 1, q = tid & 3;
        const int off = r * 2 * kDS + tau * kDS + q * 4;
        float4 v = *reinterpret_cast<const float4*>(gbc + off);
#pragma unroll
        for (int w = 1; w < C::NW; ++w) v = v + *reinterpret_cast<const float4*>(gbc + w * LS * 2 * kDS + off);
        if (t0 + r < t_lim) {
            if (p.det) {
                *reinterpret_cast<float4*>(p.part_gbc + ((int64_t(blockIdx.x) * p.B + b) * T + t0 + r) * (2 * kDS) +
                                           tau * kDS + q * 4) = v;
            } else {
                float* dst = (tau == 0 ? p.gb : p.gc) + (b * T + t0 + r) * kDS + q * 4;
                red_add_v4(dst, v.x, v.y, v.z, v.w);
            }
        }
    };

    const int64_t nck = (T + K - 1) / K;
    // chunks this CTA sweeps: all of them, or (chunk-parallel schedule) chunk blockIdx.z with
    // the adjoint entering it folded from the later chunks' carries
    int64_t jhi = nck - 1, jlo = 0;
    if (p.tpar) {
        jhi = jlo = blockIdx.z;
        if (valid) {
            for (int64_t jj = nck - 1; jj > jlo; --jj) {
                const float4 z = *reinterpret_cast<const float4*>(p.carry_Z + ((jj * p.B + b) * D + d) * kDS + s0);
                const float sd = p.carry_S[(jj * p.B + b) * D + d];
                gcarry[0] = make_float2(fmaf(ex2(A2[0].x * sd), gcarry[0].x, z.x), fmaf(ex2(A2[0].y * sd), gcarry[0].y, z.y));
                gcarry[1] = make_float2(fmaf(ex2(A2[1].x * sd), gcarry[1].x, z.z), fmaf(ex2(A2[1].y * sd), gcarry[1].y, z.w));
            }
        }
    }
    int64_t pend_t0 = -1, pend_lim = 0;       // tile whose gb/gc sums await their flush
    for (int64_t j = jhi; j >= jlo; --j) {
        const int64_t cs = j * K;
        const int64_t ce = min(T, cs + K);
        const int nsub = int((ce - cs + LS - 1) / LS);

        // ---- level 2: forward over the chunk, keeping sub-chunk start states
        float h[KS];
        {
            const float* src = p.ckpt + ((j * p.B + b) * D + (valid ? d : 0)) * kDS + s0;
#pragma unroll
            for (int s = 0; s < KS; ++s) h[s] = valid ? src[s] : 0.f;
        }
        stage(cs, ce, false);
        for (int i = 0; i < nsub; ++i) {
            cp_async_wait<0>();
            __syncthreads();
            convert(false, ce - (cs + int64_t(i) * LS));
            __syncthreads();
            if (i + 1 < nsub) stage(cs + int64_t(i + 1) * LS, ce, false);
            sub[i * NT + tid] = make_float4(h[0], h[1], h[2], h[3]);
            float2 h2[2] = {make_float2(h[0], h[1]), make_float2(h[2], h[3])};
            // one step; with `window`, the step's state and b also go into the TMEM window
            auto level2_step = [&](int r, bool window) {
                const float2 v = *reinterpret_cast<const float2*>(conv + r * C::CROW + c);   // delta, delta*x
                const float4 b4 = *reinterpret_cast<const float4*>(bf + r * kDS + s0);
                const float2 bp[2] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
                const float2 dl2 = make_float2(v.x, v.x), dx2 = make_float2(v.y, v.y);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float2 e = __fmul2_rn(dl2, A2[q]);
                    h2[q] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), h2[q], __fmul2_rn(dx2, bp[q]));
                }
                if (window) {
                    tmem_st4(tw + uint32_t(r * KS), h2[0].x, h2[0].y, h2[1].x, h2[1].y);
                    tmem_st4(tw + C::TMEM_B + uint32_t(r * KS), b4.x, b4.y, b4.z, b4.w);
                }
            };
            if (i + 1 < nsub) {
#pragma unroll 4
                for (int r = 0; r < LS; ++r) level2_step(r, false);
            } else {
                // the chunk's last sub-chunk, which the reverse takes first: its window is written
                // here, so the reverse skips level 3 for it
#pragma unroll 4
                for (int r = 0; r < LS; ++r) level2_step(r, true);
                tmem_wait_st();
            }
            h[0] = h2[0].x; h[1] = h2[0].y; h[2] = h2[1].x; h[3] = h2[1].y;
        }

        // ---- reverse over the sub-chunks
        stage(cs + int64_t(nsub - 1) * LS, ce, true);
        for (int ii = 0; ii < nsub; ++ii) {
            const int i = nsub - 1 - ii;
            const int64_t t0 = cs + int64_t(i) * LS;
            cp_async_wait<0>();
            __syncthreads();
            if (pend_t0 >= 0) flush_gbc(pend_t0, pend_lim);
            convert(true, ce - t0);
            __syncthreads();
            if (ii + 1 < nsub) stage(t0 - LS, ce, true);
            pend_t0 = t0;
            pend_lim = ce;

            // level 3: states of this sub-chunk into the TMEM window (4 columns per step)
            float hs[KS];
            {
                const float4 v = sub[i * NT + tid];
                hs[0] = v.x; hs[1] = v.y; hs[2] = v.z; hs[3] = v.w;
            }
            if (ii > 0) {       // (the chunk's last sub-chunk: written by level 2)
                float2 hc[2] = {make_float2(hs[0], hs[1]), make_float2(hs[2], hs[3])};
#pragma unroll
                for (int r = 0; r < LS; ++r) {
                    const float2 v = *reinterpret_cast<const float2*>(conv + r * C::CROW + c);
                    const float4 b4 = *reinterpret_cast<const float4*>(bf + r * kDS + s0);
                    const float2 bp[2] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
                    const float2 dl2 = make_float2(v.x, v.x), dx2 = make_float2(v.y, v.y);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float2 e = __fmul2_rn(dl2, A2[q]);
                        hc[q] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), hc[q], __fmul2_rn(dx2, bp[q]));
                    }
                    tmem_st4(tw + uint32_t(r * KS), hc[0].x, hc[0].y, hc[1].x, hc[1].y);
                    tmem_st4(tw + C::TMEM_B + uint32_t(r * KS), b4.x, b4.y, b4.z, b4.w);
                }
                tmem_wait_st();
            }

            float* gw = gbc + warp * LS * 2 * kDS;   // this warp's gb, gc sums for the tile
            // reverse sweep over the sub-chunk, 4 steps per lane reduce-scatter group
#pragma unroll
            for (int rg = LS - 4; rg >= 0; rg -= 4) {
                float hg[16], bgr[16], hprev[KS];   // h and b for steps rg..rg+3, h for step rg-1
                tmem_ld16(tw + uint32_t(rg * KS), hg);
                tmem_ld16(tw + C::TMEM_B + uint32_t(rg * KS), bgr);
                if (rg > 0) {
                    tmem_ld4(tw + uint32_t((rg - 1) * KS), hprev);
                } else {
#pragma unroll
                    for (int s = 0; s < KS; ++s) hprev[s] = hs[s];
                }
                tmem_wait_ld();
                float rr[4], qq[4];
#pragma unroll
                for (int jj = 3; jj >= 0; --jj) {
                    const int r = rg + jj;
                    // delta, delta*x and dy of this step (x is read once per 4 steps, below)
                    const float2 v2 = *reinterpret_cast<const float2*>(conv + r * C::CROW + c);
                    const float dyv = reinterpret_cast<const float*>(conv + r * C::CROW + c)[3];
                    const float4 v = make_float4(v2.x, v2.y, 0.f, dyv);
                    const float4 c4 = *reinterpret_cast<const float4*>(cf + r * kDS + s0);
                    const float2 cp[2] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
                    const float2 dl2 = make_float2(v.x, v.x), dx2 = make_float2(v.y, v.y), dy2 = make_float2(v.w, v.w);
                    float2 racc = make_float2(0.f, 0.f), qacc = racc, pgb[2], pgc[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int e0 = 2 * q;
                        const float2 e = __fmul2_rn(dl2, A2[q]);
                        const float2 a = make_float2(ex2(e.x), ex2(e.y));
                        const float2 g = __ffma2_rn(dy2, cp[q], gcarry[q]);
                        gcarry[q] = __fmul2_rn(a, g);
                        const float2 hp = (jj == 0) ? make_float2(hprev[e0], hprev[e0 + 1])
                                                    : make_float2(hg[(jj - 1) * KS + e0], hg[(jj - 1) * KS + e0 + 1]);
                        const float2 pp = __fmul2_rn(gcarry[q], hp);
                        gAacc[q] = __ffma2_rn(pp, dl2, gAacc[q]);
                        racc = __ffma2_rn(pp, Af[q], racc);
                        qacc = __ffma2_rn(g, make_float2(bgr[jj * KS + e0], bgr[jj * KS + e0 + 1]), qacc);
                        pgb[q] = __fmul2_rn(g, dx2);                                            // gb terms
                        pgc[q] = __fmul2_rn(dy2, make_float2(hg[jj * KS + e0], hg[jj * KS + e0 + 1]));   // gc terms
                    }
                    const float part[8] = {pgb[0].x, pgb[0].y, pgb[1].x, pgb[1].y, pgc[0].x, pgc[0].y, pgc[1].x, pgc[1].y};
                    rr[jj] = racc.x + racc.y;
                    qq[jj] = qacc.x + qacc.y;
                    // sum over the warp's 8 channels; this lane keeps entry (cw >> 2, cw & 3)
                    gw[r * 2 * kDS + (cw >> 2) * kDS + s0 + (cw & 3)] = warp_reduce_scatter8(part, lane);
                }
                // sums over the channel's 4 lanes: this lane takes step rg + sg
                const float rs = reduce_scatter_steps<4>(rr, sg);
                const float qs = reduce_scatter_steps<4>(qq, sg);
                const int r = rg + sg;
                const float* vr = reinterpret_cast<const float*>(conv + r * C::CROW + c);
                const float dl = vr[0], xv = vr[2];
                const int64_t t = t0 + r;
                if (valid && t < ce) {
                    float gxv = dl * qs, gdv = rs + xv * qs;
                    if constexpr (FUSE) {
                        const float dyv = vr[3];
                        gxv = fmaf(Dk, dyv, gxv);                           // skip: y += D x
                        if (p.softplus) gdv *= sigmoid_from_softplus(dl);   // w.r.t. the raw delta
                        skip_acc = fmaf(dyv, xv, skip_acc);
                    }
                    gxg[t * D + d] = gxv;
                    gdg[t * D + d] = gdv;
                }
            }
        }
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (pend_t0 >= 0) flush_gbc(pend_t0, pend_lim);
    if (warp == 0) tmem_dealloc(tmem_base, C::TMEM_COLS);

    if constexpr (FUSE) {
        if (p.Dskip != nullptr) {      // gD[d] += sum over this CTA's steps of dy x (the 4 lanes' steps)
            skip_acc += __shfl_xor_sync(0xffffffffu, skip_acc, 1);
            skip_acc += __shfl_xor_sync(0xffffffffu, skip_acc, 2);
            if (valid && sg == 0) {
                if (p.det) p.part_gD[(b * gridDim.z + blockIdx.z) * D + d] = skip_acc;
                else atomicAdd(p.gDskip + d, skip_acc);
            }
        }
    }
    if (!valid) return;
#pragma unroll
    for (int s = 0; s < KS; ++s)
        if (jlo == 0) p.gh0[(b * D + d) * kDS + s0 + s] = (s & 1) ? gcarry[s >> 1].y : gcarry[s >> 1].x;
    if (p.det) {
        *reinterpret_cast<float4*>(p.part_gA + ((b * gridDim.z + blockIdx.z) * D + d) * kDS + s0) =
            make_float4(gAacc[0].x, gAacc[0].y, gAacc[1].x, gAacc[1].y);
    } else {
        red_add_v4(p.gA + d * kDS + s0, gAacc[0].x, gAacc[0].y, gAacc[1].x, gAacc[1].y);
    }
}

// Chunk-parallel backward, pass 1. The adjoint is linear in what enters a chunk from
// its end: with G_in the carried adjoint a_{ce} g_{ce} entering chunk [cs, ce),
//   a_{cs} g_{cs} = Z + exp(A * sum_{t in chunk} delta_t) * G_in,
// where Z is a_{cs} g_{cs} of the same chunk with zero adjoint entering it (the
// forward's chunked scan splits the state recurrence the same way). This kernel
// computes Z and the delta sum of chunks 1..nck-1 (chunk 0 passes its adjoint only
// to gh0, which pass 2 computes); pass 2 folds them into each chunk's G_in.
// Layout as bwd_kernel: 32 channels x 4 lanes of 4 states per CTA, one CTA per
// (channel block, batch, chunk).
template <typename TIO, bool VEC>
__global__ void __launch_bounds__(128) bwd_carry_kernel(const BwdLaunch p) {
    constexpr int NT = 128, KS = 4, DT = 32, LS = 16;
    __shared__ __align__(16) TIO dr[2][LS * DT], yr[2][LS * DT], cr[2][LS * kDS];

    const int tid = threadIdx.x;
    const int c = tid >> 2, sg = tid & 3, s0 = sg * KS;
    const int64_t T = p.T, D = p.D, K = p.K;
    const int64_t b = blockIdx.y;
    const int64_t j = int64_t(blockIdx.z) + 1;
    const int64_t d0 = int64_t(blockIdx.x) * DT;
    const int64_t d = d0 + c;
    const bool valid = d < D;
    const int64_t cs = j * K, ce = min(T, cs + K);
    const int ntile = int((ce - cs + LS - 1) / LS);

    const TIO* dg = static_cast<const TIO*>(p.delta) + b * T * D;
    const TIO* dyg = static_cast<const TIO*>(p.dy) + b * T * D;
    const TIO* cgl = static_cast<const TIO*>(p.c) + b * T * kDS;

    float A2[KS], gcar[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        A2[s] = valid ? p.A[d * kDS + s0 + s] * kLog2e : 0.f;
        gcar[s] = 0.f;
    }
    float dsum = 0.f;

    auto stage = [&](int buf, int64_t t0) {
        stage_tile<TIO, LS, DT, NT, VEC>(dr[buf], dg, D, t0, ce, d0);
        stage_tile<TIO, LS, DT, NT, VEC>(yr[buf], dyg, D, t0, ce, d0);
        stage_tile<TIO, LS, kDS, NT, true>(cr[buf], cgl, kDS, t0, ce, 0);
        cp_async_commit();
    };
    stage(0, cs + int64_t(ntile - 1) * LS);
    for (int ii = 0; ii < ntile; ++ii) {
        const int buf = ii & 1;
        if (ii + 1 < ntile) {
            stage(buf ^ 1, cs + int64_t(ntile - 2 - ii) * LS);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
#pragma unroll 4
        const int64_t rows = ce - (cs + int64_t(ntile - 1 - ii) * LS);
        for (int r = LS - 1; r >= 0; --r) {      // rows past ce are zero: a = 1, g unchanged
            float dl = to_f32(dr[buf][r * DT + c]);
            if (p.softplus) dl = (r < rows) ? softplus_f32(dl) : 0.f;
            const float dy = to_f32(yr[buf][r * DT + c]);
            float cc[KS];
            load_vals<TIO, KS>(cr[buf] + r * kDS + s0, cc);
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const float g = fmaf(dy, cc[s], gcar[s]);
                gcar[s] = ex2(dl * A2[s]) * g;
            }
            dsum += dl;
        }
        __syncthreads();
    }
    if (!valid) return;
    *reinterpret_cast<float4*>(p.carry_Z + ((j * p.B + b) * D + d) * kDS + s0) =
        make_float4(gcar[0], gcar[1], gcar[2], gcar[3]);
    if (sg == 0) p.carry_S[(j * p.B + b) * D + d] = dsum;
}

template <typename TIO>
cudaError_t launch_bwd_carry_io(const BwdLaunch& L, cudaStream_t stream) {
    auto kern = L.vec ? bwd_carry_kernel<TIO, true> : bwd_carry_kernel<TIO, false>;
    const int64_t nck = (L.T + L.K - 1) / L.K;
    const dim3 grid(unsigned((L.D + 31) / 32), unsigned(L.B), unsigned(nck - 1));
    kern<<<grid, 128, 0, stream>>>(L);
    return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_bwd_io(const BwdLaunch& L, cudaStream_t stream) {
    using C = BwdCfg<TIO>;
    const bool fuse = L.softplus || L.Dskip != nullptr;
    auto kern = fuse ? (L.vec ? bwd_kernel<TIO, true, true> : bwd_kernel<TIO, false, true>)
                     : (L.vec ? bwd_kernel<TIO, true, false> : bwd_kernel<TIO, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
    if (e != cudaSuccess) return e;
    const unsigned nz = L.tpar ? unsigned((L.T + L.K - 1) / L.K) : 1u;
    const dim3 grid(unsigned((L.D + C::DT - 1) / C::DT), unsigned(L.B), nz);
    kern<<<grid, C::NT, C::SMEM, stream>>>(L);
    return cudaGetLastError();
}

}  // namespace ssm
