// Backward scan kernel, two channels per lane.
//
// Same gradients and the same two-level recomputation as `bwd_kernel` (page
// "pssa_kernels.py", `scan_bwd`, with the ruDNN page's chunk-boundary
// rematerialisation), laid out for shapes with many (b, d) chains:
//
//   a lane holds 4 states of 2 neighbouring channels (8 chains), a warp 16
//   channels, a CTA of 128 threads 64 channels.
//
// What the second channel buys, per element: the b and c values a lane reads
// from shared memory serve 8 chains instead of 4; the per-step sums over d of
// gb and gc first add the lane's two channels in registers, so the lane
// reduce-scatter (two shuffle stages here, into per-half-warp slots that the
// per-tile flush adds) is paid once per 8 elements instead of once per 4; the
// (delta, delta*x) pair of both channels arrives in one 16-byte shared load.
//
// The reduce-scatter needs no selects: a lane keeps its 4 states in a
// lane-dependent order (register slot j holds state s0 + (j ^ m), with
// m = bits 1-2 of the lane's channel-pair index), chosen so that at each of the
// two stages every lane keeps the same register slots and sends the others,
// and its partner's sent slots hold exactly the states it kept. The b and c
// rows are kept in shared memory in all four orders, so the per-step loads are
// unchanged; only values loaded or stored once per chunk or per CTA (A, the
// checkpoints, ghT, gh0, gA) are permuted in registers.
//
// Where the extra per-thread state goes: the level-2 sub-checkpoints (the
// state entering every 16th step of the chunk, 8 floats per thread per
// sub-chunk) are parked in this CTA's own rows of the gx output for the chunk,
// which the reverse sweep overwrites only after it has read them back (the
// sub-checkpoint of sub-chunk i sits in the 16 rows of sub-chunk i, one state
// per row, one channel per column; the last sub-chunk of a chunk, which may be
// short, keeps its start state in registers). The round trip stays in L2. The
// level-3 window (h_t of both channels, 16 steps, 128 columns) is in tensor
// memory and b_t comes from shared memory, so shared memory per CTA is 41 KB
// (48 KB with float32 I/O) and three CTAs (12 warps) are resident per SM, each
// thread with up to 168 registers. As in `bwd_kernel`, the per-state arithmetic
// is packed f32x2 on pairs of neighbouring states.
#pragma once

#include "ssm_bwd_impl.cuh"

namespace ssm {

template <typename TIO>
struct Bwd2Cfg {
    static constexpr int NT = 128;
    static constexpr int NW = NT / 32;
    static constexpr int G = 4;                         // lanes per channel pair
    static constexpr int KS = kDS / G;                  // states per lane (4)
    static constexpr int KD = 2;                        // channels per lane
    static constexpr int NP = NT / G;                   // channel pairs per CTA (32)
    static constexpr int DT = NP * KD;                  // channels per CTA (64)
    static constexpr int LS = 16;                       // sub-chunk (tile) length
    static constexpr int EPC = 16 / int(sizeof(TIO));
    static constexpr int X_CPR = DT / EPC;              // 16-byte chunks per raw tile row
    static constexpr int X_CH = LS * X_CPR;             // chunks per raw tile (128 bf16, 256 f32)
    static constexpr int X_PT = X_CH / NT;              // chunks per thread
    static constexpr int BC_CH = LS * kDS / EPC;
    static_assert(X_CH % NT == 0, "raw tile chunks must split evenly over the CTA");
    // shared memory (bytes)
    static constexpr size_t RAW_X = size_t(LS) * DT * sizeof(TIO);          // one of x, delta, dy
    static constexpr size_t RAW_BC = size_t(LS) * kDS * sizeof(TIO);        // one of b, c
    // converted records, one float4 per (step, pair); rows padded by one float4 so that the 4 lanes
    // of a pair, which read 4 different steps at once in the per-step sums, hit different banks
    static constexpr int CROW = NP + 1;
    static constexpr size_t CONV1 = size_t(LS) * CROW * 16;                 // (d0, d0*x0, d1, d1*x1)
    static constexpr size_t CONV2 = size_t(LS) * CROW * 16;                 // (dy0, dy1, x0, x1)
    static constexpr size_t BCF = size_t(4) * LS * kDS * 4;                 // one of b, c as float32, 4 state orders
    // per-half-warp gb, gc sums of a tile, [2 NW][LS][2][16] floats; sets padded by 16 floats so
    // the two sets a warp writes at once fall on different banks
    static constexpr int GSET = LS * 2 * kDS + 16;
    static constexpr size_t GBC = size_t(2 * NW) * GSET * 4;
    static constexpr size_t SMEM = 3 * RAW_X + 2 * RAW_BC + CONV1 + CONV2 + 2 * BCF + GBC + 16;
    // tensor memory columns per lane: h of both channels per step
    static constexpr uint32_t TMEM_H_STEP = KD * KS;                        // 8
    static constexpr uint32_t TMEM_COLS = LS * TMEM_H_STEP;                 // 128
    // 3 resident CTAs per SM take 384 of the 512 columns; a CTA that ever found them all
    // taken would wait in tcgen05.alloc for a resident CTA to finish, never the reverse
    static_assert(3 * TMEM_COLS <= 512, "three resident CTAs must fit in tensor memory");
};


// The lane's 4 states of one channel between state order (s0 .. s0 + 3) and its register-slot
// order (slot j = state s0 + (j ^ m)); the map is its own inverse.
__device__ __forceinline__ float4 perm4(float4 v, int m) {
    float4 r = (m & 2) ? make_float4(v.z, v.w, v.x, v.y) : v;
    return (m & 1) ? make_float4(r.y, r.x, r.w, r.z) : r;
}

template <typename TIO, bool VEC, bool FUSE>
__global__ void __launch_bounds__(128, 3) bwd2_kernel(const BwdLaunch p) {
    using C = Bwd2Cfg<TIO>;
    constexpr int NT = C::NT, KS = C::KS, NP = C::NP, DT = C::DT, LS = C::LS, EPC = C::EPC;
    constexpr int KP = KS / 2;                  // state pairs per lane and channel
    constexpr int HS = int(C::TMEM_H_STEP);

    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* ptr = smem;
    TIO* xr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_X;
    TIO* dr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_X;
    TIO* yr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_X;
    TIO* br = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_BC;
    TIO* cr = reinterpret_cast<TIO*>(ptr);  ptr += C::RAW_BC;
    float4* conv1 = reinterpret_cast<float4*>(ptr); ptr += C::CONV1;   // [LS][CROW]
    float4* conv2 = reinterpret_cast<float4*>(ptr); ptr += C::CONV2;   // [LS][CROW]
    float* bfp = reinterpret_cast<float*>(ptr);     ptr += C::BCF;     // [4 orders][LS][16]
    float* cfp = reinterpret_cast<float*>(ptr);     ptr += C::BCF;
    float* gbc = reinterpret_cast<float*>(ptr);     ptr += C::GBC;     // [2 NW][GSET]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ptr);

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int cw = lane >> 2;               // channel pair within the warp
    const int sg = lane & 3;                // state group within the pair
    const int pc = warp * 8 + cw;           // channel pair within the CTA
    const int s0 = sg * KS;
    const int m = (cw >> 1) & 3;            // register slot j holds state s0 + (j ^ m)
    // b and c rows in this lane's state order
    const float* bf = bfp + m * LS * kDS;
    const float* cf = cfp + m * LS * kDS;
    const int64_t T = p.T, D = p.D, K = p.K;
    const int64_t b = blockIdx.y;
    const int64_t d0 = int64_t(blockIdx.x) * DT;
    const int64_t dch[2] = {d0 + 2 * pc, d0 + 2 * pc + 1};
    const bool valid[2] = {dch[0] < D, dch[1] < D};
    const bool full_d = d0 + DT <= D;

    const TIO* xg = static_cast<const TIO*>(p.x) + b * T * D;
    const TIO* dg = static_cast<const TIO*>(p.delta) + b * T * D;
    const TIO* dyg = static_cast<const TIO*>(p.dy) + b * T * D;
    const TIO* bg = static_cast<const TIO*>(p.b) + b * T * kDS;
    const TIO* cgl = static_cast<const TIO*>(p.c) + b * T * kDS;
    float* gxg = p.gx + b * T * D;
    float* gdg = p.gdelta + b * T * D;

    // per channel k and state s of this lane: A*log2(e), the carried adjoint a_{t+1} g_{t+1}, gA
    float Dk[2], skip_acc[2] = {0.f, 0.f};       // skip weights, sums of dy x (fused variant)
#pragma unroll
    for (int k = 0; k < 2; ++k) Dk[k] = (FUSE && valid[k] && p.Dskip != nullptr) ? p.Dskip[dch[k]] : 0.f;
    // Per-state values are kept as pairs of neighbouring states (float2), so that the
    // arithmetic runs as packed f32x2 operations: on sm_103a these issue fewer instructions
    // per element than scalar ones (measured on the forward: 7 % faster).
    float2 A2[2][KP], gcar[2][KP], gAacc[2][KP];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), g4 = a4;
        if (valid[k]) {
            a4 = perm4(*reinterpret_cast<const float4*>(p.A + dch[k] * kDS + s0), m);
            if (p.ghT != nullptr) g4 = perm4(*reinterpret_cast<const float4*>(p.ghT + (b * D + dch[k]) * kDS + s0), m);
        }
        A2[k][0] = make_float2(a4.x * kLog2e, a4.y * kLog2e);
        A2[k][1] = make_float2(a4.z * kLog2e, a4.w * kLog2e);
        gcar[k][0] = make_float2(g4.x, g4.y);
        gcar[k][1] = make_float2(g4.z, g4.w);
        gAacc[k][0] = gAacc[k][1] = make_float2(0.f, 0.f);
    }

    // level-3 window in tensor memory: this warp's 32 lanes x 128 columns
    if (warp == 0) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t tw = tmem_base + (uint32_t((warp & 3) * 32) << 16);

    // this thread's 16-byte chunks of a full raw tile (x, delta, dy) and of b, c
    int x_goff[C::X_PT], x_soff[C::X_PT];
#pragma unroll
    for (int q = 0; q < C::X_PT; ++q) {
        const int i = tid + q * NT;
        const int r = i / C::X_CPR, col = (i % C::X_CPR) * EPC;
        x_goff[q] = r * int(D) + col;
        x_soff[q] = r * DT + col;
    }

    auto stage = [&](int64_t t0, int64_t tend, bool rev) {
        if (VEC && full_d && t0 + LS <= tend) {
            const int64_t base = t0 * D + d0;
#pragma unroll
            for (int q = 0; q < C::X_PT; ++q) {
                cp_async16(xr + x_soff[q], xg + base + x_goff[q], 16);
                cp_async16(dr + x_soff[q], dg + base + x_goff[q], 16);
                if (rev) cp_async16(yr + x_soff[q], dyg + base + x_goff[q], 16);
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
    // raw tile -> (d0, d0*x0, d1, d1*x1) and (dy0, dy1, x0, x1) per (step, pair); float32 b, c rows
    // (rows >= rows_valid are padding: with softplus their delta must stay 0, not ln 2)
    auto convert = [&](bool rev, int64_t rows_valid) {
#pragma unroll
        for (int q = 0; q < LS * NP / NT; ++q) {
            const int i = tid + NT * q;
            const int r = i / NP, pp = i % NP;
            float dl[2], xv[2];
            load_vals<TIO, 2>(dr + r * DT + 2 * pp, dl);
            if (FUSE && p.softplus) {
                const float2 sp = softplus2_f32(make_float2(dl[0], dl[1]));
                dl[0] = r < rows_valid ? sp.x : 0.f;
                dl[1] = r < rows_valid ? sp.y : 0.f;
            }
            load_vals<TIO, 2>(xr + r * DT + 2 * pp, xv);
            conv1[r * C::CROW + pp] = make_float4(dl[0], dl[0] * xv[0], dl[1], dl[1] * xv[1]);
            if (rev) {
                float dyv[2];
                load_vals<TIO, 2>(yr + r * DT + 2 * pp, dyv);
                conv2[r * C::CROW + pp] = make_float4(dyv[0], dyv[1], xv[0], xv[1]);
            }
        }
        // b (threads 0-63) and c (threads 64-127): 4 states of one row each, stored in the four
        // state orders (order mm holds state s ^ mm at position s)
        {
            const int q = tid & 63, r = q >> 2, g = (q & 3) * 4;
            if (tid < 64 || rev) {
                const TIO* raw = tid < 64 ? br : cr;
                float* dst = tid < 64 ? bfp : cfp;
                float v[4];
                load_vals<TIO, 4>(raw + r * kDS + g, v);
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    *reinterpret_cast<float4*>(dst + mm * LS * kDS + r * kDS + g) =
                        make_float4(v[0 ^ mm], v[1 ^ mm], v[2 ^ mm], v[3 ^ mm]);
            }
        }
    };
    // gb, gc of the tile starting at t0: sum the warps' slots, add to global (rows below t_lim)
    auto flush_gbc = [&](int64_t t0, int64_t t_lim) {
        const int r = tid >> 3, tau = (tid >> 2) & 1, q = tid & 3;
        const int off = r * 2 * kDS + tau * kDS + q * 4;
        float4 v4 = *reinterpret_cast<const float4*>(gbc + off);
        float2 lo = make_float2(v4.x, v4.y), hi = make_float2(v4.z, v4.w);
#pragma unroll
        for (int w = 1; w < 2 * C::NW; ++w) {
            const float4 u = *reinterpret_cast<const float4*>(gbc + w * C::GSET + off);
            lo = __fadd2_rn(lo, make_float2(u.x, u.y));
            hi = __fadd2_rn(hi, make_float2(u.z, u.w));
        }
        const float4 v = make_float4(lo.x, lo.y, hi.x, hi.y);
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
    int64_t pend_t0 = -1, pend_lim = 0;       // tile whose gb/gc sums await their flush
    for (int64_t j = nck - 1; j >= 0; --j) {
        const int64_t cs = j * K;
        const int64_t ce = min(T, cs + K);
        const int nsub = int((ce - cs + LS - 1) / LS);

        // ---- level 2: forward over the chunk, keeping sub-chunk start states
        float h[2][KS];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid[k]) v = perm4(*reinterpret_cast<const float4*>(p.ckpt + ((j * p.B + b) * D + dch[k]) * kDS + s0), m);
            h[k][0] = v.x; h[k][1] = v.y; h[k][2] = v.z; h[k][3] = v.w;
        }
        float hlast[2 * KS];                 // start state of the chunk's last sub-chunk
        stage(cs, ce, false);
        for (int i = 0; i < nsub; ++i) {
            cp_async_wait<0>();
            __syncthreads();
            convert(false, ce - (cs + int64_t(i) * LS));
            __syncthreads();
            if (i + 1 < nsub) stage(cs + int64_t(i + 1) * LS, ce, false);
            if (i + 1 < nsub) {
                // full sub-chunk: park its start state in its own gx rows (state s0+s in row t0+s0+s)
                float* dst = gxg + (cs + int64_t(i) * LS + s0) * D + dch[0];
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    if (VEC && valid[1]) {
                        *reinterpret_cast<float2*>(dst + s * D) = make_float2(h[0][s], h[1][s]);
                    } else {
                        if (valid[0]) dst[s * D] = h[0][s];
                        if (valid[1]) dst[s * D + 1] = h[1][s];
                    }
                }
            } else {
#pragma unroll
                for (int s = 0; s < KS; ++s) { hlast[s] = h[0][s]; hlast[KS + s] = h[1][s]; }
            }
            float2 hp2[2][KP];
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int q = 0; q < KP; ++q) hp2[k][q] = make_float2(h[k][2 * q], h[k][2 * q + 1]);
            auto level2_step = [&](int r) {
                const float4 v = conv1[r * C::CROW + pc];                                   // d0, d0 x0, d1, d1 x1
                const float4 b4 = *reinterpret_cast<const float4*>(bf + r * kDS + s0);
                const float2 bp[KP] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
                const float2 dl2[2] = {make_float2(v.x, v.x), make_float2(v.z, v.z)};
                const float2 dx2[2] = {make_float2(v.y, v.y), make_float2(v.w, v.w)};
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int q = 0; q < KP; ++q) {
                        const float2 e = __fmul2_rn(dl2[k], A2[k][q]);
                        hp2[k][q] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), hp2[k][q], __fmul2_rn(dx2[k], bp[q]));
                    }
            };
            if (i + 1 < nsub) {
#pragma unroll 8
                for (int r = 0; r < LS; ++r) level2_step(r);
            } else {
                // the chunk's last sub-chunk, which the reverse takes first: its states go straight
                // into the window, so the reverse skips level 3 for it
#pragma unroll 8
                for (int r = 0; r < LS; ++r) {
                    level2_step(r);
                    const float hv[8] = {hp2[0][0].x, hp2[0][0].y, hp2[0][1].x, hp2[0][1].y,
                                         hp2[1][0].x, hp2[1][0].y, hp2[1][1].x, hp2[1][1].y};
                    tmem_st8(tw + uint32_t(r * HS), hv);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int q = 0; q < KP; ++q) { h[k][2 * q] = hp2[k][q].x; h[k][2 * q + 1] = hp2[k][q].y; }
        }

        // ---- reverse over the sub-chunks
        stage(cs + int64_t(nsub - 1) * LS, ce, true);
        for (int ii = 0; ii < nsub; ++ii) {
            const int i = nsub - 1 - ii;
            const int64_t t0 = cs + int64_t(i) * LS;
            cp_async_wait<0>();
            __syncthreads();
            // start state of this sub-chunk, read back before the barrier that precedes any
            // gx store of the sub-chunk
            float hs[2 * KS];
            if (ii == 0) {
#pragma unroll
                for (int e = 0; e < 2 * KS; ++e) hs[e] = hlast[e];
            } else {
                const float* src = gxg + (t0 + s0) * D + dch[0];
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    if (VEC && valid[1]) {
                        const float2 v = *reinterpret_cast<const float2*>(src + s * D);
                        hs[s] = v.x; hs[KS + s] = v.y;
                    } else {
                        hs[s] = valid[0] ? src[s * D] : 0.f;
                        hs[KS + s] = valid[1] ? src[s * D + 1] : 0.f;
                    }
                }
            }
            if (pend_t0 >= 0) flush_gbc(pend_t0, pend_lim);
            convert(true, ce - t0);
            __syncthreads();
            if (ii + 1 < nsub) stage(t0 - LS, ce, true);
            pend_t0 = t0;
            pend_lim = ce;

            // level 3: states of this sub-chunk into the window (8 columns per step); the first
            // sub-chunk of the reverse (the chunk's last) was written by level 2
            if (ii > 0) {
                float2 hc[2][KP];
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int q = 0; q < KP; ++q) hc[k][q] = make_float2(hs[k * KS + 2 * q], hs[k * KS + 2 * q + 1]);
#pragma unroll
                for (int r = 0; r < LS; ++r) {
                    const float4 v = conv1[r * C::CROW + pc];
                    const float4 b4 = *reinterpret_cast<const float4*>(bf + r * kDS + s0);
                    const float2 bp[KP] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
                    const float2 dl2[2] = {make_float2(v.x, v.x), make_float2(v.z, v.z)};
                    const float2 dx2[2] = {make_float2(v.y, v.y), make_float2(v.w, v.w)};
#pragma unroll
                    for (int k = 0; k < 2; ++k)
#pragma unroll
                        for (int q = 0; q < KP; ++q) {
                            const float2 e = __fmul2_rn(dl2[k], A2[k][q]);
                            hc[k][q] = __ffma2_rn(make_float2(ex2(e.x), ex2(e.y)), hc[k][q], __fmul2_rn(dx2[k], bp[q]));
                        }
                    const float hv[8] = {hc[0][0].x, hc[0][0].y, hc[0][1].x, hc[0][1].y,
                                         hc[1][0].x, hc[1][0].y, hc[1][1].x, hc[1][1].y};
                    tmem_st8(tw + uint32_t(r * HS), hv);
                }
                tmem_wait_st();
            }

            // this lane's slot set: sums over the 4 channel pairs {cw, cw^2, cw^4, cw^6} of its warp;
            // the lane ends with the sums of state s0 + m
            float* gw = gbc + (warp * 2 + (cw & 1)) * C::GSET + s0 + m;
            // reverse sweep over the sub-chunk, 4 steps per lane reduce-scatter group
#pragma unroll 2
            for (int rg = LS - 4; rg >= 0; rg -= 4) {
                float hg[4 * HS], hprev[HS];   // h for steps rg..rg+3 and for step rg-1
                tmem_ld32(tw + uint32_t(rg * HS), hg);
                if (rg > 0) {
                    tmem_ld8(tw + uint32_t((rg - 1) * HS), hprev);
                } else {
#pragma unroll
                    for (int e = 0; e < HS; ++e) hprev[e] = hs[e];
                }
                tmem_wait_ld();
                float rr[2][4], qq[2][4];
#pragma unroll
                for (int jj = 3; jj >= 0; --jj) {
                    const int r = rg + jj;
                    const float4 v = conv1[r * C::CROW + pc];                                           // d0, d0 x0, d1, d1 x1
                    const float2 dyv = *reinterpret_cast<const float2*>(conv2 + r * C::CROW + pc);      // dy0, dy1
                    const float4 c4 = *reinterpret_cast<const float4*>(cf + r * kDS + s0);
                    const float4 b4 = *reinterpret_cast<const float4*>(bf + r * kDS + s0);
                    const float2 cp[KP] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
                    const float2 bp[KP] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
                    const float2 dl2[2] = {make_float2(v.x, v.x), make_float2(v.z, v.z)};
                    const float2 dx2[2] = {make_float2(v.y, v.y), make_float2(v.w, v.w)};
                    const float2 dy2[2] = {make_float2(dyv.x, dyv.x), make_float2(dyv.y, dyv.y)};
                    float2 pgb[KP], pgc[KP];                  // gb, gc terms of the lane's two channels
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float2 racc = make_float2(0.f, 0.f), qacc = racc;
#pragma unroll
                        for (int q = 0; q < KP; ++q) {
                            const int e0 = k * KS + 2 * q;
                            const float2 e = __fmul2_rn(dl2[k], A2[k][q]);
                            const float2 a = make_float2(ex2(e.x), ex2(e.y));
                            const float2 g = __ffma2_rn(dy2[k], cp[q], gcar[k][q]);
                            gcar[k][q] = __fmul2_rn(a, g);
                            const float2 hp = (jj == 0) ? make_float2(hprev[e0], hprev[e0 + 1])
                                                        : make_float2(hg[(jj - 1) * HS + e0], hg[(jj - 1) * HS + e0 + 1]);
                            const float2 pp = __fmul2_rn(gcar[k][q], hp);
                            gAacc[k][q] = __ffma2_rn(pp, dl2[k], gAacc[k][q]);
                            racc = __ffma2_rn(pp, A2[k][q], racc);      // times ln 2 below
                            qacc = __ffma2_rn(g, bp[q], qacc);
                            const float2 ht = make_float2(hg[jj * HS + e0], hg[jj * HS + e0 + 1]);
                            if (k == 0) {
                                pgb[q] = __fmul2_rn(g, dx2[0]);
                                pgc[q] = __fmul2_rn(dy2[0], ht);
                            } else {
                                pgb[q] = __ffma2_rn(g, dx2[1], pgb[q]);
                                pgc[q] = __ffma2_rn(dy2[1], ht, pgc[q]);
                            }
                        }
                        rr[k][jj] = racc.x + racc.y;
                        qq[k][jj] = qacc.x + qacc.y;
                    }
                    // Sum over the channel pairs {cw, cw^4} (lane ^ 16) and then {cw, cw^2} (lane ^ 8):
                    // every lane keeps slots 0, 1 and sends 2, 3, then keeps slot 0 and sends 1; the
                    // partner's sent slots hold the states this lane kept (its m differs in bit 1,
                    // then in bit 0), so no selects are needed.
                    {
                        const float2 rb = make_float2(__shfl_xor_sync(0xffffffffu, pgb[1].x, 16),
                                                      __shfl_xor_sync(0xffffffffu, pgb[1].y, 16));
                        const float2 rc = make_float2(__shfl_xor_sync(0xffffffffu, pgc[1].x, 16),
                                                      __shfl_xor_sync(0xffffffffu, pgc[1].y, 16));
                        const float2 sb = __fadd2_rn(pgb[0], rb);      // slots 0, 1 of gb
                        const float2 sc = __fadd2_rn(pgc[0], rc);      // slots 0, 1 of gc
                        const float2 r2 = make_float2(__shfl_xor_sync(0xffffffffu, sb.y, 8),
                                                      __shfl_xor_sync(0xffffffffu, sc.y, 8));
                        const float2 v2 = __fadd2_rn(make_float2(sb.x, sc.x), r2);
                        gw[r * 2 * kDS] = v2.x;                        // gb of state s0 + m
                        gw[r * 2 * kDS + kDS] = v2.y;                  // gc
                    }
                }
                // sums over the pair's 4 lanes: this lane takes step rg + sg of both channels
                float rs[2], qs[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float2 rq = reduce_scatter_steps4_pair(rr[k], qq[k], sg);
                    rs[k] = rq.x;
                    qs[k] = rq.y;
                }
                const int r = rg + sg;
                const float4 v = conv1[r * C::CROW + pc];
                const float4 w = conv2[r * C::CROW + pc];
                const int64_t t = t0 + r;
                if (t < ce) {
                    float gx0 = v.x * qs[0], gx1 = v.z * qs[1];
                    // (A = A2 ln 2)
                    float gd0 = fmaf(rs[0], kLn2, w.z * qs[0]), gd1 = fmaf(rs[1], kLn2, w.w * qs[1]);
                    if constexpr (FUSE) {
                        gx0 = fmaf(Dk[0], w.x, gx0);                   // skip: y += D x
                        gx1 = fmaf(Dk[1], w.y, gx1);
                        if (p.softplus) {                              // w.r.t. the raw delta
                            gd0 *= sigmoid_from_softplus(v.x);
                            gd1 *= sigmoid_from_softplus(v.z);
                        }
                        skip_acc[0] = fmaf(w.x, w.z, skip_acc[0]);
                        skip_acc[1] = fmaf(w.y, w.w, skip_acc[1]);
                    }
                    if (VEC && valid[1]) {
                        *reinterpret_cast<float2*>(gxg + t * D + dch[0]) = make_float2(gx0, gx1);
                        *reinterpret_cast<float2*>(gdg + t * D + dch[0]) = make_float2(gd0, gd1);
                    } else {
                        if (valid[0]) { gxg[t * D + dch[0]] = gx0; gdg[t * D + dch[0]] = gd0; }
                        if (valid[1]) { gxg[t * D + dch[1]] = gx1; gdg[t * D + dch[1]] = gd1; }
                    }
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
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float v = skip_acc[k];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                if (valid[k] && sg == 0) {
                    if (p.det) p.part_gD[b * D + dch[k]] = v;
                    else atomicAdd(p.gDskip + dch[k], v);
                }
            }
        }
    }

#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (!valid[k]) continue;
        *reinterpret_cast<float4*>(p.gh0 + (b * D + dch[k]) * kDS + s0) =
            perm4(make_float4(gcar[k][0].x, gcar[k][0].y, gcar[k][1].x, gcar[k][1].y), m);
        const float4 ga = perm4(make_float4(gAacc[k][0].x, gAacc[k][0].y, gAacc[k][1].x, gAacc[k][1].y), m);
        if (p.det) {
            *reinterpret_cast<float4*>(p.part_gA + (b * D + dch[k]) * kDS + s0) = ga;
        } else {
            red_add_v4(p.gA + dch[k] * kDS + s0, ga.x, ga.y, ga.z, ga.w);
        }
    }
}

template <typename TIO>
cudaError_t launch_bwd2_io(const BwdLaunch& L, cudaStream_t stream) {
    using C = Bwd2Cfg<TIO>;
    const bool fuse = L.softplus || L.Dskip != nullptr;
    auto kern = fuse ? (L.vec ? bwd2_kernel<TIO, true, true> : bwd2_kernel<TIO, false, true>)
                     : (L.vec ? bwd2_kernel<TIO, true, false> : bwd2_kernel<TIO, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
    if (e != cudaSuccess) return e;
    const dim3 grid(unsigned((L.D + C::DT - 1) / C::DT), unsigned(L.B));
    kern<<<grid, C::NT, C::SMEM, stream>>>(L);
    return cudaGetLastError();
}
}  // namespace ssm
