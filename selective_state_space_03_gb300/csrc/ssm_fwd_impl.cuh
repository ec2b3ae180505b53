// Forward scan kernels: one pass over T, the two passes of the chunked scan, and
// the chunked scan in one launch with decoupled look-back (fwd_lookback_kernel).
//
// Recurrence (page "pssa_kernels.py", module docstring and `scan_reference`):
//   h_t = exp(delta_t A) h_{t-1} + delta_t b_t x_t,   y_t = <h_t, c_t>.
// Chunked scan (for shapes with too few (b, d) chains to fill the GPU): the
// recurrence is affine in h, so chunk k maps its start state H to
// P_k * H + S_k with P_k[s] = exp(A[s] * sum of delta over the chunk) and S_k
// the chunk's end state from a zero start. Pass 1 computes S_k and the delta
// sums of every chunk but the last; pass 2 folds the carries of chunks 0..k-1
// into the start state of chunk k and rescans the chunk with readout.
//
// Work per element is one ex2 on the MUFU (32/clk/SM on GB300) and four FP32
// operations (delta*A, delta*x*b, a*h + u, h*c), i.e. the MUFU and the FP32
// pipe (128 lanes/clk/SM) are both busy 1/32 clk per element: the kernel is
// built to spend as few issue slots as possible on anything else.
//  - One-warp CTAs, so the grid spreads evenly over the SMs and late CTAs run
//    alone at full speed instead of leaving a quantised last wave.
//  - A lane owns KD neighbouring channels x 16/G states (kept in registers for
//    the whole sweep); each channel's 16 states are split over G lanes. b and c
//    are the same for every channel, so each b/c value a lane reads from
//    shared memory feeds KD channels: broadcast shared loads deliver only 4
//    bytes per wavefront, which would cap the kernel at 16*KD elements per
//    clock per SM. Layouts (G, KD): (2, 2) when there are enough (b, d) chains,
//    then (4, 2), then (4, 1) as chains get fewer; the chunk passes use (4, 2)
//    or (4, 1). State pairs use packed FP32x2 multiply/FMA.
//  - x, delta, b, c tiles of TT steps are double-buffered in shared memory with
//    16-byte cp.async, zero-filled past the end (delta = 0 gives decay 1 and no
//    input, so padded steps leave the state unchanged). bf16 b and c are
//    widened to float32 once per tile.
//  - The readout <h_t, c_t> is finished across the G lanes of a channel: with
//    G = 2 by one exchange that splits the lane pair's channels, with G = 4 by
//    a reduce-scatter over 4 steps (and the lane's KD channels). y goes to a shared-memory tile and leaves in
//    16-byte stores once per tile; checkpoints are written at tile starts when
//    every checkpoint step is one; staging offsets are per-lane constants, so a
//    full tile costs a few instructions per 16-byte chunk.
#pragma once

#include <type_traits>

#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

enum FwdMode { kSingle = 0, kPass1 = 1, kPass2 = 2, kCkptOnly = 3, kLookback = 4 };

template <typename TIO, int G, int KD>
struct FwdCfg {
    static constexpr int NT = 32;                                // one warp per CTA
    static constexpr int KS = kDS / G;                           // states per lane
    static constexpr int KP = KS / 2;                            // state pairs per lane
    static constexpr int DT = NT / G * KD;                       // channels per CTA
    static constexpr int TT = 16;                                // steps per tile
    static constexpr bool BF = std::is_same<TIO, __nv_bfloat16>::value;
    static constexpr int EPC = 16 / int(sizeof(TIO));           // I/O elements per 16-byte chunk
    static constexpr int X_CPR = DT / EPC;                       // x/delta chunks per tile row
    static constexpr int X_CH = TT * X_CPR;                      // x/delta chunks per tile
    static constexpr int X_PL = (X_CH + NT - 1) / NT;            // ... per lane
    static constexpr int BC_CPR = kDS / EPC;
    static constexpr int BC_CH = TT * BC_CPR;
    static constexpr int BC_PL = (BC_CH + NT - 1) / NT;
    static constexpr int Y_CH = TT * X_CPR;                      // y chunks per tile
    static constexpr int Y_PL = (Y_CH + NT - 1) / NT;
    // staging buffers per tensor: tiles are loaded NBUF - 1 tiles ahead (3 or 4 buffers for the
    // low-occupancy layouts measured no faster than 2)
    static constexpr int NBUF = 2;
    static constexpr size_t X_BYTES = size_t(NBUF) * TT * DT * sizeof(TIO);     // one tensor
    static constexpr size_t BC_RAW = size_t(NBUF) * TT * kDS * sizeof(TIO);    // one tensor
    static constexpr size_t BC_F32 = BF ? size_t(TT) * kDS * 4 : 0;          // widened copy (bf16)
    static constexpr size_t Y_BYTES = size_t(TT) * DT * sizeof(TIO);
    static constexpr size_t SMEM = 2 * X_BYTES + 2 * BC_RAW + 2 * BC_F32 + Y_BYTES;
    // fused variant: delta of the current tile as float32 (softplus applied when asked)
    static constexpr size_t DSF_BYTES = size_t(TT) * DT * 4;
    static constexpr size_t SMEM_FUSE = SMEM + DSF_BYTES;
    // registers: keep enough warps resident for the whole grid of the largest shapes
    static constexpr int MINB = (KD == 2) ? 20 : 1;
    static_assert(KD == 1 || (KD == 2 && (G == 2 || G == 4)), "layouts: (4,1), (4,2), (2,2)");
    static_assert(X_CPR >= 1 && DT % EPC == 0, "tile rows must be whole 16-byte chunks");
};

// The lane's KD x KS states into a (.., D, 16) array (rows of chains b * D + d); channel slot k
// of the lane holds channel dfirst + (k ^ perm).
template <int G, int KD>
__device__ __forceinline__ void store_lane_states(float* base, int64_t b, int64_t D, int64_t dfirst, int s0,
                                                  const bool (&valid)[KD], const float2 (&h)[KD][kDS / G / 2],
                                                  int perm = 0) {
#pragma unroll
    for (int k = 0; k < KD; ++k) {
        if (!valid[k]) continue;
        float4* dst = reinterpret_cast<float4*>(base + (b * D + dfirst + (k ^ perm)) * kDS + s0);
#pragma unroll
        for (int q = 0; q < kDS / G / 2; q += 2)
            dst[q / 2] = make_float4(h[k][q].x, h[k][q].y, h[k][q + 1].x, h[k][q + 1].y);
    }
}

// One sweep of one warp over steps [t_begin, t_end) of batch b, channels d0 .. d0 + DT - 1,
// starting from the state in h and leaving the end state there. MODE selects the work:
// kSingle / kPass2 read out y (and write checkpoints), kPass1 adds up delta per channel into
// dsum (no readout, no checkpoints), kCkptOnly writes checkpoints only.
template <typename TIO, int G, int KD, bool VEC, int MODE, bool CKT, bool FUSE>
__device__ __forceinline__ void fwd_sweep(const FwdLaunch& p, int64_t b, int64_t d0, int64_t t_begin, int64_t t_end,
                                          const float2 (&A2)[KD][FwdCfg<TIO, G, KD>::KP], const bool (&valid)[KD],
                                          float2 (&h)[KD][FwdCfg<TIO, G, KD>::KP], float (&dsum)[KD]) {
    using C = FwdCfg<TIO, G, KD>;
    constexpr int NT = C::NT, KS = C::KS, KP = C::KP, DT = C::DT, TT = C::TT, EPC = C::EPC;
    constexpr bool READ = (MODE == kSingle || MODE == kPass2);

    extern __shared__ __align__(16) unsigned char smem[];
    TIO* xs = reinterpret_cast<TIO*>(smem);
    TIO* ds = reinterpret_cast<TIO*>(smem + C::X_BYTES);
    TIO* bsr = reinterpret_cast<TIO*>(smem + 2 * C::X_BYTES);
    TIO* csr = reinterpret_cast<TIO*>(smem + 2 * C::X_BYTES + C::BC_RAW);
    float* bsf = reinterpret_cast<float*>(smem + 2 * C::X_BYTES + 2 * C::BC_RAW);
    float* csf = bsf + (C::BF ? TT * kDS : 0);
    TIO* ys = reinterpret_cast<TIO*>(smem + 2 * C::X_BYTES + 2 * C::BC_RAW + 2 * C::BC_F32);
    float* dsf = reinterpret_cast<float*>(smem + C::SMEM);           // FUSE only

    const int lane = threadIdx.x;
    const int gl = lane % G;                 // lane within the channel group
    const int c0 = (lane / G) * KD;          // first channel of this lane within the CTA
    const int s0 = gl * KS;
    const int64_t T = p.T, D = p.D;
    const bool full_d = d0 + DT <= D;
    // Two lanes per channel pair with bf16 I/O: lane gl holds its channels in the order
    // (c0 + gl, c0 + (gl ^ 1)), so that the readout exchange keeps slot 0 and sends slot 1 on
    // every lane (no selects); the bf16 pairs are unpacked into that order by byte permutes
    // whose selectors are per-lane constants.
    constexpr bool PERM = (G == 2 && C::BF);
    const int perm = PERM ? gl : 0;
    const uint32_t sel0 = gl ? 0x3244u : 0x1044u, sel1 = gl ? 0x1044u : 0x3244u;

    const TIO* xg = static_cast<const TIO*>(p.x) + b * T * D;
    const TIO* dg = static_cast<const TIO*>(p.delta) + b * T * D;
    const TIO* bg = static_cast<const TIO*>(p.b) + b * T * kDS;
    const TIO* cgl = static_cast<const TIO*>(p.c) + b * T * kDS;
    TIO* yg = static_cast<TIO*>(p.y) + b * T * D;

    // Readout: with G = 4 the lanes of a chain group each finish one step of every G steps,
    // for all KD channels; with G = 2 each finishes KD / 2 of the channels, every step.
    constexpr bool BY_STEP = (G == 4);
    // skip weights of the channels whose y this lane stores
    constexpr int NKEEP = BY_STEP ? KD : KD / 2;
    float Dkeep[NKEEP];
#pragma unroll
    for (int i = 0; i < NKEEP; ++i) {
        const int cc = BY_STEP ? c0 + i : c0 + gl * NKEEP + i;
        Dkeep[i] = (FUSE && READ && p.Dskip != nullptr && d0 + cc < D) ? p.Dskip[d0 + cc] : 0.f;
    }
    const int64_t K = p.K;
    const bool want_ckpt = (MODE != kPass1) && p.ckpt != nullptr && K > 0;
    int64_t next_ck = want_ckpt ? ((t_begin + K - 1) / K) * K : INT64_MAX;

    // This lane's share of the 16-byte chunks of a full tile, as element offsets from
    // the tile's first row (x, delta and y tiles share one geometry; b and c another).
    int x_goff[C::X_PL], x_soff[C::X_PL], bc_off[C::BC_PL];
#pragma unroll
    for (int k = 0; k < C::X_PL; ++k) {
        const int i = lane + NT * k;
        const int r = i / C::X_CPR, cc = i % C::X_CPR;
        x_goff[k] = r * int(D) + cc * EPC;
        x_soff[k] = r * DT + cc * EPC;
    }
#pragma unroll
    for (int k = 0; k < C::BC_PL; ++k) bc_off[k] = (lane + NT * k) * EPC;   // rows of 16 are contiguous

    const int64_t ntiles = (t_end - t_begin + TT - 1) / TT;
    auto stage = [&](int64_t tile, int buf) {
        const int64_t t0 = t_begin + tile * TT;
        if (VEC && full_d && t0 + TT <= t_end) {
            const TIO* xsrc = xg + t0 * D + d0;
            const TIO* dsrc = dg + t0 * D + d0;
#pragma unroll
            for (int k = 0; k < C::X_PL; ++k) {
                if (C::X_CH % NT == 0 || lane + NT * k < C::X_CH) {
                    cp_async16(xs + buf * TT * DT + x_soff[k], xsrc + x_goff[k], 16);
                    cp_async16(ds + buf * TT * DT + x_soff[k], dsrc + x_goff[k], 16);
                }
            }
#pragma unroll
            for (int k = 0; k < C::BC_PL; ++k) {
                if (C::BC_CH % NT == 0 || lane + NT * k < C::BC_CH) {
                    cp_async16(bsr + buf * TT * kDS + bc_off[k], bg + t0 * kDS + bc_off[k], 16);
                    if (READ) cp_async16(csr + buf * TT * kDS + bc_off[k], cgl + t0 * kDS + bc_off[k], 16);
                }
            }
        } else {
            stage_tile<TIO, TT, DT, NT, VEC>(xs + buf * TT * DT, xg, D, t0, t_end, d0);
            stage_tile<TIO, TT, DT, NT, VEC>(ds + buf * TT * DT, dg, D, t0, t_end, d0);
            stage_tile<TIO, TT, kDS, NT, true>(bsr + buf * TT * kDS, bg, kDS, t0, t_end, 0);
            if (READ) stage_tile<TIO, TT, kDS, NT, true>(csr + buf * TT * kDS, cgl, kDS, t0, t_end, 0);
        }
    };
    auto store_state = [&](float* base) { store_lane_states<G, KD>(base, b, D, d0 + c0, s0, valid, h, perm); };

    // one cp.async group per tile (empty past the end), so every wait has the same depth
#pragma unroll
    for (int u = 0; u < C::NBUF - 1; ++u) {
        if (u < ntiles) stage(u, u);
        cp_async_commit();
    }
    for (int64_t tile = 0; tile < ntiles; ++tile) {
        const int buf = int(tile % C::NBUF);
        if (tile + C::NBUF - 1 < ntiles) stage(tile + C::NBUF - 1, int((tile + C::NBUF - 1) % C::NBUF));
        cp_async_commit();
        cp_async_wait<C::NBUF - 1>();
        __syncwarp();
        const float* bt;
        const float* ct;
        if constexpr (C::BF) {
            widen_bf16<NT>(bsf, reinterpret_cast<const __nv_bfloat16*>(bsr + buf * TT * kDS), TT * kDS);
            if (READ) widen_bf16<NT>(csf, reinterpret_cast<const __nv_bfloat16*>(csr + buf * TT * kDS), TT * kDS);
            __syncwarp();
            bt = bsf;
            ct = csf;
        } else {
            bt = reinterpret_cast<const float*>(bsr + buf * TT * kDS);
            ct = reinterpret_cast<const float*>(csr + buf * TT * kDS);
        }
        const TIO* xt = xs + buf * TT * DT;
        const TIO* dt = ds + buf * TT * DT;
        if constexpr (FUSE) {      // delta tile as float32, through softplus when asked
            if (p.softplus) {
                // rows past the end stay 0 (zero-filled raw rows would give softplus(0) = ln 2,
                // and padded steps must leave the state unchanged)
                const int rows = int(min(int64_t(TT), t_end - (t_begin + tile * TT)));
                static_assert(DT % 2 == 0, "softplus pairs stay within a tile row");
                for (int i = 2 * lane; i < TT * DT; i += 2 * NT) {      // two neighbouring channels
                    float raw[2];
                    load_vals<TIO, 2>(dt + i, raw);
                    const float2 sp = softplus2_f32(make_float2(raw[0], raw[1]));
                    *reinterpret_cast<float2*>(dsf + i) = (i / DT < rows) ? sp : make_float2(0.f, 0.f);
                }
            } else {
                for (int i = lane; i < TT * DT; i += NT) dsf[i] = to_f32(dt[i]);
            }
            __syncwarp();
        }
        const int64_t t0 = t_begin + tile * TT;
        if (CKT && t0 == next_ck) {               // checkpoints fall on tile starts
            if (next_ck < t_end) store_state(p.ckpt + (next_ck / K) * p.B * D * kDS);
            next_ck += K;
        }
        constexpr int RG = BY_STEP ? G : 1;     // steps per readout group

#pragma unroll
        for (int tt = 0; tt < TT; tt += RG) {
            float part[RG][KD];
#pragma unroll
            for (int j = 0; j < RG; ++j) {
                const int r = tt + j;
                if (!CKT && want_ckpt && t0 + r == next_ck) {
                    if (next_ck < t_end) store_state(p.ckpt + (next_ck / K) * p.B * D * kDS);
                    next_ck += K;
                }
                float dl[KD], xv[KD];
                if constexpr (PERM) {
                    if constexpr (FUSE) {
                        dl[0] = dsf[r * DT + c0 + gl];
                        dl[1] = dsf[r * DT + c0 + (gl ^ 1)];
                    } else {
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(dt + r * DT + c0);
                        dl[0] = __uint_as_float(__byte_perm(w, 0u, sel0));
                        dl[1] = __uint_as_float(__byte_perm(w, 0u, sel1));
                    }
                    const uint32_t wx = *reinterpret_cast<const uint32_t*>(xt + r * DT + c0);
                    xv[0] = __uint_as_float(__byte_perm(wx, 0u, sel0));
                    xv[1] = __uint_as_float(__byte_perm(wx, 0u, sel1));
                } else {
                    if constexpr (FUSE) load_vals<float, KD>(dsf + r * DT + c0, dl);
                    else load_vals<TIO, KD>(dt + r * DT + c0, dl);
                    load_vals<TIO, KD>(xt + r * DT + c0, xv);
                }
                float2 bb[KP], cc[KP];
#pragma unroll
                for (int q = 0; q < KP; q += 2) {
                    const float4 b4 = *reinterpret_cast<const float4*>(bt + r * kDS + s0 + 2 * q);
                    bb[q] = make_float2(b4.x, b4.y);
                    bb[q + 1] = make_float2(b4.z, b4.w);
                    if (READ) {
                        const float4 c4 = *reinterpret_cast<const float4*>(ct + r * kDS + s0 + 2 * q);
                        cc[q] = make_float2(c4.x, c4.y);
                        cc[q + 1] = make_float2(c4.z, c4.w);
                    }
                }
#pragma unroll
                for (int k = 0; k < KD; ++k) {
                    if (MODE == kPass1) dsum[k] += dl[k];
                    const float dx = dl[k] * xv[k];
                    // Packed (f32x2) multiplies for the exponent arguments and the input
                    // term, packed FMA for the state update, scalar readout: on sm_103a this
                    // mix issues the fewest instructions per element for the time it takes
                    // (measured; a packed readout, with one or two accumulators, was 2-4 %
                    // slower).
                    float acc0 = 0.f, acc1 = 0.f;
                    const float2 dl2 = make_float2(dl[k], dl[k]), dx2 = make_float2(dx, dx);
#pragma unroll
                    for (int q = 0; q < KP; ++q) {
                        const float2 e = __fmul2_rn(dl2, A2[k][q]);
                        const float2 a = make_float2(ex2(e.x), ex2(e.y));
                        const float2 u = __fmul2_rn(dx2, bb[q]);
                        h[k][q] = __ffma2_rn(a, h[k][q], u);
                        if (READ) {
                            acc0 = fmaf(h[k][q].x, cc[q].x, acc0);
                            acc1 = fmaf(h[k][q].y, cc[q].y, acc1);
                        }
                    }
                    part[j][k] = acc0 + acc1;
                }
            }
            if (READ) {
                if constexpr (BY_STEP && KD == 1) {
                    float v[G];
#pragma unroll
                    for (int j = 0; j < G; ++j) v[j] = part[j][0];
                    float yv = reduce_scatter_steps<G>(v, gl);
                    if constexpr (FUSE) yv = fmaf(Dkeep[0], to_f32(xt[(tt + gl) * DT + c0]), yv);   // skip
                    ys[(tt + gl) * DT + c0] = from_f32<TIO>(yv);
                } else if constexpr (BY_STEP) {
                    // 4 steps x 2 channels over the 4 lanes: lane gl takes step tt + gl of both
                    float v[8];
#pragma unroll
                    for (int j = 0; j < G; ++j) { v[2 * j] = part[j][0]; v[2 * j + 1] = part[j][1]; }
                    const float2 r2 = reduce_scatter8_over4(v, gl);
                    float out[2] = {r2.x, r2.y};
                    if constexpr (FUSE) {                                                  // skip
#pragma unroll
                        for (int k = 0; k < 2; ++k)
                            out[k] = fmaf(Dkeep[k], to_f32(xt[(tt + gl) * DT + c0 + k]), out[k]);
                    }
                    store_vals<TIO, 2>(ys + (tt + gl) * DT + c0, out);
                } else {
                    // two lanes per channel group: lane gl keeps channels [gl*KD/2, (gl+1)*KD/2)
                    constexpr int H = KD / 2;
                    float out[H];
#pragma unroll
                    for (int i = 0; i < H; ++i) {
                        // (with PERM, slot 0 is already this lane's own channel)
                        const float send = PERM ? part[0][1] : (gl ? part[0][i] : part[0][H + i]);
                        const float keep = PERM ? part[0][0] : (gl ? part[0][H + i] : part[0][i]);
                        out[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                        if constexpr (FUSE)                                                // skip
                            out[i] = fmaf(Dkeep[i], to_f32(xt[tt * DT + c0 + gl * H + i]), out[i]);
                    }
                    store_vals<TIO, H>(ys + tt * DT + c0 + gl * H, out);
                }
            }
        }
        __syncwarp();
        if (READ) {
            // y tile -> global, 16-byte chunks
            const int64_t rows = min(int64_t(TT), t_end - t0);
            if (VEC && full_d && rows == TT) {
                TIO* ydst = yg + t0 * D + d0;
#pragma unroll
                for (int k = 0; k < C::X_PL; ++k)
                    if (C::X_CH % NT == 0 || lane + NT * k < C::X_CH)
                        *reinterpret_cast<uint4*>(ydst + x_goff[k]) = *reinterpret_cast<const uint4*>(ys + x_soff[k]);
            } else {
                for (int i = lane; i < TT * DT; i += NT) {
                    const int r = i / DT, cc = i % DT;
                    if (r < rows && d0 + cc < D) yg[(t0 + r) * D + d0 + cc] = ys[i];
                }
            }
            __syncwarp();
        }
    }

}

// Lane layout, A * log2(e) and the start state of the lane's chains (channels d0 + c0 + k).
// Channel slot k of the lane is channel d0 + c0 + (k ^ perm).
template <typename TIO, int G, int KD>
__device__ __forceinline__ void fwd_lane_setup(const FwdLaunch& p, int64_t b, int64_t d0, bool with_h0,
                                               bool (&valid)[KD], float2 (&A2)[KD][FwdCfg<TIO, G, KD>::KP],
                                               float2 (&h)[KD][FwdCfg<TIO, G, KD>::KP], int perm = 0) {
    constexpr int KP = FwdCfg<TIO, G, KD>::KP, KS = FwdCfg<TIO, G, KD>::KS;
    const int lane = threadIdx.x;
    const int c0 = (lane / G) * KD, s0 = (lane % G) * KS;
#pragma unroll
    for (int k = 0; k < KD; ++k) {
        const int64_t d = d0 + c0 + (k ^ perm);
        valid[k] = d < p.D;
#pragma unroll
        for (int q = 0; q < KP; ++q) {
            A2[k][q] = valid[k] ? make_float2(p.A[d * kDS + s0 + 2 * q] * kLog2e, p.A[d * kDS + s0 + 2 * q + 1] * kLog2e)
                                : make_float2(0.f, 0.f);
            h[k][q] = make_float2(0.f, 0.f);
        }
        if (with_h0 && valid[k] && p.h0 != nullptr) {
            const float* src = p.h0 + (b * p.D + d) * kDS + s0;
#pragma unroll
            for (int q = 0; q < KP; ++q) h[k][q] = make_float2(src[2 * q], src[2 * q + 1]);
        }
    }
}

template <typename TIO, int G, int KD, bool VEC, int MODE, bool CKT, bool FUSE>
__global__ void __launch_bounds__(32, FwdCfg<TIO, G, KD>::MINB) fwd_kernel(const FwdLaunch p) {
    using C = FwdCfg<TIO, G, KD>;
    constexpr int KP = C::KP, KS = C::KS;
    const int lane = threadIdx.x;
    const int gl = lane % G, c0 = (lane / G) * KD, s0 = gl * KS;
    const int64_t D = p.D;
    const int64_t b = blockIdx.z;
    const int64_t d0 = int64_t(blockIdx.x) * C::DT;
    const int64_t nprev = p.nchunk - 1;      // chunks with a stored carry
    const int64_t chunk = (MODE == kPass1 || MODE == kPass2) ? int64_t(blockIdx.y) : 0;
    const int64_t t_begin = chunk * p.Lc;
    const int64_t t_end = (MODE == kPass1 || MODE == kPass2) ? min(p.T, t_begin + p.Lc) : p.T;

    constexpr bool PERM = (G == 2 && C::BF);        // the channel order fwd_sweep uses
    const int perm = PERM ? gl : 0;
    bool valid[KD];
    float2 A2[KD][KP], h[KD][KP];
    fwd_lane_setup<TIO, G, KD>(p, b, d0, MODE != kPass1, valid, A2, h, perm);
    if constexpr (MODE == kPass2) {
        // (channel slot k of the lane is channel d0 + c0 + (k ^ perm); a carry row holds a chain's
        // 16 states, of which the lane's KS start at s0)
        if (p.carry_scanned) {
            // the middle pass left this chunk's start state in the carry of the chunk before it
            if (chunk > 0) {
#pragma unroll
                for (int k = 0; k < KD; ++k) {
                    if (!valid[k]) continue;
                    const int64_t row = (b * nprev + chunk - 1) * D + d0 + c0 + (k ^ perm);
                    const float4* src = reinterpret_cast<const float4*>(p.ws_S + row * kDS + s0);
#pragma unroll
                    for (int q = 0; q < KP; q += 2) {
                        const float4 v = src[q / 2];
                        h[k][q] = make_float2(v.x, v.y);
                        h[k][q + 1] = make_float2(v.z, v.w);
                    }
                }
            }
        }
        // otherwise: start state of this chunk: fold the carries of the chunks before it, in
        // order; the loads of NB chunks are issued together (one round trip to L2 per NB chunks)
        constexpr int NB = KP == 2 ? 4 : 2;
        for (int64_t j0 = 0; j0 < (p.carry_scanned ? 0 : chunk); j0 += NB) {
            float sd[NB][KD];
            float4 Sv[NB][KD][KP / 2];
#pragma unroll
            for (int u = 0; u < NB; ++u)
#pragma unroll
                for (int k = 0; k < KD; ++k) {
                    sd[u][k] = 0.f;
#pragma unroll
                    for (int q = 0; q < KP / 2; ++q) Sv[u][k][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (j0 + u < chunk && valid[k]) {
                        const int64_t row = (b * nprev + j0 + u) * D + d0 + c0 + (k ^ perm);
                        sd[u][k] = p.ws_Sd[row];
#pragma unroll
                        for (int q = 0; q < KP / 2; ++q)
                            Sv[u][k][q] = reinterpret_cast<const float4*>(p.ws_S + row * kDS + s0)[q];
                    }
                }
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                if (j0 + u >= chunk) break;
#pragma unroll
                for (int k = 0; k < KD; ++k) {
#pragma unroll
                    for (int q = 0; q < KP; ++q) {
                        const float4 v = Sv[u][k][q / 2];
                        const float2 S2 = (q & 1) ? make_float2(v.z, v.w) : make_float2(v.x, v.y);
                        const float2 P = make_float2(ex2(A2[k][q].x * sd[u][k]), ex2(A2[k][q].y * sd[u][k]));
                        h[k][q] = __ffma2_rn(P, h[k][q], S2);
                    }
                }
            }
        }
    }
    float dsum[KD];
#pragma unroll
    for (int k = 0; k < KD; ++k) dsum[k] = 0.f;

    fwd_sweep<TIO, G, KD, VEC, MODE, CKT, FUSE>(p, b, d0, t_begin, t_end, A2, valid, h, dsum);

    if (MODE == kPass1) {
#pragma unroll
        for (int k = 0; k < KD; ++k) {
            if (!valid[k]) continue;
            const int64_t row = (b * nprev + chunk) * D + d0 + c0 + (k ^ perm);
            float4* S = reinterpret_cast<float4*>(p.ws_S + row * kDS + s0);
#pragma unroll
            for (int q = 0; q < KP; q += 2) S[q / 2] = make_float4(h[k][q].x, h[k][q].y, h[k][q + 1].x, h[k][q + 1].y);
            if (gl == 0) p.ws_Sd[row] = dsum[k];
        }
        return;
    }
    const bool last = (MODE != kPass2) || (chunk == p.nchunk - 1);
    if (last && p.hT != nullptr) store_lane_states<G, KD>(p.hT, b, D, d0 + c0, s0, valid, h, perm);
}

__device__ __forceinline__ int ld_acquire_gpu(const int* ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* ptr, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// The chunked scan in one launch, with decoupled look-back (the single-pass prefix scan of
// Merrill and Garland, 2016, applied to the affine chunk maps h -> exp(A sum(delta)) h + S):
//  1. a CTA of chain block (b, d-block) takes the next ticket of that block's counter as its
//     chunk, so every CTA it will wait for took an earlier ticket and is already running;
//  2. chunks before the last sweep once without readout: chunk 0 from h0 (its end state is
//     the inclusive state, published with flag 2), the others from 0 (their map: end state S
//     and delta sum, published with flag 1);
//  3. a chunk k > 0 walks back over k-1, k-2, ...: it folds in each map published there until
//     it reaches an inclusive state, which gives its start state; it then publishes its own
//     inclusive state (flag 2);
//  4. every chunk rescans from its start state with readout, as pass 2 of the two-launch
//     schedule does.
// Each wait polls a flag at most lb_polls times per CTA; a wait that runs out adds 1 to
// lb_status and the chunk carries on with the part of the prefix it has, so the launch always
// finishes (with wrong values for that chunk) and the host can report the failure.
template <typename TIO, int KD, bool VEC, bool CKT, bool FUSE>
__global__ void __launch_bounds__(32, FwdCfg<TIO, 4, KD>::MINB) fwd_lookback_kernel(const FwdLaunch p) {
    constexpr int G = 4;
    using C = FwdCfg<TIO, G, KD>;
    constexpr int KP = C::KP, KS = C::KS;
    const int lane = threadIdx.x;
    const int c0 = (lane / G) * KD, s0 = (lane % G) * KS;
    const int64_t D = p.D, B = p.B, nch = p.nchunk;
    const int64_t nblk = (D + C::DT - 1) / C::DT;

    // the chain block is the CTA's; its chunk is a ticket from the block's own counter
    const int64_t b = blockIdx.y, dblk = blockIdx.x, d0 = dblk * C::DT;
    int tk = 0;
    if (lane == 0) tk = atomicAdd(p.lb_ticket + b * nblk + dblk, 1);
    const int64_t chunk = __shfl_sync(0xffffffffu, tk, 0);
    const int64_t rem = dblk;
    const int64_t t_begin = chunk * p.Lc, t_end = min(p.T, t_begin + p.Lc);
    const bool last = chunk == nch - 1;
    int* my_flag = p.lb_flags + (chunk * B + b) * nblk + rem % nblk;
    auto row = [&](int64_t j, int k) { return (b * nch + j) * D + d0 + c0 + k; };

    bool valid[KD];
    float2 A2[KD][KP], h[KD][KP], hin[KD][KP];
    fwd_lane_setup<TIO, G, KD>(p, b, d0, chunk == 0, valid, A2, hin);   // hin = h0 for chunk 0, else 0
    float dsum[KD];
#pragma unroll
    for (int k = 0; k < KD; ++k) {
        dsum[k] = 0.f;
#pragma unroll
        for (int q = 0; q < KP; ++q) h[k][q] = hin[k][q];
    }

    // 2. the chunk's map (or, for chunk 0, its inclusive state)
    if (!last) {
        fwd_sweep<TIO, G, KD, VEC, kPass1, CKT, FUSE>(p, b, d0, t_begin, t_end, A2, valid, h, dsum);
        float* dst = chunk == 0 ? p.lb_X : p.lb_S;
#pragma unroll
        for (int k = 0; k < KD; ++k) {
            if (!valid[k]) continue;
            float4* o = reinterpret_cast<float4*>(dst + row(chunk, k) * kDS + s0);
#pragma unroll
            for (int q = 0; q < KP; q += 2) o[q / 2] = make_float4(h[k][q].x, h[k][q].y, h[k][q + 1].x, h[k][q + 1].y);
            if (lane % G == 0) p.lb_Sd[row(chunk, k)] = dsum[k];
        }
        __threadfence();
        __syncwarp();
        if (lane == 0 && !(p.lb_test_drop && chunk == 0)) st_release_gpu(my_flag, chunk == 0 ? 2 : 1);
    }

    // 3. look back for the start state
    if (chunk > 0) {
        float sdacc[KD];
        float2 sacc[KD][KP];
#pragma unroll
        for (int k = 0; k < KD; ++k) {
            sdacc[k] = 0.f;
#pragma unroll
            for (int q = 0; q < KP; ++q) sacc[k][q] = make_float2(0.f, 0.f);
        }
        // Windowed look-back: lane i probes the flag of predecessor j - i, so one round trip
        // sees 32 predecessors; the maps up to the nearest unpublished one or the nearest
        // inclusive state are then folded, their loads issued NB predecessors at a time.
        constexpr int NB = 4;
        int64_t polls = 0;
        bool timed_out = false;
        int64_t j = chunk - 1;                   // nearest predecessor not yet folded
        while (true) {
            const int64_t jl = j - lane;
            int f = 0;
            if (jl >= 0) f = ld_acquire_gpu(p.lb_flags + (jl * B + b) * nblk + rem % nblk);
            const unsigned zero = __ballot_sync(0xffffffffu, jl >= 0 && f == 0);
            const unsigned incl = __ballot_sync(0xffffffffu, jl >= 0 && f == 2);
            // (chunk 0 publishes flag 2 only, so a window reaching it always stops there)
            const unsigned stop = zero | incl;
            const int first = stop ? __ffs(int(stop)) - 1 : 32;
            const bool done = first < 32 && ((incl >> first) & 1u);
            const int n = first + (done ? 1 : 0);          // predecessors to fold now (warp-uniform)
            // lane i's acquire load saw predecessor j - i published; the barrier orders that
            // acquire before every lane's loads of the predecessor's payload below
            __syncwarp();
            for (int i0 = 0; i0 < n; i0 += NB) {
                float2 v[NB][KD][KP];
                float sdv[NB][KD];
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    const int i = i0 + u;
                    const int fi = __shfl_sync(0xffffffffu, f, i & 31);
#pragma unroll
                    for (int k = 0; k < KD; ++k) {
                        sdv[u][k] = 0.f;
#pragma unroll
                        for (int q = 0; q < KP; ++q) v[u][k][q] = make_float2(0.f, 0.f);
                        if (i >= n || !valid[k]) continue;
                        const float* src = (fi == 2 ? p.lb_X : p.lb_S) + row(j - i, k) * kDS + s0;
#pragma unroll
                        for (int q = 0; q < KP; ++q) v[u][k][q] = __ldcg(reinterpret_cast<const float2*>(src) + q);
                        if (fi == 1) sdv[u][k] = __ldcg(p.lb_Sd + row(j - i, k));
                    }
                }
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    if (i0 + u >= n) break;
#pragma unroll
                    for (int k = 0; k < KD; ++k) {
#pragma unroll
                        for (int q = 0; q < KP; ++q) {
                            // fold predecessor j - i in front of the later ones
                            const float2 P = make_float2(ex2(A2[k][q].x * sdacc[k]), ex2(A2[k][q].y * sdacc[k]));
                            sacc[k][q] = __ffma2_rn(P, v[u][k][q], sacc[k][q]);
                        }
                        sdacc[k] += sdv[u][k];
                    }
                }
            }
            if (done) break;
            j -= n;
            if (n == 0) {                                  // the nearest predecessor has not published yet
                if (polls >= p.lb_polls) {
                    timed_out = true;
                    break;
                }
                ++polls;
                __nanosleep(128);
            }
        }
        if (timed_out && lane == 0) atomicAdd(p.lb_status, 1u);
#pragma unroll
        for (int k = 0; k < KD; ++k)
#pragma unroll
            for (int q = 0; q < KP; ++q) hin[k][q] = sacc[k][q];
        if (!last) {
            // inclusive state of this chunk: exp(A dsum) hin + S (h holds S)
#pragma unroll
            for (int k = 0; k < KD; ++k) {
                if (!valid[k]) continue;
                float4* o = reinterpret_cast<float4*>(p.lb_X + row(chunk, k) * kDS + s0);
#pragma unroll
                for (int q = 0; q < KP; q += 2) {
                    float2 x2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float2 P = make_float2(ex2(A2[k][q + u].x * dsum[k]), ex2(A2[k][q + u].y * dsum[k]));
                        x2[u] = __ffma2_rn(P, hin[k][q + u], h[k][q + u]);
                    }
                    o[q / 2] = make_float4(x2[0].x, x2[0].y, x2[1].x, x2[1].y);
                }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_gpu(my_flag, 2);
        }
    }

    // 4. rescan with readout from the start state
    __syncwarp();
#pragma unroll
    for (int k = 0; k < KD; ++k)
#pragma unroll
        for (int q = 0; q < KP; ++q) h[k][q] = hin[k][q];
    fwd_sweep<TIO, G, KD, VEC, kPass2, CKT, FUSE>(p, b, d0, t_begin, t_end, A2, valid, h, dsum);
    if (last && p.hT != nullptr) store_lane_states<G, KD>(p.hT, b, D, d0 + c0, s0, valid, h);
}

template <typename TIO, int KD, bool VEC, bool CKT, bool FUSE>
cudaError_t launch_fwd_lookback_t(const FwdLaunch& L, cudaStream_t stream) {
    using C = FwdCfg<TIO, 4, KD>;
    constexpr size_t smem = FUSE ? C::SMEM_FUSE : C::SMEM;
    auto kern = fwd_lookback_kernel<TIO, KD, VEC, CKT, FUSE>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(unsigned((L.D + C::DT - 1) / C::DT), unsigned(L.B), unsigned(L.nchunk));
    kern<<<grid, C::NT, smem, stream>>>(L);
    return cudaGetLastError();
}

template <typename TIO, int G, int KD, bool VEC, int MODE, bool CKT, bool FUSE>
cudaError_t launch_fwd_t(const FwdLaunch& L, cudaStream_t stream) {
    using C = FwdCfg<TIO, G, KD>;
    constexpr size_t smem = FUSE ? C::SMEM_FUSE : C::SMEM;
    auto kern = fwd_kernel<TIO, G, KD, VEC, MODE, CKT, FUSE>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
    }
    unsigned gy = 1;
    if (MODE == kPass1) gy = unsigned(L.nchunk - 1);
    if (MODE == kPass2) gy = unsigned(L.nchunk);
    const dim3 grid(unsigned((L.D + C::DT - 1) / C::DT), gy, unsigned(L.B));
    kern<<<grid, C::NT, smem, stream>>>(L);
    return cudaGetLastError();
}

// All instantiations for one I/O type and fusion choice. Checkpoints are checked once per
// tile when every checkpoint step is a tile start (K and the chunk length multiples of 16).
template <typename TIO, bool FUSE>
cudaError_t launch_fwd_fuse(const FwdLaunch& L, int mode, cudaStream_t stream) {
    constexpr int TT = FwdCfg<TIO, 4, 1>::TT;
    const bool ckt = L.K == 0 || (L.K % TT == 0 && (mode == kSingle || mode == kCkptOnly || L.Lc % TT == 0));
    // (kLookback sweeps chunks of L.Lc steps like kPass2)
#define SSM_FWD_CK(G_, KD_, MODE_, VEC_)                                                   \
    return ckt ? launch_fwd_t<TIO, G_, KD_, VEC_, MODE_, true, FUSE>(L, stream)           \
               : launch_fwd_t<TIO, G_, KD_, VEC_, MODE_, false, FUSE>(L, stream)
#define SSM_FWD_VEC(G_, KD_, MODE_)                                                       \
    if (L.vec) { SSM_FWD_CK(G_, KD_, MODE_, true); } else { SSM_FWD_CK(G_, KD_, MODE_, false); }
    switch (mode) {
        case kSingle:
            if (L.G == 2) { SSM_FWD_VEC(2, 2, kSingle); }
            if (L.kd == 2) { SSM_FWD_VEC(4, 2, kSingle); }
            SSM_FWD_VEC(4, 1, kSingle);
        case kPass1:
            if (L.G == 2) {
                if (L.vec) return launch_fwd_t<TIO, 2, 2, true, kPass1, true, FUSE>(L, stream);
                return launch_fwd_t<TIO, 2, 2, false, kPass1, true, FUSE>(L, stream);
            }
            if (L.kd == 2) {
                if (L.vec) return launch_fwd_t<TIO, 4, 2, true, kPass1, true, FUSE>(L, stream);
                return launch_fwd_t<TIO, 4, 2, false, kPass1, true, FUSE>(L, stream);
            }
            if (L.vec) return launch_fwd_t<TIO, 4, 1, true, kPass1, true, FUSE>(L, stream);
            return launch_fwd_t<TIO, 4, 1, false, kPass1, true, FUSE>(L, stream);
        case kPass2:
            if (L.G == 2) { SSM_FWD_VEC(2, 2, kPass2); }
            if (L.kd == 2) { SSM_FWD_VEC(4, 2, kPass2); }
            SSM_FWD_VEC(4, 1, kPass2);
        case kCkptOnly: SSM_FWD_VEC(4, 1, kCkptOnly);
        case kLookback:
#define SSM_FWD_LB(KD_, VEC_) \
    return ckt ? launch_fwd_lookback_t<TIO, KD_, VEC_, true, FUSE>(L, stream) \
               : launch_fwd_lookback_t<TIO, KD_, VEC_, false, FUSE>(L, stream)
            if (L.kd == 2) {
                if (L.vec) { SSM_FWD_LB(2, true); } else { SSM_FWD_LB(2, false); }
            }
            if (L.vec) { SSM_FWD_LB(1, true); } else { SSM_FWD_LB(1, false); }
#undef SSM_FWD_LB
        default: return cudaErrorInvalidValue;
    }
#undef SSM_FWD_VEC
#undef SSM_FWD_CK
}

template <typename TIO>
cudaError_t launch_fwd_io(const FwdLaunch& L, int mode, cudaStream_t stream) {
    // the skip is applied where y is read out: the one-pass scan, pass 2, the look-back scan
    const bool fuse = L.softplus || (L.Dskip != nullptr && (mode == kSingle || mode == kPass2 || mode == kLookback));
    return fuse ? launch_fwd_fuse<TIO, true>(L, mode, stream) : launch_fwd_fuse<TIO, false>(L, mode, stream);
}

}  // namespace ssm
