// Forward scan kernels: one pass over T, and the two passes of the chunked scan.
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
// Thread layout: a CTA of NT threads covers DT = NT / G channels d of one
// batch b; each channel's DS = 16 states are split over G neighbouring lanes
// (KS = 16 / G states per lane, kept in registers for the whole sweep). Time
// is walked in tiles of TT steps; x, delta, b, c tiles are double-buffered in
// shared memory with cp.async (zero-filled past the end, which leaves the
// state unchanged: delta = 0 gives decay 1 and no input). With G > 1 the
// readout <h_t, c_t> is finished by a reduce-scatter over G steps, and y is
// written back a tile at a time with 16-byte stores.
#pragma once

#include <type_traits>

#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {

enum FwdMode { kSingle = 0, kPass1 = 1, kPass2 = 2, kCkptOnly = 3 };

template <typename TIO, int G>
struct FwdCfg {
    static constexpr int NT = 128;
    static constexpr int KS = kDS / G;
    static constexpr int DT = NT / G;
    static constexpr int TT = 32;
    static constexpr bool BF = std::is_same<TIO, __nv_bfloat16>::value;
    static constexpr size_t X_BYTES = size_t(2) * TT * DT * sizeof(TIO);     // one tensor, 2 buffers
    static constexpr size_t BC_RAW = size_t(2) * TT * kDS * sizeof(TIO);    // one tensor, 2 buffers
    static constexpr size_t BC_F32 = BF ? size_t(TT) * kDS * 4 : 0;          // widened copy (bf16)
    static constexpr size_t Y_BYTES = size_t(TT) * DT * 4;
    static constexpr size_t SMEM = 2 * X_BYTES + 2 * BC_RAW + 2 * BC_F32 + Y_BYTES;
};

template <typename TIO, int G, bool VEC, int MODE>
__global__ void __launch_bounds__(128) fwd_kernel(const FwdLaunch p) {
    using C = FwdCfg<TIO, G>;
    constexpr int NT = C::NT, KS = C::KS, DT = C::DT, TT = C::TT;
    constexpr bool READ = (MODE == kSingle || MODE == kPass2);

    extern __shared__ __align__(16) unsigned char smem[];
    TIO* xs = reinterpret_cast<TIO*>(smem);
    TIO* ds = reinterpret_cast<TIO*>(smem + C::X_BYTES);
    TIO* bsr = reinterpret_cast<TIO*>(smem + 2 * C::X_BYTES);
    TIO* csr = reinterpret_cast<TIO*>(smem + 2 * C::X_BYTES + C::BC_RAW);
    float* bsf = reinterpret_cast<float*>(smem + 2 * C::X_BYTES + 2 * C::BC_RAW);
    float* csf = bsf + (C::BF ? TT * kDS : 0);
    float* ys = reinterpret_cast<float*>(smem + 2 * C::X_BYTES + 2 * C::BC_RAW + 2 * C::BC_F32);

    const int tid = threadIdx.x;
    const int cg = tid / G;          // channel within the CTA
    const int gl = tid % G;          // lane within the channel's group
    const int s0 = gl * KS;
    const int64_t T = p.T, D = p.D;
    const int64_t b = blockIdx.z;
    const int64_t d0 = int64_t(blockIdx.x) * DT;
    const int64_t d = d0 + cg;
    const bool valid = d < D;
    const int64_t chunk = (MODE == kPass1 || MODE == kPass2) ? int64_t(blockIdx.y) : 0;
    const int64_t t_begin = chunk * p.Lc;
    const int64_t t_end = (MODE == kPass1 || MODE == kPass2) ? min(T, t_begin + p.Lc) : T;
    const int64_t nprev = p.nchunk - 1;   // chunks with a stored carry

    const TIO* xg = static_cast<const TIO*>(p.x) + b * T * D;
    const TIO* dg = static_cast<const TIO*>(p.delta) + b * T * D;
    const TIO* bg = static_cast<const TIO*>(p.b) + b * T * kDS;
    const TIO* cgl = static_cast<const TIO*>(p.c) + b * T * kDS;

    float A2[KS], h[KS];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        A2[s] = valid ? p.A[d * kDS + s0 + s] * kLog2e : 0.f;
        h[s] = 0.f;
    }
    if (MODE != kPass1 && valid && p.h0 != nullptr) {
#pragma unroll
        for (int s = 0; s < KS; ++s) h[s] = p.h0[(b * D + d) * kDS + s0 + s];
    }
    if (MODE == kPass2 && valid) {
        // start state of this chunk: fold the carries of the chunks before it
        for (int64_t j = 0; j < chunk; ++j) {
            const int64_t row = (b * nprev + j) * D + d;
            const float sd = p.ws_Sd[row];
#pragma unroll
            for (int s = 0; s < KS; ++s) h[s] = fmaf(ex2(A2[s] * sd), h[s], p.ws_S[row * kDS + s0 + s]);
        }
    }
    float dsum = 0.f;
    const int64_t K = p.K;
    const bool want_ckpt = (MODE != kPass1) && p.ckpt != nullptr && K > 0;
    int64_t next_ck = want_ckpt ? ((t_begin + K - 1) / K) * K : INT64_MAX;

    const int64_t ntiles = (t_end - t_begin + TT - 1) / TT;
    auto stage = [&](int64_t tile, int buf) {
        const int64_t t0 = t_begin + tile * TT;
        stage_tile<TIO, TT, DT, NT, VEC>(xs + buf * TT * DT, xg, D, t0, t_end, d0);
        stage_tile<TIO, TT, DT, NT, VEC>(ds + buf * TT * DT, dg, D, t0, t_end, d0);
        stage_tile<TIO, TT, kDS, NT, true>(bsr + buf * TT * kDS, bg, kDS, t0, t_end, 0);
        if (READ) stage_tile<TIO, TT, kDS, NT, true>(csr + buf * TT * kDS, cgl, kDS, t0, t_end, 0);
    };

    if (ntiles > 0) {
        stage(0, 0);
        cp_async_commit();
    }
    for (int64_t tile = 0; tile < ntiles; ++tile) {
        const int buf = int(tile & 1);
        if (tile + 1 < ntiles) {
            stage(tile + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float* bt;
        const float* ct;
        if constexpr (C::BF) {
            widen_bf16<NT>(bsf, reinterpret_cast<const __nv_bfloat16*>(bsr + buf * TT * kDS), TT * kDS);
            if (READ) widen_bf16<NT>(csf, reinterpret_cast<const __nv_bfloat16*>(csr + buf * TT * kDS), TT * kDS);
            __syncthreads();
            bt = bsf;
            ct = csf;
        } else {
            bt = reinterpret_cast<const float*>(bsr + buf * TT * kDS);
            ct = reinterpret_cast<const float*>(csr + buf * TT * kDS);
        }
        const TIO* xt = xs + buf * TT * DT;
        const TIO* dt = ds + buf * TT * DT;
        const int64_t t0 = t_begin + tile * TT;

#pragma unroll
        for (int tt = 0; tt < TT; tt += G) {
            float part[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int r = tt + j;
                if (want_ckpt && t0 + r == next_ck) {
                    if (valid && next_ck < t_end) {
                        float* dst = p.ckpt + ((next_ck / K * p.B + b) * D + d) * kDS + s0;
#pragma unroll
                        for (int s = 0; s < KS; ++s) dst[s] = h[s];
                    }
                    next_ck += K;
                }
                const float dl = to_f32(dt[r * DT + cg]);
                const float xv = to_f32(xt[r * DT + cg]);
                const float dx = dl * xv;
                if (MODE == kPass1) dsum += dl;
                float acc = 0.f;
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    const float a = ex2(dl * A2[s]);
                    h[s] = fmaf(a, h[s], dx * bt[r * kDS + s0 + s]);
                    if (READ) acc = fmaf(h[s], ct[r * kDS + s0 + s], acc);
                }
                part[j] = acc;
            }
            if (READ) ys[(tt + gl) * DT + cg] = reduce_scatter_steps<G>(part, gl);
        }
        __syncthreads();
        if (READ) {
            // y tile -> global, rows [t0, t_end), columns [d0, D)
            TIO* yg = static_cast<TIO*>(p.y) + b * T * D;
            const int64_t rows = min(int64_t(TT), t_end - t0);
            if constexpr (VEC) {
                constexpr int EPC = 16 / sizeof(TIO);
                constexpr int CPR = DT / EPC;
                for (int i = tid; i < TT * CPR; i += NT) {
                    const int r = i / CPR, cc = i % CPR;
                    const int64_t col = d0 + int64_t(cc) * EPC;
                    if (r < rows && col < D) {
                        const float* src = ys + r * DT + cc * EPC;
                        uint4 v;
                        if constexpr (C::BF) {
                            __nv_bfloat162 q[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) q[k] = __floats2bfloat162_rn(src[2 * k], src[2 * k + 1]);
                            v = *reinterpret_cast<const uint4*>(q);
                        } else {
                            v = *reinterpret_cast<const uint4*>(src);
                        }
                        *reinterpret_cast<uint4*>(yg + (t0 + r) * D + col) = v;
                    }
                }
            } else {
                for (int i = tid; i < TT * DT; i += NT) {
                    const int r = i / DT, cc = i % DT;
                    if (r < rows && d0 + cc < D) yg[(t0 + r) * D + d0 + cc] = from_f32<TIO>(ys[i]);
                }
            }
        }
    }

    if (!valid) return;
    if (MODE == kPass1) {
        const int64_t row = (b * nprev + chunk) * D + d;
#pragma unroll
        for (int s = 0; s < KS; ++s) p.ws_S[row * kDS + s0 + s] = h[s];
        if (gl == 0) p.ws_Sd[row] = dsum;
        return;
    }
    const bool last = (MODE != kPass2) || (chunk == p.nchunk - 1);
    if (last && p.hT != nullptr) {
#pragma unroll
        for (int s = 0; s < KS; ++s) p.hT[(b * D + d) * kDS + s0 + s] = h[s];
    }
}

template <typename TIO, int G, bool VEC, int MODE>
cudaError_t launch_fwd_t(const FwdLaunch& L, cudaStream_t stream) {
    using C = FwdCfg<TIO, G>;
    auto kern = fwd_kernel<TIO, G, VEC, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
    if (e != cudaSuccess) return e;
    unsigned gy = 1;
    if (MODE == kPass1) gy = unsigned(L.nchunk - 1);
    if (MODE == kPass2) gy = unsigned(L.nchunk);
    const dim3 grid(unsigned((L.D + C::DT - 1) / C::DT), gy, unsigned(L.B));
    kern<<<grid, C::NT, C::SMEM, stream>>>(L);
    return cudaGetLastError();
}

// All instantiations for one I/O type.
template <typename TIO>
cudaError_t launch_fwd_io(const FwdLaunch& L, int mode, cudaStream_t stream) {
#define SSM_FWD_VEC(G_, MODE_)                                               \
    return L.vec ? launch_fwd_t<TIO, G_, true, MODE_>(L, stream)             \
                 : launch_fwd_t<TIO, G_, false, MODE_>(L, stream)
    switch (mode) {
        case kSingle:
            if (L.G == 1) { SSM_FWD_VEC(1, kSingle); }
            if (L.G == 2) { SSM_FWD_VEC(2, kSingle); }
            SSM_FWD_VEC(4, kSingle);
        case kPass1: SSM_FWD_VEC(4, kPass1);
        case kPass2: SSM_FWD_VEC(4, kPass2);
        case kCkptOnly: SSM_FWD_VEC(4, kCkptOnly);
        default: return cudaErrorInvalidValue;
    }
#undef SSM_FWD_VEC
}

}  // namespace ssm
