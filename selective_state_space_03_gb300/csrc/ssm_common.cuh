// Device helpers shared by the scan kernels (sm_103a).
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ssm_internal.h"

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;   // exp(v) = 2^(v * log2(e))

// 2^v on the special-function unit (MUFU), denormal results flushed to zero.
// Its relative error is a few units in the last place of float32, far inside
// the scan's tolerance; decays are in (0, 1] so flushing only affects values
// below 2^-126.
__device__ __forceinline__ float ex2(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// log2(v) on the MUFU; absolute error about 2^-22 for v in [1, 2].
__device__ __forceinline__ float lg2(float v) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

constexpr float kLn2 = 0.6931471805599453f;

// softplus(v) = log(1 + e^v) = max(v, 0) + log1p(e^-|v|), the activation the trace page's
// model applies to delta. log1p(e) comes from its Taylor series e - e^2/2 + ... + e^5/5 when
// e < 1/32 (where 1 + e would round most of e away; truncation below 1e-8 relative), else
// from log2(1 + e) on the MUFU (relative error below 1e-5 there).
__device__ __forceinline__ float softplus_f32(float v) {
    const float e = ex2(-fabsf(v) * kLog2e);                 // in (0, 1]
    const float l = e < 0.03125f
        ? e * (1.f - e * (0.5f - e * (0.33333334f - e * (0.25f - e * 0.2f))))
        : lg2(1.f + e) * kLn2;
    return fmaxf(v, 0.f) + l;
}

// softplus of two values with packed f32x2 arithmetic (same formula and accuracy as
// softplus_f32): the exponent arguments, the series, 1 + e and the ln 2 scaling run as
// f32x2 operations, the two exponentials and logarithms on the MUFU.
__device__ __forceinline__ float2 softplus2_f32(float2 v) {
    const float2 m = __fmul2_rn(make_float2(fabsf(v.x), fabsf(v.y)), make_float2(-kLog2e, -kLog2e));
    const float2 e = make_float2(ex2(m.x), ex2(m.y));                       // in (0, 1]
    const float2 ne = make_float2(-e.x, -e.y);
    // e (1 - e (1/2 - e (1/3 - e (1/4 - e/5)))), nested from the inside
    float2 p = __ffma2_rn(ne, make_float2(0.2f, 0.2f), make_float2(0.25f, 0.25f));
    p = __ffma2_rn(ne, p, make_float2(0.33333334f, 0.33333334f));
    p = __ffma2_rn(ne, p, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(ne, p, make_float2(1.f, 1.f));
    const float2 series = __fmul2_rn(e, p);
    const float2 ope = __fadd2_rn(e, make_float2(1.f, 1.f));
    const float2 lg = __fmul2_rn(make_float2(lg2(ope.x), lg2(ope.y)), make_float2(kLn2, kLn2));
    return make_float2(fmaxf(v.x, 0.f) + (e.x < 0.03125f ? series.x : lg.x),
                       fmaxf(v.y, 0.f) + (e.y < 0.03125f ? series.y : lg.y));
}

// sigmoid(v), the derivative of softplus, from sp = softplus(v): sigmoid(v) = 1 - e^-sp.
// Small sp from the series sp - sp^2/2 + sp^3/6 - sp^4/24 (no cancellation).
__device__ __forceinline__ float sigmoid_from_softplus(float sp) {
    return sp < 0.03125f ? sp * (1.f - sp * (0.5f - sp * (0.16666667f - sp * 0.041666668f)))
                         : 1.f - ex2(-sp * kLog2e);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);   // round to nearest even
}

// ---------------------------------------------------------------- cp.async

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes == 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory"); }

// ---------------------------------------------------------------- tile staging
//
// Rows [t0, t0 + TT) x columns [d0, d0 + W) of one batch of a (B, T, W_total)
// tensor into dst[TT][W] (same element type). Rows at or past t_end and
// columns at or past ncols are zero-filled. VEC uses 16-byte cp.async and
// needs ncols * sizeof(E) % 16 == 0 and a 16-byte aligned base; otherwise the
// copy is element by element with plain loads.
template <typename E, int TT, int W, int NT, bool VEC>
__device__ __forceinline__ void stage_tile(E* dst, const E* src_b, int64_t ncols, int64_t t0,
                                           int64_t t_end, int64_t d0) {
    if constexpr (VEC) {
        constexpr int EPC = 16 / sizeof(E);
        static_assert(W % EPC == 0, "tile width must be a whole number of 16-byte chunks");
        constexpr int CPR = W / EPC;
        constexpr int NCH = TT * CPR;
        for (int i = threadIdx.x; i < NCH; i += NT) {
            const int r = i / CPR, cc = i % CPR;
            const int64_t t = t0 + r, col = d0 + int64_t(cc) * EPC;
            const bool ok = (t < t_end) && (col < ncols);
            const E* g = ok ? src_b + t * ncols + col : src_b;
            cp_async16(dst + r * W + cc * EPC, g, ok ? 16 : 0);
        }
    } else {
        for (int i = threadIdx.x; i < TT * W; i += NT) {
            const int r = i / W, cc = i % W;
            const int64_t t = t0 + r, col = d0 + cc;
            dst[i] = (t < t_end && col < ncols) ? src_b[t * ncols + col] : E(0.0f);
        }
    }
}

// Widen a bf16 tile in shared memory to float32 (n elements, n % 8 == 0).
template <int NT>
__device__ __forceinline__ void widen_bf16(float* dst, const __nv_bfloat16* src, int n) {
    for (int i = threadIdx.x * 8; i < n; i += NT * 8) {
        const uint4 raw = *reinterpret_cast<const uint4*>(src + i);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        float4 lo, hi;
        lo.x = __uint_as_float(w[0] << 16); lo.y = __uint_as_float(w[0] & 0xffff0000u);
        lo.z = __uint_as_float(w[1] << 16); lo.w = __uint_as_float(w[1] & 0xffff0000u);
        hi.x = __uint_as_float(w[2] << 16); hi.y = __uint_as_float(w[2] & 0xffff0000u);
        hi.z = __uint_as_float(w[3] << 16); hi.w = __uint_as_float(w[3] & 0xffff0000u);
        *reinterpret_cast<float4*>(dst + i) = lo;
        *reinterpret_cast<float4*>(dst + i + 4) = hi;
    }
}

// ---------------------------------------------------------------- small vector loads / stores
//
// N consecutive I/O elements (N * sizeof(T) bytes, naturally aligned) in one
// shared- or global-memory access, widened to / narrowed from float32.
template <typename T, int N>
__device__ __forceinline__ void load_vals(const T* p, float (&v)[N]) {
    if constexpr (std::is_same<T, float>::value) {
        if constexpr (N == 4) {
            const float4 q = *reinterpret_cast<const float4*>(p);
            v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else if constexpr (N == 2) {
            const float2 q = *reinterpret_cast<const float2*>(p);
            v[0] = q.x; v[1] = q.y;
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) v[i] = p[i];
        }
    } else {
        if constexpr (N == 4) {
            const uint2 q = *reinterpret_cast<const uint2*>(p);
            v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
            v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
        } else if constexpr (N == 2) {
            const uint32_t q = *reinterpret_cast<const uint32_t*>(p);
            v[0] = __uint_as_float(q << 16); v[1] = __uint_as_float(q & 0xffff0000u);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) v[i] = to_f32(p[i]);
        }
    }
}

template <typename T, int N>
__device__ __forceinline__ void store_vals(T* p, const float (&v)[N]) {
    if constexpr (std::is_same<T, float>::value) {
        if constexpr (N == 2) {
            *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) p[i] = v[i];
        }
    } else {
        if constexpr (N == 2) {
            *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) p[i] = __float2bfloat16_rn(v[i]);
        }
    }
}

// ---------------------------------------------------------------- lane reductions
//
// A chain's DS states are split over G neighbouring lanes. Each lane holds its
// partial sums for G consecutive steps (v[0..G-1]). After the call, lane gl of
// the group returns the full sum for step gl: a reduce-scatter that needs G-1
// shuffles per lane for G steps instead of log2(G) per step.
template <int G>
__device__ __forceinline__ float reduce_scatter_steps(const float (&v)[G], int gl) {
    if constexpr (G == 1) {
        return v[0];
    } else if constexpr (G == 2) {
        const bool hi = gl & 1;
        const float send = hi ? v[0] : v[1];
        const float keep = hi ? v[1] : v[0];
        return keep + __shfl_xor_sync(0xffffffffu, send, 1);
    } else {
        static_assert(G == 4, "G must be 1, 2 or 4");
        const bool hi2 = gl & 2;
        const float s0 = hi2 ? v[0] : v[2], s1 = hi2 ? v[1] : v[3];
        const float k0 = hi2 ? v[2] : v[0], k1 = hi2 ? v[3] : v[1];
        const float q0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 2);
        const float q1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 2);
        const bool hi1 = gl & 1;
        const float send = hi1 ? q0 : q1;
        const float keep = hi1 ? q1 : q0;
        return keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
}

// reduce_scatter_steps<4> of two arrays at once (lane gl returns the step-gl totals of both as
// one float2); the additions run as packed f32x2 operations.
__device__ __forceinline__ float2 reduce_scatter_steps4_pair(const float (&a)[4], const float (&b)[4], int gl) {
    const bool hi2 = gl & 2;
    float2 q[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float sa = hi2 ? a[i] : a[i + 2], sb = hi2 ? b[i] : b[i + 2];
        const float ka = hi2 ? a[i + 2] : a[i], kb = hi2 ? b[i + 2] : b[i];
        q[i] = __fadd2_rn(make_float2(ka, kb), make_float2(__shfl_xor_sync(0xffffffffu, sa, 2),
                                                           __shfl_xor_sync(0xffffffffu, sb, 2)));
    }
    const bool hi1 = gl & 1;
    const float2 send = hi1 ? q[0] : q[1];
    const float2 keep = hi1 ? q[1] : q[0];
    return __fadd2_rn(keep, make_float2(__shfl_xor_sync(0xffffffffu, send.x, 1),
                                        __shfl_xor_sync(0xffffffffu, send.y, 1)));
}

// Eight values per lane summed over the 4 lanes of a group (gl = lane & 3): lane gl
// returns the totals of entries 2 gl and 2 gl + 1 (two reduce-scatter stages).
__device__ __forceinline__ float2 reduce_scatter8_over4(const float (&v)[8], int gl) {
    const bool hi2 = gl & 2;
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = hi2 ? v[i] : v[i + 4];
        const float keep = hi2 ? v[i + 4] : v[i];
        w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const bool hi1 = gl & 1;
    float u[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = hi1 ? w[i] : w[i + 2];
        const float keep = hi1 ? w[i + 2] : w[i];
        u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
    return make_float2(u[0], u[1]);
}

}  // namespace ssm
