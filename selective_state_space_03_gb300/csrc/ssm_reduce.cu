// Deterministic backward: the fixed-order sums that replace the atomic adds.
//
// In deterministic mode every backward CTA writes its partial sums instead of
// adding them atomically: for gb and gc one row of 2 x 16 values per (channel
// block, b, t) (its sum over its channels), for gA one row of 16 values per
// (b, chunk, d) (its sum over its steps), and for the skip weights' gradient one value
// per (b, chunk, d). These kernels add the partials in
// increasing block (resp. batch-then-chunk) order, so the result does not
// depend on which CTA finished first. Each thread sums one 16-byte column of
// the partials; the partial arrays are read once (HBM-bound).
#include "ssm_common.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// parts [nblk][B*T][2][16] -> gb, gc [B*T][16]
__global__ void __launch_bounds__(256) reduce_gbc_kernel(const float* __restrict__ parts, int64_t nblk, int64_t rows,
                                                         float* __restrict__ gb, float* __restrict__ gc) {
    const int64_t n4 = rows * 8;                   // float4 columns per block
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4* src = reinterpret_cast<const float4*>(parts) + i;
        float4 acc = src[0];
        for (int64_t k = 1; k < nblk; ++k) acc = add4(acc, src[k * n4]);
        const int64_t row = i >> 3;
        const int tau = int(i >> 2) & 1, q = int(i & 3);
        *reinterpret_cast<float4*>((tau ? gc : gb) + row * kDS + q * 4) = acc;
    }
}

// parts [nparts][D][16] -> gA [D][16]
__global__ void __launch_bounds__(256) reduce_gA_kernel(const float* __restrict__ parts, int64_t nparts, int64_t D,
                                                        float* __restrict__ gA) {
    const int64_t n4 = D * 4;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4* src = reinterpret_cast<const float4*>(parts) + i;
        float4 acc = src[0];
        for (int64_t k = 1; k < nparts; ++k) acc = add4(acc, src[k * n4]);
        reinterpret_cast<float4*>(gA)[i] = acc;
    }
}

// parts [nparts][D] -> gD [D]
__global__ void __launch_bounds__(256) reduce_gD_kernel(const float* __restrict__ parts, int64_t nparts, int64_t D,
                                                        float* __restrict__ gD) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < D; i += int64_t(gridDim.x) * blockDim.x) {
        float acc = parts[i];
        for (int64_t k = 1; k < nparts; ++k) acc += parts[k * D + i];
        gD[i] = acc;
    }
}

unsigned grid_for(int64_t n4) {
    const int64_t want = (n4 + 255) / 256;
    const int64_t cap = int64_t(device_sm_count()) * 8;
    return unsigned(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_bwd_reduce(const BwdLaunch& L, int64_t nblk, int64_t nz, cudaStream_t stream) {
    const int64_t rows = L.B * L.T;
    reduce_gbc_kernel<<<grid_for(rows * 8), 256, 0, stream>>>(L.part_gbc, nblk, rows, L.gb, L.gc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    reduce_gA_kernel<<<grid_for(L.D * 4), 256, 0, stream>>>(L.part_gA, L.B * nz, L.D, L.gA);
    e = cudaGetLastError();
    if (e != cudaSuccess || L.Dskip == nullptr) return e;
    reduce_gD_kernel<<<grid_for(L.D), 256, 0, stream>>>(L.part_gD, L.B * nz, L.D, L.gDskip);
    return cudaGetLastError();
}

}  // namespace ssm
