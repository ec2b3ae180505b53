// Per-SM throughput probes behind the roofline figures that bench.py reports.
//
// The scan's kernels are bound by instruction throughput on the SM, not by
// DRAM, so their roofline needs the GB300's per-SM rates of the units they use:
//   ex2      ex2.approx.ftz.f32 on the special-function unit (MUFU), one per
//            element of the forward, two per element of the backward;
//   ffma     scalar FP32 fused multiply-add;
//   ffma2    packed f32x2 fused multiply-add (one instruction, two lanes' worth);
//   mix      one ex2 and four FFMA per element (the forward's arithmetic);
//   shfl     warp shuffles (the lane reductions);
//   lds      shared-memory loads in the patterns the kernels use, counted as
//            warp-instructions per clock: 16-byte loads where groups of four
//            neighbouring lanes share an address (lane >> 2: the per-channel-pair
//            records), 16-byte loads where the four lanes of a group read four
//            different addresses (lane & 3: the b/c rows), 8-byte loads shared by
//            groups of four, and a shuffle interleaved with a 16-byte load;
//   copy     a device-memory copy of 2 GiB (read + write bytes), for HBM.
// Each compute probe runs one CTA of 1024 threads per SM with 8 independent
// chains per thread, times its loop with clock64 and reports operations per
// clock per SM; the copy is timed with CUDA events. Prints one JSON object.
//
// Build and run (bench.py --rates does both):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o bench_rates bench_rates.cu && ./bench_rates
#include <cstdio>
#include <cuda_runtime.h>

#define CHECK(x)                                                                     \
    do {                                                                             \
        cudaError_t e_ = (x);                                                        \
        if (e_ != cudaSuccess) {                                                     \
            std::printf("{\"error\": \"%s: %s\"}\n", #x, cudaGetErrorString(e_));    \
            return 1;                                                                \
        }                                                                            \
    } while (0)

__device__ __forceinline__ float mufu_ex2(float v) {
    float r;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

enum Probe { kEx2 = 0, kFfma, kFfma2, kMix, kShfl, kLds128, kLds128Quad, kLds128Spread, kLds64Quad, kShflLds,
             kNumProbes };

// ops counted per inner iteration per thread: 8 chains x (1 op), except the mix (8 elements)
// and the shared loads (8 loads; shfl + load: 8 pairs)
template <int P>
__global__ void __launch_bounds__(1024, 1) probe(float* sink, long long* cycles, int iters, float a, float b) {
    __shared__ float4 tile[64];
    if (threadIdx.x < 64) tile[threadIdx.x] = make_float4(threadIdx.x, 1.f, 2.f, 3.f);
    const int lane = threadIdx.x & 31;
    // 16-byte column of the shared-load probes: groups of 4 lanes share one (quad) or the
    // 4 lanes of a group read 4 different ones (spread)
    const int qcol = (P == kLds128Spread) ? (lane & 3) : (lane >> 2);
    float v[8];
    float2 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = -0.01f * float(i + 1) - 1e-6f * float(threadIdx.x);
        w[i] = make_float2(v[i], 0.5f * v[i]);
    }
    __syncthreads();
    const int row = (threadIdx.x >> 3) & 3;          // 4 distinct 16-byte rows per 8 lanes
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (P == kEx2) v[i] = mufu_ex2(v[i]);
            if (P == kFfma) v[i] = fmaf(v[i], a, b);
            if (P == kFfma2) w[i] = __ffma2_rn(w[i], make_float2(a, a), make_float2(b, b));
            if (P == kMix) {
                const float e = mufu_ex2(v[i] * a);
                v[i] = fmaf(fmaf(e, v[i], b), a, e * b);
            }
            if (P == kShfl) v[i] = __shfl_xor_sync(0xffffffffu, v[i], 1 + (i & 7)) + b;
            if (P == kLds128) {             // all four words used: one 16-byte load, two packed adds
                const float4 q = tile[(row + i + it) & 63];
                w[i] = __fadd2_rn(w[i], make_float2(q.x, q.y));
                w[i] = __fadd2_rn(w[i], make_float2(q.z, q.w));
            }
            if (P == kLds128Quad || P == kLds128Spread || P == kShflLds) {
                const float4 q = tile[(qcol + 8 * i + it) & 63];
                w[i] = __fadd2_rn(w[i], make_float2(q.x, q.y));
                w[i] = __fadd2_rn(w[i], make_float2(q.z, q.w));
                if (P == kShflLds) v[i] = __shfl_xor_sync(0xffffffffu, v[i], 1 + (i & 7)) + b;
            }
            if (P == kLds64Quad) {
                const float2 q = reinterpret_cast<const float2*>(tile)[(qcol + 8 * i + it) & 127];
                w[i] = __fadd2_rn(w[i], q);
            }
        }
    }
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i] + w[i].x + w[i].y;
    sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

__global__ void copy_kernel(const float4* __restrict__ src, float4* __restrict__ dst, size_t n) {
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

template <int P>
int run_probe(int sms, float* sink, long long* cycles, long long* host, double* rate, double* mhz) {
    const int iters = 4096;
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    double best = 0.0;
    for (int rep = 0; rep < 3; ++rep) {
        CHECK(cudaEventRecord(e0));
        probe<P><<<sms, 1024>>>(sink, cycles, iters, 0.999f, 0.001f);
        CHECK(cudaEventRecord(e1));
        CHECK(cudaEventSynchronize(e1));
        CHECK(cudaGetLastError());
        float ms = 0.f;
        CHECK(cudaEventElapsedTime(&ms, e0, e1));
        CHECK(cudaMemcpy(host, cycles, sizeof(long long) * sms, cudaMemcpyDeviceToHost));
        double avg = 0.0;
        for (int i = 0; i < sms; ++i) avg += double(host[i]);
        avg /= sms;
        const double ops = 1024.0 * iters * 8;       // per CTA = per SM
        if (ops / avg > best) {
            best = ops / avg;
            *mhz = avg / (ms * 1e3);
        }
    }
    *rate = best;
    CHECK(cudaEventDestroy(e0));
    CHECK(cudaEventDestroy(e1));
    return 0;
}

int main() {
    int dev = 0, sms = 0, clk_khz = 0;
    CHECK(cudaSetDevice(dev));
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CHECK(cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev));
    cudaDeviceProp prop;
    CHECK(cudaGetDeviceProperties(&prop, dev));
    float* sink = nullptr;
    long long* cycles = nullptr;
    CHECK(cudaMalloc(&sink, sizeof(float) * 1024 * sms));
    CHECK(cudaMalloc(&cycles, sizeof(long long) * sms));
    long long* host = new long long[sms];
    const char* names[kNumProbes] = {"ex2", "ffma", "ffma2_pairs", "ex2_plus_4_fp32", "shfl", "lds128_loads",
                                     "lds128_quad_shared_loads", "lds128_quad_spread_loads",
                                     "lds64_quad_shared_loads", "shfl_plus_lds128_pairs"};
    double rate[kNumProbes] = {}, mhz[kNumProbes] = {};
    if (run_probe<kEx2>(sms, sink, cycles, host, &rate[kEx2], &mhz[kEx2])) return 1;
    if (run_probe<kFfma>(sms, sink, cycles, host, &rate[kFfma], &mhz[kFfma])) return 1;
    if (run_probe<kFfma2>(sms, sink, cycles, host, &rate[kFfma2], &mhz[kFfma2])) return 1;
    if (run_probe<kMix>(sms, sink, cycles, host, &rate[kMix], &mhz[kMix])) return 1;
    if (run_probe<kShfl>(sms, sink, cycles, host, &rate[kShfl], &mhz[kShfl])) return 1;
    if (run_probe<kLds128>(sms, sink, cycles, host, &rate[kLds128], &mhz[kLds128])) return 1;
    if (run_probe<kLds128Quad>(sms, sink, cycles, host, &rate[kLds128Quad], &mhz[kLds128Quad])) return 1;
    if (run_probe<kLds128Spread>(sms, sink, cycles, host, &rate[kLds128Spread], &mhz[kLds128Spread])) return 1;
    if (run_probe<kLds64Quad>(sms, sink, cycles, host, &rate[kLds64Quad], &mhz[kLds64Quad])) return 1;
    if (run_probe<kShflLds>(sms, sink, cycles, host, &rate[kShflLds], &mhz[kShflLds])) return 1;

    // HBM: copy 2 GiB, best of 10
    const size_t bytes = size_t(2) << 30, n4 = bytes / 16;
    float4 *src = nullptr, *dst = nullptr;
    CHECK(cudaMalloc(&src, bytes));
    CHECK(cudaMalloc(&dst, bytes));
    CHECK(cudaMemset(src, 0, bytes));
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    float best_ms = 1e30f;
    for (int rep = 0; rep < 10; ++rep) {
        CHECK(cudaEventRecord(e0));
        copy_kernel<<<sms * 8, 512>>>(src, dst, n4);
        CHECK(cudaEventRecord(e1));
        CHECK(cudaEventSynchronize(e1));
        CHECK(cudaGetLastError());
        float ms = 0.f;
        CHECK(cudaEventElapsedTime(&ms, e0, e1));
        if (ms < best_ms) best_ms = ms;
    }
    const double copy_gbs = 2.0 * double(bytes) / (best_ms * 1e-3) / 1e9;

    std::printf("{\"gpu\": \"%s\", \"sms\": %d, \"max_sm_mhz\": %.0f, \"per_sm_per_clk\": {", prop.name, sms,
                clk_khz / 1e3);
    for (int p = 0; p < kNumProbes; ++p)
        std::printf("%s\"%s\": %.2f", p ? ", " : "", names[p], rate[p]);
    std::printf("}, \"sm_mhz_during_probe\": {");
    for (int p = 0; p < kNumProbes; ++p)
        std::printf("%s\"%s\": %.0f", p ? ", " : "", names[p], mhz[p]);
    std::printf("}, \"copy_gbs\": %.1f, \"copy_bytes\": %zu}\n", copy_gbs, 2 * bytes);
    delete[] host;
    return 0;
}
