// ssm_scan_fwd_noalloc: the chunked forward scan with its scratch memory in a
// fixed device array owned by this library, for callers that cannot allocate.
//
// The chunked forward needs scratch for the per-chunk carries (partial end
// states and delta sums). ssm_scan_fwd takes that scratch from the caller.
// Some callers cannot provide it: code running inside another runtime that
// owns all device memory and forbids allocation while it executes (a plugin
// in an inference engine, a step replayed from a captured graph), or services
// that must never call cudaMalloc on the hot path because it synchronises the
// device and can fail under memory pressure. This entry point takes the
// scratch from `g_scratch` below instead, so it allocates nothing.
//
// Costs and rules of that choice:
//  - every GPU that loads the library holds kNoallocScratchBytes of device
//    memory for this array until the process exits;
//  - host code cannot use the array's name as a device address, so every call
//    looks the address up (cudaGetSymbolAddress) in the context current on the
//    calling thread: each CUDA context (each device's primary context, a
//    driver-API context of the caller's, the context that replaces one after a
//    device reset) has its own copy of the array, and a cached address would
//    outlive its context. The first call in a context loads the library's device
//    code there, so make it before any stream capture;
//  - every call on a device shares the one array: calls that overlap on the
//    GPU (other streams, other host threads) race on it and must be ordered by
//    the caller. Pass 1 overwrites every entry pass 2 reads, so nothing in the
//    array needs clearing between calls.
#include <algorithm>

#include "ssm_internal.h"
#include "ssm_scan.h"

namespace ssm {

namespace {

constexpr size_t kNoallocScratchBytes = SSM_SCAN_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_scratch[kNoallocScratchBytes];

// Device address of g_scratch in the calling thread's current context (a host-side lookup
// once the context has loaded the library's device code; it allocates nothing).
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" ssm_status ssm_scan_fwd_noalloc(const ssm_scan_desc* desc, const void* x, const void* delta,
                                           const float* A, const void* b, const void* c, const float* h0,
                                           void* y, float* hT, float* ckpt, void* stream) {
    if (desc == nullptr) return SSM_ERR_INVALID_ARG;
    const ssm_scan_desc& d = *desc;
    if (d.B < 0 || d.T < 0 || d.D < 0 || d.DS < 0) return SSM_ERR_INVALID_ARG;
    if (d.io != SSM_IO_F32 && d.io != SSM_IO_BF16) return SSM_ERR_INVALID_ARG;
    if (d.ckpt_interval < 0 || (d.flags & ~(SSM_SCAN_DETERMINISTIC | SSM_SCAN_DELTA_SOFTPLUS | SSM_SCAN_LOOKBACK | SSM_SCAN_STEP_INPUTS_READY)) != 0 || d.B > 65535) return SSM_ERR_INVALID_ARG;
    if (d.DS != kDS) return SSM_ERR_UNSUPPORTED;
    if (d.D > kMaxD) return SSM_ERR_UNSUPPORTED;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool work = d.B > 0 && d.T > 0 && d.D > 0;
    if (work && (!x || !delta || !A || !b || !c || !y)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, delta, A, b, c, h0, y, hT, ckpt};
    for (const void* p : ptrs)
        if (p && !is_aligned16(p)) return SSM_ERR_MISALIGNED;
    if (!work) {
        if (hT && d.B > 0 && d.D > 0) {
            const size_t bytes = size_t(d.B) * size_t(d.D) * kDS * 4;
            const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, s)
                                     : cudaMemsetAsync(hT, 0, bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }

    // chunk length and lanes: the schedule ssm_scan_fwd uses for its chunked scan (with the
    // caller's chunk length when given); a chunk length the library chose is doubled until the
    // carries fit the scratch array
    auto carry_bytes = [&](int64_t n) {
        return up256(size_t(d.B) * size_t(n - 1) * size_t(d.D) * kDS * 4) + up256(size_t(d.B) * size_t(n - 1) * size_t(d.D) * 4);
    };
    ChunkSchedule cs = chunk_schedule(d.T, d.B * d.D, d.chunk_len > 0 ? d.chunk_len : 0, device_sm_count());
    if (d.chunk_len <= 0) {
        while (cdiv64(d.T, cs.Lc) >= 2 && carry_bytes(cdiv64(d.T, cs.Lc)) > kNoallocScratchBytes)
            cs = chunk_schedule(d.T, d.B * d.D, cs.Lc * 2, device_sm_count());
    }
    const int64_t Lc = cs.Lc;
    const int64_t nchunk = cdiv64(d.T, Lc);
    if (nchunk > kMaxChunks) return SSM_ERR_UNSUPPORTED;      // one grid dimension per chunk

    FwdLaunch L{};
    L.x = x; L.delta = delta; L.A = A; L.b = b; L.c = c; L.h0 = h0;
    L.y = y; L.hT = hT; L.ckpt = d.ckpt_interval > 0 ? ckpt : nullptr;
    L.B = d.B; L.T = d.T; L.D = d.D; L.K = d.ckpt_interval;
    L.io = d.io == SSM_IO_BF16 ? IO::BF16 : IO::F32;
    L.vec = (d.D * (d.io == SSM_IO_BF16 ? 2 : 4)) % 16 == 0;
    L.ckpt_only = false;
    L.G = cs.G;
    L.kd = cs.kd;
    L.softplus = (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0;
    auto run = [&](int mode) {
        return d.io == SSM_IO_BF16 ? launch_fwd_bf16(L, mode, s) : launch_fwd_f32(L, mode, s);
    };
    if (nchunk < 2) {            // one chunk: the one-pass scan, which needs no scratch
        L.Lc = d.T;
        L.nchunk = 1;
        return run(0) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    }
    const size_t bytes_S = up256(size_t(d.B) * size_t(nchunk - 1) * size_t(d.D) * kDS * 4);
    if (carry_bytes(nchunk) > kNoallocScratchBytes) return SSM_ERR_WORKSPACE;

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return SSM_ERR_CUDA;
    L.Lc = Lc;
    L.nchunk = nchunk;
    L.ws_S = static_cast<float*>(base);
    L.ws_Sd = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + bytes_S);
    cudaError_t e = run(1);
    if (e == cudaSuccess && nchunk - 1 > kCarryScanMinCarries) {    // start states folded in place
        L.carry_scanned = true;
        e = launch_fwd_carry_scan(L, s);
    }
    if (e == cudaSuccess) e = run(2);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
