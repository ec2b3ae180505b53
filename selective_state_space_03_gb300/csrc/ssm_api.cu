// C ABI of libssm_scan.so: argument checks, schedule choice and launches.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "ssm_internal.h"
#include "ssm_scan.h"

// Schedule overrides for tests, read from the environment at each call. They exist only in
// the testing build of the library (libssm_scan_testing.so, compiled with SSM_SCAN_TESTING);
// in the release library the macro is a null pointer, so the names are not even compiled in
// and these variables have no effect.
#ifdef SSM_SCAN_TESTING
#define SSM_TEST_ENV(name) std::getenv(name)
#else
#define SSM_TEST_ENV(name) (static_cast<const char*>(nullptr))
#endif

namespace ssm {

#ifdef SSM_SCAN_TESTING
// testing build only: the SM count the schedule queries assume (0 = the device's)
thread_local int g_test_sms = 0;
#endif

int device_sm_count() {
#ifdef SSM_SCAN_TESTING
    if (g_test_sms > 0) return g_test_sms;
#endif
    static std::atomic<int> cache[64];      // per device, filled on first use (0 = not yet)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    if (dev >= 0 && dev < 64 && cache[dev].load() > 0) return cache[dev].load();
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 152;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(n);
    return n;
}

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssm_status check_desc(const ssm_scan_desc* d) {
    if (d == nullptr) return SSM_ERR_INVALID_ARG;
    if (d->B < 0 || d->T < 0 || d->D < 0 || d->DS < 0) return SSM_ERR_INVALID_ARG;
    if (d->io != SSM_IO_F32 && d->io != SSM_IO_BF16) return SSM_ERR_INVALID_ARG;
    constexpr int32_t kFlags = SSM_SCAN_DETERMINISTIC | SSM_SCAN_DELTA_SOFTPLUS | SSM_SCAN_LOOKBACK | SSM_SCAN_STEP_INPUTS_READY;
    if (d->ckpt_interval < 0 || (d->flags & ~kFlags) != 0) return SSM_ERR_INVALID_ARG;
    if (d->B > 65535) return SSM_ERR_INVALID_ARG;
    if (d->DS != kDS) return SSM_ERR_UNSUPPORTED;
    if (d->D > kMaxD) return SSM_ERR_UNSUPPORTED;     // kernels use 32-bit in-tile offsets
    return SSM_OK;
}

int64_t io_size(const ssm_scan_desc& d) { return d.io == SSM_IO_BF16 ? 2 : 4; }

// 16-byte staging needs rows of x-like tensors to be whole 16-byte chunks.
bool vec_ok(const ssm_scan_desc& d) { return (d.D * io_size(d)) % 16 == 0; }

struct FwdPlan {
    int mode;        // kSingle (0), chunked (2, meaning pass 1 + pass 2) or chunked in one launch (4)
    int G;
    int kd;          // channels per lane of the G = 4 layout (1 or 2)
    int64_t Lc;
    int64_t nchunk;
    size_t ws_S, ws_Sd;   // byte sizes of the two workspace arrays (mode 2)
    // mode 4: maps, inclusive states, delta sums, then the zeroed block (flags, ticket, status)
    size_t lb_S, lb_X, lb_Sd, lb_zero;
    size_t ws_total() const { return mode == 4 ? lb_S + lb_X + lb_Sd + lb_zero : ws_S + ws_Sd; }
};

// polls of a predecessor's flag before a look-back wait gives up (about a second)
int64_t lookback_polls() {
    if (const char* env = SSM_TEST_ENV("SSM_SCAN_LOOKBACK_POLLS")) {     // testing build only
        const long long v = std::atoll(env);
        if (v > 0) return v;
    }
    return int64_t(1) << 20;
}

FwdPlan plan_fwd(const ssm_scan_desc& d) {
    FwdPlan P{0, 4, 1, d.T, 1, 0, 0, 0, 0, 0, 0};
    const int64_t chains = d.B * d.D;
    const int64_t want = int64_t(device_sm_count()) * 512;   // ~16 resident warps per SM
    // Chosen by the library: chunked when one pass would leave fewer than about 16 warps per SM
    // (4 lanes per chain), and for long sequences up to about 84 chains per SM, where the one-pass
    // grid leaves one or two warps per SMSP and the second sweep over T costs less than the
    // latency it hides (4096 steps, bf16, one pass -> chunked: 8192 chains 298 -> 216 us, 10240
    // chains 341 -> 259 us, 12288 chains 343 -> 310 us; 16384 chains one pass 349 us, chunked
    // 382-431 us).
    const bool few_chains = chains * 4 * 2 < want ||
                            (chains < int64_t(device_sm_count()) * 84 && d.T >= 2048);
    bool chunked = false;
    ChunkSchedule cs{0, 1, 4};
    if (d.chunk_len > 0 || (d.chunk_len == 0 && few_chains && d.T >= 256)) {
        cs = chunk_schedule(d.T, chains, d.chunk_len, device_sm_count());
        chunked = cdiv(d.T, cs.Lc) >= 2;
    }
    if (chunked) {
        P.mode = 2;
        P.G = cs.G;
        P.kd = cs.kd;
        // testing build only: channels per lane of both chunk passes with 4 lanes per chain (1 or
        // 2), or their layout ("2x2", "4x2", "4x1")
        if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_CHUNK_KD")) {
            P.G = 4;
            P.kd = std::atoi(env) == 2 ? 2 : 1;
        }
        if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_CHUNK_LAYOUT")) {
            if (std::strcmp(env, "2x2") == 0) { P.G = 2; P.kd = 2; }
            if (std::strcmp(env, "4x2") == 0) { P.G = 4; P.kd = 2; }
            if (std::strcmp(env, "4x1") == 0) { P.G = 4; P.kd = 1; }
        }
        P.Lc = cs.Lc;
        P.nchunk = cdiv(d.T, cs.Lc);
        P.ws_S = align_up(size_t(d.B) * size_t(P.nchunk - 1) * size_t(d.D) * kDS * 4);
        P.ws_Sd = align_up(size_t(d.B) * size_t(P.nchunk - 1) * size_t(d.D) * 4);
        if (d.flags & SSM_SCAN_LOOKBACK) {
            P.mode = 4;
            P.G = 4;                  // the look-back kernel runs 4 lanes per chain
            const size_t rows = size_t(d.B) * size_t(P.nchunk) * size_t(d.D);
            const size_t nblk = size_t(cdiv(d.D, 8 * P.kd));
            P.lb_S = align_up(rows * kDS * 4);
            P.lb_X = align_up(rows * kDS * 4);
            P.lb_Sd = align_up(rows * 4);
            P.lb_zero = align_up((size_t(P.nchunk) + 1) * size_t(d.B) * nblk * 4 + 16);
        }
    } else {
        // Lane layout: the most channels per warp (fewest lanes re-reading each b, c value
        // from shared memory) that still keeps enough warps resident: 2 lanes per chain x 2
        // channels per lane (32 channels per warp) from about 12 warps per SM, 4 lanes x 2
        // channels (16 per warp) from about 4 warps per SM, else 4 lanes x 1 channel (8).
        const int64_t sms = device_sm_count();
        P.G = chains >= sms * 12 * 32 ? 2 : 4;
        P.kd = (P.G == 2 || chains >= sms * 4 * 16) ? 2 : 1;
        // testing build only: force the layout ("2x2", "4x2", "4x1"; the older SSM_SCAN_FORCE_LANES
        // takes 2 for 2x2 and 4 for 4x1)
        if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_LANES")) {
            const int g = std::atoi(env);
            if (g == 2 || g == 4) { P.G = g; P.kd = g == 2 ? 2 : 1; }
        }
        if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_FWD_LAYOUT")) {
            if (std::strcmp(env, "2x2") == 0) { P.G = 2; P.kd = 2; }
            if (std::strcmp(env, "4x2") == 0) { P.G = 4; P.kd = 2; }
            if (std::strcmp(env, "4x1") == 0) { P.G = 4; P.kd = 1; }
        }
    }
    return P;
}

cudaError_t run_fwd(const ssm_scan_desc& d, FwdLaunch L, int mode, cudaStream_t st) {
    return d.io == SSM_IO_BF16 ? launch_fwd_bf16(L, mode, st) : launch_fwd_f32(L, mode, st);
}

// Backward layout: 2 channels per lane (64 per CTA, 3 CTAs per SM) when that gives
// at least 4 CTAs per SM; otherwise 1 (32 per CTA, 4 per SM with bf16 I/O), which
// keeps more SMs busy on shapes with few (b, d) chains.
int bwd_channels_per_lane(const ssm_scan_desc& d) {
    int kd = d.B * cdiv(d.D, 64) >= int64_t(device_sm_count()) * 4 ? 2 : 1;
    // testing build only: force the layout (1 or 2)
    if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_BWD_KD")) {
        const int k = std::atoi(env);
        if (k == 1 || k == 2) kd = k;
    }
    return kd;
}

int64_t bwd_internal_K(const ssm_scan_desc& d) {
    return (d.ckpt_interval > 0 && d.ckpt_interval <= kMaxBwdK) ? d.ckpt_interval : kMaxBwdK;
}

// Chunk-parallel backward: when one CTA per (channel block, batch) would not fill one
// wave of the GPU (4 CTAs per SM of the one-channel layout) and there are at least two
// checkpoint chunks, each chunk gets its own CTA (a carry pass first supplies the adjoint
// entering it). Needs the carries in the workspace.
bool bwd_chunk_parallel(const ssm_scan_desc& d) {
    const int64_t nck = cdiv(d.T, bwd_internal_K(d));
    if (nck < 2 || nck > 65535) return false;
    bool on = bwd_channels_per_lane(d) == 1 && d.B * cdiv(d.D, 32) < int64_t(device_sm_count()) * 4;
    // testing build only: force the schedule on (1) or off (0)
    if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_BWD_TPAR")) {
        const int k = std::atoi(env);
        if (k == 0 || k == 1) on = k == 1;
    }
    return on;
}

// Workspace of the chunk-parallel backward: carry_Z [nck][B][D][16], then carry_S [nck][B][D].
size_t bwd_carry_Z_bytes(const ssm_scan_desc& d) {
    return align_up(size_t(cdiv(d.T, bwd_internal_K(d))) * size_t(d.B) * size_t(d.D) * kDS * 4);
}
size_t bwd_carry_bytes(const ssm_scan_desc& d) {
    if (!bwd_chunk_parallel(d)) return 0;
    return bwd_carry_Z_bytes(d) + align_up(size_t(cdiv(d.T, bwd_internal_K(d))) * size_t(d.B) * size_t(d.D) * 4);
}

// Backward workspace, in this order: chunk-parallel carries, deterministic partials of
// gb/gc and of gA, rebuilt checkpoints. A call with the forward's checkpoints uses the
// first three (`with_ckpt`), a call without them all four.
struct BwdWorkspace {
    size_t carry = 0, part_gbc = 0, part_gA = 0, part_gD = 0, rebuild = 0;
    int64_t nblk = 0, nz = 1;      // channel blocks and chunks per (b, block) of the partials
    size_t with_ckpt() const { return carry + part_gbc + part_gA + part_gD; }
    size_t total() const { return with_ckpt() + rebuild; }
};

BwdWorkspace bwd_workspace(const ssm_scan_desc& d) {
    BwdWorkspace w;
    const int64_t nck = cdiv(d.T, bwd_internal_K(d));
    w.carry = bwd_carry_bytes(d);
    const bool tpar = w.carry > 0;
    const int kd = tpar ? 1 : bwd_channels_per_lane(d);
    w.nblk = cdiv(d.D, kd == 2 ? 64 : 32);
    w.nz = tpar ? nck : 1;
    if (d.flags & SSM_SCAN_DETERMINISTIC) {
        w.part_gbc = align_up(size_t(w.nblk) * size_t(d.B) * size_t(d.T) * 2 * kDS * 4);
        w.part_gA = align_up(size_t(d.B) * size_t(w.nz) * size_t(d.D) * kDS * 4);
        w.part_gD = align_up(size_t(d.B) * size_t(w.nz) * size_t(d.D) * 4);    // skip weights' gradient
    }
    w.rebuild = align_up(size_t(nck) * size_t(d.B) * size_t(d.D) * kDS * 4);
    return w;
}

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" {

const char* ssm_status_str(ssm_status s) {
    switch (s) {
        case SSM_OK: return "ok";
        case SSM_ERR_INVALID_ARG: return "invalid argument";
        case SSM_ERR_UNSUPPORTED: return "unsupported shape (DS must be 16, D at most 2^27, at most 65535 chunks)";
        case SSM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case SSM_ERR_WORKSPACE: return "workspace missing or too small";
        case SSM_ERR_CUDA: return "CUDA error";
        case SSM_ERR_TIMEOUT: return "a look-back wait of the one-launch chunked scan ran out";
    }
    return "unknown status";
}

size_t ssm_scan_ckpt_bytes(const ssm_scan_desc* d) {
    if (check_desc(d) != SSM_OK || d->ckpt_interval <= 0) return 0;
    return size_t(cdiv(d->T, d->ckpt_interval)) * size_t(d->B) * size_t(d->D) * size_t(d->DS) * 4;
}

size_t ssm_scan_fwd_workspace_bytes(const ssm_scan_desc* d) {
    if (check_desc(d) != SSM_OK || d->B == 0 || d->T == 0 || d->D == 0) return 0;
    const FwdPlan P = plan_fwd(*d);
    return P.mode == 0 ? 0 : P.ws_total();
}

size_t ssm_scan_bwd_ckpt_workspace_bytes(const ssm_scan_desc* d) {
    if (check_desc(d) != SSM_OK || d->B == 0 || d->T == 0 || d->D == 0) return 0;
    return bwd_workspace(*d).with_ckpt();
}

size_t ssm_scan_bwd_workspace_bytes(const ssm_scan_desc* d) {
    if (check_desc(d) != SSM_OK || d->B == 0 || d->T == 0 || d->D == 0) return 0;
    return bwd_workspace(*d).total();
}

ssm_status ssm_scan_fwd_fused(const ssm_scan_desc* desc, const void* x, const void* delta, const float* A,
                              const void* b, const void* c, const float* D_skip, const float* h0, void* y,
                              float* hT, float* ckpt, void* workspace, size_t workspace_bytes, void* stream) {
    ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    const ssm_scan_desc& d = *desc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool work = d.B > 0 && d.T > 0 && d.D > 0;
    if (work && (!x || !delta || !A || !b || !c || !y)) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, delta, A, b, c, D_skip, h0, y, hT, ckpt};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_MISALIGNED;
    if (!work) {
        // empty sequence (or no chains): hT = h0, nothing else to write
        if (hT && d.B > 0 && d.D > 0) {
            const size_t bytes = size_t(d.B) * size_t(d.D) * kDS * 4;
            const cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, s)
                                     : cudaMemsetAsync(hT, 0, bytes, s);
            if (e != cudaSuccess) return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    const FwdPlan P = plan_fwd(d);
    if (P.mode != 0 && P.nchunk > kMaxChunks) return SSM_ERR_UNSUPPORTED;   // one grid dimension per chunk
    if (P.mode != 0 && (workspace == nullptr || workspace_bytes < P.ws_total())) return SSM_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return SSM_ERR_MISALIGNED;

    FwdLaunch L{};
    L.x = x; L.delta = delta; L.A = A; L.b = b; L.c = c; L.h0 = h0;
    L.y = y; L.hT = hT; L.ckpt = d.ckpt_interval > 0 ? ckpt : nullptr;
    L.B = d.B; L.T = d.T; L.D = d.D; L.K = d.ckpt_interval;
    L.io = d.io == SSM_IO_BF16 ? IO::BF16 : IO::F32;
    L.vec = vec_ok(d);
    L.ckpt_only = false;
    L.G = P.G;
    L.kd = P.kd;
    L.softplus = (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0;
    L.Dskip = D_skip;
    cudaError_t e;
    if (P.mode == 2) {
        L.Lc = P.Lc;
        L.nchunk = P.nchunk;
        L.ws_S = static_cast<float*>(workspace);
        L.ws_Sd = reinterpret_cast<float*>(static_cast<char*>(workspace) + P.ws_S);
        e = run_fwd(d, L, 1, s);
        bool scan = P.nchunk - 1 > kCarryScanMinCarries;
        // testing build only: force the middle pass on (1) or off (0)
        if (const char* env = SSM_TEST_ENV("SSM_SCAN_FORCE_CARRY_SCAN")) scan = std::atoi(env) == 1;
        if (e == cudaSuccess && scan) {
            L.carry_scanned = true;
            e = launch_fwd_carry_scan(L, s);
        }
        if (e == cudaSuccess) e = run_fwd(d, L, 2, s);
    } else if (P.mode == 4) {
        char* w = static_cast<char*>(workspace);
        L.Lc = P.Lc;
        L.nchunk = P.nchunk;
        L.lb_S = reinterpret_cast<float*>(w);
        L.lb_X = reinterpret_cast<float*>(w + P.lb_S);
        L.lb_Sd = reinterpret_cast<float*>(w + P.lb_S + P.lb_X);
        char* z = w + P.lb_S + P.lb_X + P.lb_Sd;      // status (4 B), pad, flags, tickets
        const size_t nblk = size_t(cdiv(d.D, 8 * P.kd));
        L.lb_status = reinterpret_cast<unsigned int*>(z + 8);
        L.lb_flags = reinterpret_cast<int*>(z + 16);
        L.lb_ticket = reinterpret_cast<int*>(z + 16 + size_t(P.nchunk) * size_t(d.B) * nblk * 4);
        L.lb_polls = lookback_polls();
        L.lb_test_drop = SSM_TEST_ENV("SSM_SCAN_TEST_LOOKBACK_DROP") != nullptr;   // testing build only
        e = cudaMemsetAsync(z, 0, P.lb_zero, s);
        if (e == cudaSuccess) e = run_fwd(d, L, 4, s);
    } else {
        L.Lc = d.T;
        L.nchunk = 1;
        e = run_fwd(d, L, 0, s);
    }
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_scan_fwd_lookback_status(const ssm_scan_desc* desc, const void* workspace, size_t workspace_bytes,
                                         void* stream) {
    ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    const FwdPlan P = plan_fwd(*desc);
    if (P.mode != 4 || desc->B == 0 || desc->T == 0 || desc->D == 0) return SSM_OK;    // nothing waited
    // the status word's place does not depend on the lane layout (which sizes the flags)
    if (workspace == nullptr || workspace_bytes < P.lb_S + P.lb_X + P.lb_Sd + 16) return SSM_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SSM_ERR_MISALIGNED;
    unsigned int n = 0;
    const char* z = static_cast<const char*>(workspace) + P.lb_S + P.lb_X + P.lb_Sd;
    if (cudaMemcpyAsync(&n, z + 8, sizeof(n), cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SSM_ERR_CUDA;
    return n == 0 ? SSM_OK : SSM_ERR_TIMEOUT;
}

ssm_status ssm_scan_fwd(const ssm_scan_desc* desc, const void* x, const void* delta, const float* A,
                        const void* b, const void* c, const float* h0, void* y, float* hT, float* ckpt,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return ssm_scan_fwd_fused(desc, x, delta, A, b, c, nullptr, h0, y, hT, ckpt, workspace, workspace_bytes,
                              stream);
}

ssm_status ssm_scan_bwd_fused(const ssm_scan_desc* desc, const void* x, const void* delta, const float* A,
                              const void* b, const void* c, const float* D_skip, const float* h0,
                              const float* ckpt, const void* dy, const float* ghT, float* gx, float* gdelta,
                              float* gA, float* gb, float* gc, float* gh0, float* gD_skip, void* workspace,
                              size_t workspace_bytes, void* stream) {
    ssm_status st = check_desc(desc);
    if (st != SSM_OK) return st;
    const ssm_scan_desc& d = *desc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool work = d.B > 0 && d.T > 0 && d.D > 0;
    if (work && (!x || !delta || !A || !b || !c || !dy || !gx || !gdelta || !gb || !gc)) return SSM_ERR_INVALID_ARG;
    if (d.D > 0 && !gA) return SSM_ERR_INVALID_ARG;
    if (d.B > 0 && d.D > 0 && !gh0) return SSM_ERR_INVALID_ARG;
    if (D_skip && d.D > 0 && !gD_skip) return SSM_ERR_INVALID_ARG;
    const void* ptrs[] = {x, delta, A, b, c, D_skip, h0, ckpt, dy, ghT, gx, gdelta, gA, gb, gc, gh0, gD_skip};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return SSM_ERR_MISALIGNED;
    if (!work) {
        // no steps: gA = 0, gh0 = ghT (zeros without ghT); gb, gc have no rows unless D == 0
        cudaError_t e = cudaSuccess;
        if (d.D > 0) e = cudaMemsetAsync(gA, 0, size_t(d.D) * kDS * 4, s);
        if (e == cudaSuccess && D_skip && d.D > 0) e = cudaMemsetAsync(gD_skip, 0, size_t(d.D) * 4, s);
        if (e == cudaSuccess && d.B > 0 && d.D > 0) {
            const size_t bytes = size_t(d.B) * size_t(d.D) * kDS * 4;
            e = ghT ? cudaMemcpyAsync(gh0, ghT, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(gh0, 0, bytes, s);
        }
        if (e == cudaSuccess && d.D == 0 && d.B > 0 && d.T > 0) {
            // no channels: the sums over d are empty
            const size_t bytes = size_t(d.B) * size_t(d.T) * kDS * 4;
            if (gb) e = cudaMemsetAsync(gb, 0, bytes, s);
            if (e == cudaSuccess && gc) e = cudaMemsetAsync(gc, 0, bytes, s);
        }
        return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    }

    // workspace: [carries][deterministic partials][rebuilt checkpoints]
    const BwdWorkspace W = bwd_workspace(d);
    const bool det = (d.flags & SSM_SCAN_DETERMINISTIC) != 0;
    if (workspace != nullptr && !aligned16(workspace)) return SSM_ERR_MISALIGNED;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    // checkpoints: the forward's, or rebuilt in the workspace
    const float* ck = ckpt;
    int64_t K = d.ckpt_interval;
    const bool rebuild = (ckpt == nullptr) || K <= 0 || K > kMaxBwdK;
    if (rebuild && (workspace == nullptr || workspace_bytes < W.total())) return SSM_ERR_WORKSPACE;
    if (det && (workspace == nullptr || workspace_bytes < W.with_ckpt())) return SSM_ERR_WORKSPACE;
    // with the forward's checkpoints and no deterministic partials the carries are optional:
    // without room for them the backward sweeps every chain in one CTA
    const bool tpar = W.carry > 0 && workspace != nullptr && workspace_bytes >= W.carry;
    if (rebuild) {
        K = bwd_internal_K(d);
        FwdLaunch L{};
        L.x = x; L.delta = delta; L.A = A; L.b = b; L.c = c; L.h0 = h0;
        L.y = nullptr; L.hT = nullptr;
        L.ckpt = reinterpret_cast<float*>(ws + W.with_ckpt());
        L.B = d.B; L.T = d.T; L.D = d.D; L.K = K; L.Lc = d.T; L.nchunk = 1;
        L.io = d.io == SSM_IO_BF16 ? IO::BF16 : IO::F32;
        L.vec = vec_ok(d);
        L.G = 4;
        L.ckpt_only = true;
        L.softplus = (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0;
        if (run_fwd(d, L, 3, s) != cudaSuccess) return SSM_ERR_CUDA;
        ck = L.ckpt;
    }

    if (!det) {   // atomic accumulation targets (the deterministic sums overwrite them instead)
        if (cudaMemsetAsync(gA, 0, size_t(d.D) * kDS * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
        const size_t bts = size_t(d.B) * size_t(d.T) * kDS * 4;
        if (cudaMemsetAsync(gb, 0, bts, s) != cudaSuccess) return SSM_ERR_CUDA;
        if (cudaMemsetAsync(gc, 0, bts, s) != cudaSuccess) return SSM_ERR_CUDA;
        if (D_skip && cudaMemsetAsync(gD_skip, 0, size_t(d.D) * 4, s) != cudaSuccess) return SSM_ERR_CUDA;
    }

    BwdLaunch L{};
    L.x = x; L.delta = delta; L.A = A; L.b = b; L.c = c; L.ckpt = ck; L.dy = dy; L.ghT = ghT;
    L.gx = gx; L.gdelta = gdelta; L.gA = gA; L.gb = gb; L.gc = gc; L.gh0 = gh0;
    L.B = d.B; L.T = d.T; L.D = d.D; L.K = K;
    L.io = d.io == SSM_IO_BF16 ? IO::BF16 : IO::F32;
    L.vec = vec_ok(d);
    L.kd = bwd_channels_per_lane(d);
    L.tpar = tpar;
    L.softplus = (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0;
    if (tpar) {
        L.kd = 1;
        L.carry_Z = reinterpret_cast<float*>(ws);
        L.carry_S = reinterpret_cast<float*>(ws + bwd_carry_Z_bytes(d));
        const cudaError_t e1 = d.io == SSM_IO_BF16 ? launch_bwd_carry_bf16(L, s) : launch_bwd_carry_f32(L, s);
        if (e1 != cudaSuccess) return SSM_ERR_CUDA;
    }
    L.softplus = (d.flags & SSM_SCAN_DELTA_SOFTPLUS) != 0;
    L.Dskip = D_skip;
    L.gDskip = gD_skip;
    L.det = det;
    if (det) {
        L.part_gbc = reinterpret_cast<float*>(ws + W.carry);
        L.part_gA = reinterpret_cast<float*>(ws + W.carry + W.part_gbc);
        L.part_gD = reinterpret_cast<float*>(ws + W.carry + W.part_gbc + W.part_gA);
    }
    cudaError_t e = d.io == SSM_IO_BF16 ? launch_bwd_bf16(L, s) : launch_bwd_f32(L, s);
    if (e == cudaSuccess && det) e = launch_bwd_reduce(L, W.nblk, W.nz, s);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

ssm_status ssm_scan_bwd(const ssm_scan_desc* desc, const void* x, const void* delta, const float* A,
                        const void* b, const void* c, const float* h0, const float* ckpt, const void* dy,
                        const float* ghT, float* gx, float* gdelta, float* gA, float* gb, float* gc,
                        float* gh0, void* workspace, size_t workspace_bytes, void* stream) {
    return ssm_scan_bwd_fused(desc, x, delta, A, b, c, nullptr, h0, ckpt, dy, ghT, gx, gdelta, gA, gb, gc, gh0,
                              nullptr, workspace, workspace_bytes, stream);
}

}  // extern "C"

#ifdef SSM_SCAN_TESTING
// Testing build only: the schedule the library would choose for desc on a GPU with `sms` SMs,
// computed on the host without touching a device. out[0..4]: forward mode (0 one pass,
// 2 chunked, 4 chunked with look-back), lanes per chain, channels per lane, chunk length,
// chunks; out[5..7]: backward channels per lane, chunk-parallel (0/1), its chunk length.
extern "C" int ssm_testing_schedule(const ssm_scan_desc* desc, int sms, int64_t* out) {
    if (desc == nullptr || out == nullptr || sms <= 0) return SSM_ERR_INVALID_ARG;
    ssm::g_test_sms = sms;
    const ssm::FwdPlan P = ssm::plan_fwd(*desc);
    out[0] = P.mode;
    out[1] = P.G;
    out[2] = P.kd;
    out[3] = P.Lc;
    out[4] = P.nchunk;
    const bool tpar = ssm::bwd_chunk_parallel(*desc);
    out[5] = tpar ? 1 : ssm::bwd_channels_per_lane(*desc);
    out[6] = tpar ? 1 : 0;
    out[7] = ssm::bwd_internal_K(*desc);
    ssm::g_test_sms = 0;
    return SSM_OK;
}
#endif
