// Host-side interface between the C ABI (ssm_api.cu) and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ssm {

constexpr int kDS = 16;                  // state size the kernels are built for
constexpr int64_t kMaxD = int64_t(1) << 27;   // channels: in-tile offsets (16 rows x D) stay in 32 bits
constexpr int64_t kMaxChunks = 65535;         // chunks of the chunked forward (a grid dimension)

enum class IO { F32 = 0, BF16 = 1 };

// Forward launch description. `mode` selects the schedule:
//   0: one pass over T per (b, d) chain;
//   1: chunked pass 1, per chunk the local end state (zero start) and the
//      delta sum, written to the workspace (all chunks but the last);
//   2: chunked pass 2, per chunk the start state from the carries of all
//      earlier chunks, then the scan of the chunk with readout.
struct FwdLaunch {
    const void* x;
    const void* delta;
    const float* A;
    const void* b;
    const void* c;
    const float* h0;
    void* y;        // may be null only in mode 1, or when ckpt_only
    float* hT;      // may be null
    float* ckpt;    // may be null
    float* ws_S;    // [B][nchunk-1][D][16]   (chunked modes)
    float* ws_Sd;   // [B][nchunk-1][D]       (chunked modes)
    bool carry_scanned;  // mode 2: ws_S holds the start states of chunks 1.. (launch_fwd_carry_scan)
    int64_t B, T, D;
    int64_t K;      // checkpoint interval, 0 = none
    int64_t Lc;     // chunk length (chunked modes; T in mode 0)
    int64_t nchunk; // number of chunks (1 in mode 0)
    IO io;
    int G;          // lane layout: 2 (2 lanes per chain x 2 channels per lane) or 4 (4 lanes per chain)
    int kd;         // with G = 4: channels per lane, 1 or 2 (one-pass schedule only)
    bool vec;       // 16-byte staging allowed
    bool ckpt_only; // mode 0 without readout (checkpoint rebuild for the backward)
    // fused prologue / epilogue (the fused kernel variants only)
    bool softplus;       // delta holds raw values; the scan uses softplus(delta)
    const float* Dskip;  // (D) or null: y += Dskip[d] * x
    // chunked scan in one launch with decoupled look-back (mode 4)
    float* lb_S;                    // [B][nchunk][D][16] chunk maps' offsets (end state from a zero start)
    float* lb_X;                    // [B][nchunk][D][16] inclusive states (state after the chunk)
    float* lb_Sd;                   // [B][nchunk][D] delta sums of the chunks
    int* lb_flags;                  // [nchunk][B][nblk]: 0 nothing, 1 map, 2 inclusive state published
    int* lb_ticket;                 // [B][nblk] next chunk of each chain block, taken in launch order
    unsigned int* lb_status;        // number of waits that ran out (0 after a good launch)
    int64_t lb_polls;               // polls of a predecessor's flag (per CTA) before giving up
    bool lb_test_drop;              // testing aid: chunk 0 publishes nothing, so its successors time out
};

cudaError_t launch_fwd_f32(const FwdLaunch& L, int mode, cudaStream_t stream);
cudaError_t launch_fwd_bf16(const FwdLaunch& L, int mode, cudaStream_t stream);
// Between the chunked passes: overwrite each chunk's carry S_j in ws_S with the start state of
// chunk j + 1 (one sweep per chain), for pass 2 with carry_scanned set.
cudaError_t launch_fwd_carry_scan(const FwdLaunch& L, cudaStream_t stream);
// Chunked forwards with more carries than this fold them in the middle pass above (linear in
// the chunk count) instead of in every pass-2 CTA (quadratic).
constexpr int64_t kCarryScanMinCarries = 48;

struct BwdLaunch {
    const void* x;
    const void* delta;
    const float* A;
    const void* b;
    const void* c;
    const float* ckpt;   // (ceil(T/K), B, D, 16), slot 0 = h0
    const void* dy;
    const float* ghT;    // may be null
    float* gx;
    float* gdelta;
    float* gA;           // zeroed by the launcher
    float* gb;           // zeroed by the launcher
    float* gc;           // zeroed by the launcher
    float* gh0;
    int64_t B, T, D;
    int64_t K;           // checkpoint interval of ckpt, 1 <= K <= kMaxBwdK
    IO io;
    bool vec;
    int kd;              // channels per lane: 1 (32 channels per CTA) or 2 (64 per CTA)
    // chunk-parallel schedule (kd == 1 only): one CTA per (channel block, batch, chunk); the
    // adjoint entering each chunk comes from the carries of all later chunks
    bool tpar;
    float* carry_Z;      // [nck][B][D][16]: a_{cs} g_{cs} of chunk j with zero adjoint entering it
    float* carry_S;      // [nck][B][D]: sum of delta over chunk j
    // deterministic sums: partials instead of atomic adds, reduced in a fixed order afterwards
    bool det;
    float* part_gbc;     // [channel blocks][B][T][2][16]: per-CTA sums over d of gb (0) and gc (1)
    float* part_gA;      // [B * chunks][D][16]: per-CTA sums over t of gA (chunks = gridDim.z)
    // fused prologue / epilogue (the fused kernel variants only)
    bool softplus;       // delta holds raw values; gdelta is with respect to them
    const float* Dskip;  // (D) or null: the forward added Dskip[d] * x to y
    float* gDskip;       // (D), with Dskip: sum over b, t of dy * x (zeroed by the launcher)
    float* part_gD;      // deterministic: [B * chunks][D] partials of gDskip
};

// Deterministic backward: sums of the per-CTA partials in a fixed order into gb, gc and gA.
cudaError_t launch_bwd_reduce(const BwdLaunch& L, int64_t nblk, int64_t nz, cudaStream_t stream);

constexpr int64_t kMaxBwdK = 256;   // largest checkpoint interval the backward reads directly

cudaError_t launch_bwd_f32(const BwdLaunch& L, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const BwdLaunch& L, cudaStream_t stream);
cudaError_t launch_bwd_carry_f32(const BwdLaunch& L, cudaStream_t stream);
cudaError_t launch_bwd_carry_bf16(const BwdLaunch& L, cudaStream_t stream);

int device_sm_count();

// Schedule of the chunked forward (both passes use G lanes per chain; kd channels per lane).
// Two channels per lane whenever that leaves at least 4 pass-2 warps per SM, else one.
// Chosen by the library (chunk_len == 0): with two channels, chunks for about 21 resident
// pass-2 warps per SM but at least 128 steps; with one, chunks for about 14 warps per SM, at
// least 64 steps; two-channel chunks are at most 512 steps (with 8192 chains and 4096 steps, 6
// chunks of 704 steps took 254 us, 8 of 512 228 us). Measured on the 2048-chain workloads (after
// the carry fold's loads were batched): 4096 steps in 22 chunks at two channels 72.3 us, 8 at one
// 76.4 us (earlier rule); 1024 steps in 8 chunks at two channels 29.4 us, at one 32.4 us.
// Lanes per chain G: 2 lanes (8 states each, two channels per lane) from about 40 chains per SM
// as below, or with a given chunk length when the chunk passes still have about 12 warps per SM
// that way (the one-pass layout rule); else 4.
struct ChunkSchedule {
    int64_t Lc;
    int kd;
    int G;
};
inline ChunkSchedule chunk_schedule(int64_t T, int64_t chains, int64_t chunk_len, int64_t sms) {
    auto round32 = [](int64_t v) { return (v + 31) / 32 * 32; };
    auto kd_for = [&](int64_t Lc) { return chains * ((T + Lc - 1) / Lc) >= 64 * sms ? 2 : 1; };
    auto with_lanes = [&](int64_t Lc, int kd) {
        const bool two = kd == 2 && chains * ((T + Lc - 1) / Lc) >= 12 * 32 * sms;
        return ChunkSchedule{Lc, kd, two ? 2 : 4};
    };
    if (chunk_len > 0) return with_lanes(chunk_len, kd_for(chunk_len));
    const int64_t n2 = sms * 336 / chains > 2 ? sms * 336 / chains : 2;
    int64_t L2 = round32((T + n2 - 1) / n2);
    if (L2 < 128) L2 = 128;
    if (L2 > 512) L2 = 512;
    if (kd_for(L2) == 2) {
        // from about 40 chains per SM: 2 lanes per chain in chunks of 256 steps (4096 steps, bf16,
        // against 4 lanes in chunks of 512: 8192 chains 228 -> 216 us, 10240 285 -> 259 us, 12288
        // 335 -> 312 us; at 4096 chains 4 lanes stay ahead, 133 against 130-140 us)
        if (chains >= 40 * sms && T >= 512) return {256, 2, 2};
        return with_lanes(L2, 2);
    }
    const int64_t n1 = sms * 448 / (chains * 4) > 2 ? sms * 448 / (chains * 4) : 2;
    const int64_t L1 = round32((T + n1 - 1) / n1);
    return {L1 < 64 ? 64 : L1, 1, 4};
}

}  // namespace ssm
