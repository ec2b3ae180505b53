/*
 * ssm_scan.h: C ABI of libssm_scan.so, the selective diagonal state-space scan
 * on one GB300 GPU (sm_103a).
 *
 * The operation (page "pssa_kernels.py", NSC64/pssa-100m, module docstring and
 * `scan_reference`): for every batch b, channel d, state s and t = 0..T-1,
 *     a_t[s]    = exp(delta[b,t,d] * A[d,s])
 *     h_t[s]    = a_t[s] * h_{t-1}[s] + delta[b,t,d] * b[b,t,s] * x[b,t,d]
 *     y[b,t,d]  = sum_s h_t[s] * c[b,t,s]          (reads the updated state)
 *     hT[b,d,s] = h_{T-1}[s],   h_{-1} = h0[b,d,:]
 * The backward (same page, `scan_bwd`) is the reverse sweep for the loss
 * L = sum dy*y + sum ghT*hT; with g_t = dL/dh_t,
 *     g_{T-1} = dy_{T-1} c_{T-1} + ghT,   g_t = dy_t c_t + a_{t+1} g_{t+1},
 *     gx = delta * sum_s g b,   gdelta = sum_s (g a h_{t-1} A + g b x),
 *     gb[b,t,s] = sum_d g delta x,   gc[b,t,s] = sum_d dy h_t,
 *     gA[d,s] = sum_{b,t} g a h_{t-1} delta,   gh0 = a_0 g_0.
 * Checkpoints follow the chunk-boundary retention of the ruDNN page
 * ("src/kda/chunk.rs", `chunk_kda`): slot j holds the state entering step j*K.
 *
 * Layouts: every buffer is contiguous and row-major.
 *   x, delta, y, dy              (B, T, D)   io dtype
 *   gx, gdelta                   (B, T, D)   float32
 *   b, c                         (B, T, DS)  io dtype
 *   gb, gc                       (B, T, DS)  float32
 *   A, gA                        (D, DS)     float32
 *   h0, hT, ghT, gh0             (B, D, DS)  float32
 *   ckpt                         (ceil(T/K), B, D, DS) float32, slot j = h entering step j*K
 * io dtype is float32 or bf16 (selected by ssm_scan_desc.io). The state and
 * all gradients are float32 in both cases.
 *
 * Ownership: the caller owns every buffer. All data pointers are DEVICE
 * pointers on the current CUDA device and must be 16-byte aligned. The library
 * never allocates, frees or synchronises; it only enqueues work on `stream`
 * (a cudaStream_t passed as void*, NULL = the legacy default stream) and
 * returns without waiting. Inputs are never written. Outputs are fully
 * overwritten; the backward clears its own accumulation targets (gA, gb, gc).
 *
 * Errors: every argument is checked on the host before anything is enqueued;
 * a failing check returns a status and enqueues nothing. Not checked (the
 * caller's preconditions): A < 0, delta > 0, finite inputs, buffer sizes, and
 * that buffers do not overlap. Values outside the numeric preconditions give
 * unspecified but memory-safe results; buffers that are too small or overlap
 * are undefined behaviour (the backward, for one, uses its gx output as
 * scratch space before it writes the gradient there).
 *
 * Supported: DS == 16; B, T, D >= 0; B <= 65535; D <= 2^27; at most 65535
 * chunks of a chunked forward, ceil(T / chunk_len) (SSM_ERR_UNSUPPORTED beyond). T == 0 or B == 0 or D == 0
 * launches no kernel: hT <- h0 (zeros if h0 is NULL), gh0 <- ghT (zeros if
 * NULL), gA <- 0, as the ruDNN page's `chunk_kda` returns the initial state for
 * an empty sequence.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype of x, delta, b, c, y and dy */
typedef enum { SSM_IO_F32 = 0, SSM_IO_BF16 = 1 } ssm_io_dtype;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,  /* NULL required pointer, negative size, bad enum or flag, B > 65535 */
    SSM_ERR_UNSUPPORTED = 2,  /* DS != 16, D > 2^27, or more than 65535 forward chunks */
    SSM_ERR_MISALIGNED = 3,   /* a data pointer is not 16-byte aligned */
    SSM_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than the query returned */
    SSM_ERR_CUDA = 5,         /* a CUDA runtime call or a launch failed */
    SSM_ERR_TIMEOUT = 6       /* ssm_scan_fwd_lookback_status: a look-back wait ran out */
} ssm_status;

typedef struct {
    int64_t B, T, D, DS;
    int32_t io;             /* ssm_io_dtype */
    int32_t ckpt_interval;  /* K >= 0: the forward writes ceil(T/K) checkpoint slots when
                               K > 0; the backward reads them (see ssm_scan_bwd) */
    int32_t chunk_len;      /* forward schedule: 0 = chosen by the library; > 0 = chunked
                               two-pass scan with chunks of this many steps; < 0 = one
                               pass over T. Every schedule computes the same function. */
    int32_t flags;          /* SSM_SCAN_DETERMINISTIC | SSM_SCAN_DELTA_SOFTPLUS |
                               SSM_SCAN_LOOKBACK | SSM_SCAN_STEP_INPUTS_READY or 0;
                               other bits must be 0 */
} ssm_scan_desc;

/* ssm_scan_desc.flags: the backward sums gb, gc and gA from per-CTA partials in
 * the workspace in a fixed order instead of with atomic adds, so every output
 * is bitwise identical from run to run for the same desc, inputs and GPU
 * model. The forward and ssm_scan_step ignore the flag (they have no sums
 * across CTAs). */
#define SSM_SCAN_DETERMINISTIC 1

/* ssm_scan_desc.flags: delta holds raw pre-activation values and every entry
 * point scans with softplus(delta) = log(1 + exp(delta)) instead, computed in
 * float32 inside the kernels; the backward's gdelta is then with respect to
 * the raw values (gdelta_raw = gdelta * sigmoid(delta_raw)). This is the
 * activation the model on the POPCORNBENCH trace page ("FW-GLM-5-1__l2_p30",
 * its forward() op list) applies to its delta projection before the scan. */
#define SSM_SCAN_DELTA_SOFTPLUS 2

/* ssm_scan_desc.flags: when the forward's schedule is chunked (chunk_len > 0,
 * or chosen by the library for shapes with few (b, d) chains), run it as ONE
 * launch with decoupled look-back (Merrill and Garland, "Single-pass Parallel
 * Prefix Scan with Decoupled Look-back", 2016) instead of two: each chunk's CTA
 * first publishes its affine map h -> exp(A sum(delta)) h + S (chunk 0: its
 * end state from h0), then reads its predecessors' maps back to the nearest
 * published end state, publishes its own end state and rescans its chunk with
 * readout. CTAs take their order from a counter, so a CTA only ever waits for
 * CTAs that started before it. Every wait is bounded (about a second of
 * polling per CTA); a wait that runs out does not hang the GPU: the launch
 * finishes, that chunk's outputs are wrong, and ssm_scan_fwd_lookback_status
 * returns SSM_ERR_TIMEOUT. The workspace (ssm_scan_fwd_workspace_bytes with
 * this flag set) holds the maps, end states and flags; the call zeroes the
 * flags with cudaMemsetAsync before the launch. The one-pass schedule, the
 * backward, ssm_scan_fwd_noalloc and ssm_scan_step ignore the flag. */
#define SSM_SCAN_LOOKBACK 4

/* ssm_scan_desc.flags, ssm_scan_step only: the caller promises that the kernel
 * launched before this step on the stream writes none of x, delta, A, b, c
 * (for example another session's step, all sessions' inputs having been
 * computed earlier). The step then loads those five while that kernel is still
 * running and waits for it only before reading h. Without the flag every load
 * waits. Every other entry point ignores the flag. */
#define SSM_SCAN_STEP_INPUTS_READY 8

/* Bytes of the checkpoint buffer: ceil(T/K)*B*D*DS*4, 0 when K == 0.
 * Defined by: the chunk-boundary retention of the ruDNN page ("src/kda/chunk.rs",
 * `chunk_kda` with retained boundaries): one state per chunk of K steps, slot j
 * the state entering step j*K. */
size_t ssm_scan_ckpt_bytes(const ssm_scan_desc* desc);

/* Bytes of device scratch memory ssm_scan_fwd needs for this desc (0 when the
 * schedule needs none). The workspace holds the chunked scan's per-chunk
 * decay sums and partial states; with SSM_SCAN_LOOKBACK, every chunk's map,
 * end state and publication flag. Defined by: the state carried across chunks
 * of the sequence (pssa page, "pssa_kernels.py", module docstring: h0 in, hT
 * out; ruDNN `chunk_kda`, the state carried from chunk to chunk). */
size_t ssm_scan_fwd_workspace_bytes(const ssm_scan_desc* desc);

/* Bytes of device scratch memory ssm_scan_bwd needs for this desc when it is
 * called with ckpt == NULL: what ssm_scan_bwd_ckpt_workspace_bytes counts plus
 * the checkpoints it rebuilds (the ruDNN page's `chunk_kda_backward` needs the
 * retained chunk boundaries; without them they are recomputed first). */
size_t ssm_scan_bwd_workspace_bytes(const ssm_scan_desc* desc);

/* Bytes of device scratch memory for a backward call with the forward's
 * checkpoints; 0 for most shapes. It holds
 *  - with SSM_SCAN_DETERMINISTIC, the per-CTA partial sums of gb, gc and gA
 *    (required: a smaller workspace gives SSM_ERR_WORKSPACE);
 *  - for shapes with few (b, d) chains (one CTA per chain block would leave
 *    SMs idle) and at least two checkpoint chunks, the carries of the
 *    chunk-parallel backward: a carry pass computes, per chunk, the adjoint
 *    a_t g_t at the chunk's start with zero adjoint entering it, plus the
 *    chunk's delta sum; each chunk then runs on its own CTAs with the adjoint
 *    entering it folded from the later chunks (the adjoint recurrence is
 *    linear, as the state recurrence is for the chunked forward). Without
 *    SSM_SCAN_DETERMINISTIC these carries are optional: with less workspace
 *    the backward sweeps each chain in one CTA, computing the same function up
 *    to rounding. */
size_t ssm_scan_bwd_ckpt_workspace_bytes(const ssm_scan_desc* desc);

/* Forward scan: y, hT and (if K > 0 and ckpt != NULL) the checkpoints.
 * Defined by: the pssa page ("pssa_kernels.py"), `scan_reference` (the plain
 * loop: decay, injection, readout of the updated state) and `scan_fwd` (the
 * same recurrence with y and the final state stored); checkpoints as in
 * ssm_scan_ckpt_bytes.
 *   h0    may be NULL (zero initial state)
 *   hT    may be NULL (not written)
 *   ckpt  may be NULL (not written); ignored when K == 0
 *   workspace/workspace_bytes: at least ssm_scan_fwd_workspace_bytes(desc)
 *         (may be NULL when that is 0)
 * Chained calls with hT of one call passed as h0 of the next compute the same
 * function as one call over the concatenated sequence (up to rounding). */
ssm_status ssm_scan_fwd(const ssm_scan_desc* desc,
                        const void* x, const void* delta, const float* A,
                        const void* b, const void* c, const float* h0,
                        void* y, float* hT, float* ckpt,
                        void* workspace, size_t workspace_bytes, void* stream);

/* After a forward call with SSM_SCAN_LOOKBACK whose schedule was chunked
 * (the single-pass prefix scan with decoupled look-back of Merrill and Garland,
 * 2016, applied to the chunk maps; the pages have no counterpart of the status
 * query):
 * waits for `stream` (cudaStreamSynchronize) and reads the count of look-back
 * waits that ran out from `workspace` (the same workspace and desc as that
 * call). SSM_OK when none ran out, or when desc's schedule is not the
 * one-launch chunked scan (nothing waited); SSM_ERR_TIMEOUT otherwise (that
 * call's y, hT and checkpoints are then not valid); SSM_ERR_WORKSPACE /
 * SSM_ERR_MISALIGNED for a bad workspace; SSM_ERR_CUDA if the copy or the
 * synchronisation failed. The count is reset by the next forward call. */
ssm_status ssm_scan_fwd_lookback_status(const ssm_scan_desc* desc, const void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Backward scan: gx, gdelta, gA, gb, gc, gh0 (all float32) for
 * L = sum dy*y + sum ghT*hT.
 * Defined by: the pssa page, `scan_bwd` (the reverse sweep: adjoint carried
 * with the next step's decay, the per-step gradient terms, gb/gc/gA summed over
 * chains, gh0 = a_0 g_0) and `ScanFn` (inputs and outputs of the autograd
 * function; hT not differentiated there, ghT = NULL here); the states are
 * rematerialised from the checkpoints as the ruDNN page's `chunk_kda_backward`
 * rematerialises each chunk from its retained boundary state.
 *   ckpt  the checkpoints the forward wrote with the same desc (K > 0), or
 *         NULL: the backward then rebuilds them from h0 in the workspace
 *   h0    may be NULL (zero initial state); used only when ckpt is NULL
 *   ghT   may be NULL (hT not differentiated, as on the pssa page)
 *   workspace/workspace_bytes: with ckpt == NULL (or K outside 1..256) at
 *         least ssm_scan_bwd_workspace_bytes(desc), else SSM_ERR_WORKSPACE;
 *         with checkpoints, ssm_scan_bwd_ckpt_workspace_bytes(desc) (see
 *         there for what is optional); NULL or 16-byte aligned
 * gA, gb and gc are sums over many (b, d) chains accumulated with atomic adds,
 * so their last bits can differ from run to run. */
ssm_status ssm_scan_bwd(const ssm_scan_desc* desc,
                        const void* x, const void* delta, const float* A,
                        const void* b, const void* c, const float* h0,
                        const float* ckpt, const void* dy, const float* ghT,
                        float* gx, float* gdelta, float* gA, float* gb, float* gc,
                        float* gh0,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Defined by: the POPCORNBENCH trace page ("FW-GLM-5-1__l2_p30"), its model's
 * forward() op list and kernel (softplus on delta, y + x * D after the scan).
 * The forward with the trace page's skip connection fused into its readout:
 * y[b,t,d] = <h_t, c_t> + D_skip[d] * x[b,t,d] (its forward() op list, and the
 * skip its kernel adds before storing y). D_skip is (D) float32 or NULL (no
 * skip: then this is ssm_scan_fwd). Everything else as ssm_scan_fwd, including
 * SSM_SCAN_DELTA_SOFTPLUS. */
ssm_status ssm_scan_fwd_fused(const ssm_scan_desc* desc,
                              const void* x, const void* delta, const float* A,
                              const void* b, const void* c, const float* D_skip, const float* h0,
                              void* y, float* hT, float* ckpt,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Defined by: the chain rule through the trace page's skip and softplus (see
 * ssm_scan_fwd_fused) around the pssa page's `scan_bwd`.
 * The backward of ssm_scan_fwd_fused with the same D_skip: gx gets
 * + dy * D_skip[d] and gD_skip[d] = sum_{b,t} dy[b,t,d] * x[b,t,d] ((D)
 * float32, required when D_skip is not NULL; accumulated with atomic adds, or
 * in a fixed order under SSM_SCAN_DETERMINISTIC). Everything else as
 * ssm_scan_bwd. */
ssm_status ssm_scan_bwd_fused(const ssm_scan_desc* desc,
                              const void* x, const void* delta, const float* A,
                              const void* b, const void* c, const float* D_skip, const float* h0,
                              const float* ckpt, const void* dy, const float* ghT,
                              float* gx, float* gdelta, float* gA, float* gb, float* gc,
                              float* gh0, float* gD_skip,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Forward scan that allocates nothing and takes no workspace. The pages have
 * no counterpart of this call; it exists for callers that cannot allocate
 * device memory while they run: code hosted inside another runtime that owns
 * all device memory (an engine plugin, a replayed graph step), or services that
 * must not call cudaMalloc on the hot path because it synchronises the device
 * and can fail under memory pressure.
 *
 * It always uses the chunked two-pass schedule (chunk length desc->chunk_len
 * when > 0, else chosen by the library and doubled until the carries fit; one
 * chunk falls back to the one-pass scan, which needs no scratch) and keeps the
 * chunk carries in a fixed device array inside the library of
 * SSM_SCAN_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library
 * holds until the process exits. Carries take B*(nchunk-1)*D*68 bytes (each
 * part rounded up to 256); a caller's chunk length that needs more is rejected
 * with SSM_ERR_WORKSPACE before anything is enqueued.
 *
 * Each call looks up the array's device address in the CUDA context current on
 * the calling thread (cudaGetSymbolAddress, a host-side lookup that allocates
 * nothing): every context has its own copy of the array, so calls from another
 * context of the same device, or after a device reset, use that context's copy.
 * The first call in a context loads the library's device code there, so make
 * it before any stream capture. All calls in a context share the array: calls
 * that overlap on the GPU race on it, so the caller must order them (one
 * stream, or events).
 * Nothing in the array needs clearing: each call writes every entry it reads.
 * Arguments, layouts, results and other errors are those of ssm_scan_fwd. */
#define SSM_SCAN_NOALLOC_SCRATCH_BYTES (8u << 20)
ssm_status ssm_scan_fwd_noalloc(const ssm_scan_desc* desc,
                                const void* x, const void* delta, const float* A,
                                const void* b, const void* c, const float* h0,
                                void* y, float* hT, float* ckpt, void* stream);

/* Defined by: the pssa page's `scan_reference` over one step (T = 1) with the
 * state carried between calls, as the ruDNN page's fused recurrent decode
 * (`chunk_kda` with one token) advances its state one token per call.
 * One step of the scan for every (b, d) chain, the state updated in place:
 * the decode form of the recurrence (one token per call, the state carried
 * between calls, as the ruDNN page's fused recurrent decode does for KDA).
 *     h[b,d,s] <- exp(delta[b,d] A[d,s]) h[b,d,s] + delta[b,d] b[b,s] x[b,d]
 *     y[b,d]   <- sum_s h[b,d,s] c[b,s]
 * i.e. ssm_scan_fwd with T = 1 and hT written over h0. desc->T must be 1;
 * ckpt_interval and chunk_len are ignored.
 *   x, delta, y   (B, D)      io dtype
 *   b, c          (B, DS)     io dtype
 *   A             (D, DS)     float32
 *   h             (B, D, DS)  float32, read and overwritten (not NULL)
 * No workspace; B == 0 or D == 0 launches nothing. Errors as ssm_scan_fwd,
 * except that x, delta and y need only be aligned to their element size (A,
 * b, c and h: 16 bytes), so one step's rows of (B, T, D) tensors can be passed
 * as they are.
 * Steps are launched as programmatic dependents of the preceding kernel on the
 * stream: a step's CTAs may be scheduled while that kernel finishes, but every
 * load waits until it has completed and its writes are visible, so any input
 * may be the output of the preceding kernel (a projection, or the previous
 * step's h and y). With SSM_SCAN_STEP_INPUTS_READY in desc->flags only the load
 * of h waits (see there). */
ssm_status ssm_scan_step(const ssm_scan_desc* desc,
                         const void* x, const void* delta, const float* A,
                         const void* b, const void* c, float* h, void* y, void* stream);

/* Static description of a status code (the error results of the ruDNN page's
 * `validate` / `KdaError`, as C status codes). */
const char* ssm_status_str(ssm_status status);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
