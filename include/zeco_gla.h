/*
 * zeco_gla.h -- C ABI of the segmented (ZeCO-style) gated linear attention
 * operator for one NVIDIA GB300 (sm_103a).
 *
 * The operator (diagonal-decay GLA; ZeCO: Zero-Communication Overhead Sequence
 * Parallelism for Linear Attention, Approach and Limitations):
 *
 *     S_t = diag(alpha_t) S_{t-1} + k_t^T v_t,   alpha_t = exp(log_alpha_t),
 *     o_t = q_t S_t,                             S_{-1} = S0,  S_final = S_{T-1},
 *
 * with S in R^{dk x dv} per (batch, head) and the decay acting on the d_k rows
 * (Pith review of ZeCO, "What carries the argument": the All-Scan update scales
 * the state by the cumulative decay broadcast along d_v).
 *
 * It is evaluated the ZeCO way (Pith review of ZeCO, referee major comment 3:
 * the two-pass schedule of Algorithm 1; assumptions: Appendix A.1 linear
 * decomposition):
 *   1. the sequence is cut into P segments of L = T/P tokens; every segment
 *      computes its local state from zero (chunks of C tokens) and its
 *      cumulative decay gamma_p = prod_{t in p} alpha_t;
 *   2. a segment scan -- the All-Scan update S_in[p+1] = (gamma_p^T 1) .* S_in[p]
 *      + S_loc[p], run independently on K contiguous blocks of d_k rows
 *      (Pith review of ZeCO, "What carries the argument") -- gives every
 *      segment its incoming global state; the accumulated state is what is
 *      carried on (the pages' Algorithm 2 forwards the local state in one
 *      branch, which the review's major comment 4 identifies as a bug);
 *   3. every segment recomputes its chunks from S_in[p] and writes o (intra-
 *      chunk decay-masked attention plus the inter-chunk state term).
 * The backward keeps S_in from the forward, so it needs no forward re-scan
 * (Pith review of ZeCO, assumptions: Appendix A.4); the adjoint state runs a
 * reverse segment scan (the dKV pass of Linear Attention Sequence Parallelism,
 * summary).  P, K and C change the grouping only: results equal the token
 * recurrence up to rounding.
 *
 * Conventions (all entry points):
 *   - Tensors are contiguous, row-major: q, k, log_alpha [B,H,T,dk];
 *     v, o, d_o [B,H,T,dv]; gradients have the shape of their input.  They are
 *     in the I/O dtype (shape->dtype).  S0, S_final, dS_final, dS0 are fp32
 *     [B,H,dk,dv].  Arithmetic is fp32 throughout (bf16 inputs are widened;
 *     bf16 tensor-core products accumulate in fp32).
 *   - Every pointer is DEVICE memory owned by the caller and must be 16-byte
 *     aligned.  The library never allocates, never frees, never synchronises
 *     (except zeco_last_device_status, whose job it is) and never prints.
 *     Work is enqueued on `stream` (NULL: the legacy default stream) and is
 *     asynchronous; outputs are valid once the stream reaches that point.
 *     Calls that share `saved` or `workspace` must be ordered.
 *   - Return value: ZECO_OK (0) or a negative ZECO_ERR_* code; nothing is
 *     enqueued when argument checks fail.  ZECO_ERR_CUDA means a launch failed
 *     (the CUDA error is left for cudaGetLastError of the caller's choosing).
 *   - Supported shapes: B, H, T, P >= 1, T % P == 0, C in {16, 32, 64, 128}
 *     with (T/P) % C == 0, dk % K == 0, dk a multiple of 16 in [16, 256], dv a
 *     multiple of 32 in [32, 512], B*H <= 65,535 and B*H*P <= 67,108,863 (the
 *     grid limits of the kernels).  The chunked form factors the decay inside a
 *     chunk as exp(b_t) * exp(-b_s); this is exact in fp32 as long as the sum
 *     of log_alpha over any chunk stays above -80 (for every d_k row).
 */
#ifndef ZECO_GLA_H
#define ZECO_GLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, spelled without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *zeco_stream_t;

enum {
    ZECO_OK = 0,
    ZECO_ERR_ARG = -1,         /* null / misaligned pointer or invalid shape value */
    ZECO_ERR_UNSUPPORTED = -2, /* valid shape outside the supported set above */
    ZECO_ERR_WORKSPACE = -3,   /* ws_bytes smaller than zeco_gla_workspace_bytes() */
    ZECO_ERR_CUDA = -4,        /* a kernel launch failed */
    ZECO_ERR_TIMEOUT = -5      /* a bounded device wait gave up (zeco_check_device_status) */
};

typedef enum { ZECO_F32 = 0, ZECO_BF16 = 1 } zeco_dtype;

/* Kernel path.  AUTO picks the tcgen05 tensor-core kernels for bf16 shapes they
 * support and the fp32 SIMT kernels otherwise; SIMT and TC force one path
 * (TC on an unsupported shape returns ZECO_ERR_UNSUPPORTED).  The tensor-core
 * path takes bf16 shapes whose d_k and d_v are multiples of 64: with C = 64 and
 * d_k in {64, 128, 256} every step of the forward and backward runs on tensor
 * cores; otherwise (d_k = 192, or C = 16 or 32) the segment states do, and the
 * chunk sweeps run on CUDA cores.  A call with C = 128 that is not forced onto
 * the SIMT path is evaluated with C = 64 where that is what runs it (bf16; fp32
 * with d_k above 128, where a 128-token chunk does not fit the SIMT kernels):
 * results do not depend on C, and the decay range of a 128-token chunk implies
 * that of its halves (shorter chunks are kept as asked). */
typedef enum { ZECO_PATH_AUTO = 0, ZECO_PATH_SIMT = 1, ZECO_PATH_TC = 2 } zeco_path;

/* Form of the decay (the ZeCO pages study the diagonal, per-d_k-row decay of
 * gated linear attention and leave other linear-attention forms to future
 * work: ZeCO, Limitations; the LASP page's linear attention has none).
 *   DIAG:   log_alpha [B,H,T,dk]; dlog_alpha [B,H,T,dk].
 *   SCALAR: one log-decay per token for all d_k rows (RetNet / Lightning
 *           style); log_alpha [B,H,T], dlog_alpha [B,H,T] (the sum over d_k
 *           of the per-row gradient).
 *   NONE:   alpha = 1 (plain causal linear attention); log_alpha and
 *           dlog_alpha are not used and may be NULL.
 * On the tensor-core path with C = 64 the kernels that read the log-decay
 * have each form built in: SCALAR is read once per token and its gradient is
 * summed from fp32 partials over blocks of 32 d_k rows; NONE reads no decay
 * and skips the dlog_alpha work.  Elsewhere SCALAR and NONE run the DIAG
 * kernels on a log-decay broadcast to [B,H,T,dk] in the workspace (and,
 * backward, a [B,H,T,dk] gradient that SCALAR reduces over d_k). */
typedef enum { ZECO_DECAY_DIAG = 0, ZECO_DECAY_SCALAR = 1, ZECO_DECAY_NONE = 2 } zeco_decay;

typedef struct zeco_shape {
    int64_t B, H, T; /* batch, heads, tokens per sequence */
    int64_t dk, dv;  /* key/query width and value width (state is dk x dv) */
    int32_t P;       /* segments per sequence (ZeCO's devices; here all on one GPU) */
    int32_t K;       /* d_k blocks of the segment scan */
    int32_t C;       /* chunk length inside a segment */
    int32_t dtype;   /* zeco_dtype of q, k, v, log_alpha, o and all their gradients */
    int32_t path;    /* zeco_path */
    int32_t decay;   /* zeco_decay (0 = DIAG, the default of a zeroed struct) */
} zeco_shape;

/*
 * Number of segments the library evaluates on one GPU for this shape (or a
 * negative ZECO_ERR_* code).  The segmented decomposition is exact for any
 * split of the sequence (ZeCO two-pass operator: the local states plus the
 * segment scan reproduce the recurrence), so when B*H*P gives the chunk sweeps
 * fewer CTAs than one wave of the GPU (152), each of the P segments is split
 * further into 2^m equal sub-segments of at least 4 chunks (m <= 6): config-2
 * shapes with P = 1 run as 16 segments.  Results differ only by rounding.
 * Below, "P_eff" is this number.
 */
int64_t zeco_gla_segments(const zeco_shape *shape);

/*
 * Bytes of the `saved` buffer written by zeco_gla_fwd and read by
 * zeco_gla_bwd: the incoming global state of every segment, S_in
 * [B,H,P_eff+1,dk,dv] fp32 (S_in[0] = S0, S_in[P_eff] = S_final), then the
 * segment decays gamma [B,H,P_eff,dk] fp32.  When the shape resolves to the
 * tensor-core path with its decay pass (d_k in {64, 128, 256}, d_v a multiple
 * of 64, C = 64), `saved` also keeps the operands the forward computes once
 * and the backward reads again instead of recomputing them: the
 * decay-weighted Q~ = q .* e^{b} and K~ = k .* e^{-b} [B,H,T,dk] bf16 (Pith
 * review of ZeCO, minor comment 4; b the cumulative log-decay from the chunk
 * start), e^{b_last} of every 64-token chunk [B,H,T/64,dk] fp32 and the masked
 * intra-chunk scores A = Q~ K~^T [B,H,T,64] bf16 (row t holds its chunk's 64
 * scores).  The size depends on the resolved path, so the forward and the
 * backward must be given the same shape, path included.  Returns 0 for an
 * invalid or unsupported shape.
 */
size_t zeco_gla_saved_bytes(const zeco_shape *shape);

/*
 * Bytes of scratch memory the forward (bwd = 0) or backward (bwd = 1) needs,
 * for the path the shape resolves to (shape->path, see zeco_gla_resolve_path).
 * The backward holds the adjoint of every segment's incoming state
 * [B,H,P_eff+1,dk,dv] fp32, one dlog_alpha carry row per segment [B,H,P_eff,dk] fp32,
 * and q .* dq in fp32 [B,H,T,dk] (dlog_alpha is a long suffix sum of
 * q .* dq - k .* dk that cancels heavily, so its terms are kept in fp32).
 * On the tensor-core path the backward also holds the masked gradient of the
 * intra-chunk scores dA = do v^T [B,H,T,64] bf16; where the dq/dk step runs on
 * CUDA cores (the SIMT path, and the tensor-core path's shapes whose sweeps run
 * there: d_k = 192, C = 16 or 32) it holds dA [B,H,T,C] fp32 instead.  Where the kernels read the SCALAR / NONE decay forms in their own
 * layout (see zeco_decay), SCALAR's
 * backward adds the fp32 partial sums of its gradient [dk/32][B,H,T] and NONE
 * adds nothing; elsewhere both forms add the log-decay broadcast to
 * [B,H,T,dk] (both directions) and its per-row gradient (backward).  Returns
 * 0 when no scratch is needed or the shape is invalid or unsupported.
 */
size_t zeco_gla_workspace_bytes(const zeco_shape *shape, int bwd);

/*
 * Forward: writes o, S_final (skipped when NULL) and `saved`.
 *   S0 == NULL means a zero initial state.
 *   saved: zeco_gla_saved_bytes(shape) bytes, kept unchanged until the matching
 *          zeco_gla_bwd has run.
 *   workspace / ws_bytes: at least zeco_gla_workspace_bytes(shape, 0) bytes,
 *          16-byte aligned and overwritten (may be NULL when that is 0);
 *          ZECO_ERR_WORKSPACE when ws_bytes is smaller, ZECO_ERR_ARG when a
 *          needed workspace is NULL or misaligned.
 */
int zeco_gla_fwd(const zeco_shape *shape, const void *q, const void *k, const void *v,
                 const void *log_alpha, const float *S0, void *o, float *S_final, void *saved,
                 void *workspace, size_t ws_bytes, zeco_stream_t stream);

/*
 * Backward of the loss L(o, S_final) given d_o = dL/do and dS_final = dL/dS_final
 * (NULL: zero).  Writes every element of dq, dk, dv, dlog_alpha and, when not
 * NULL, dS0 = dL/dS0.  q, k, v, log_alpha must be the forward's inputs and
 * `saved` the buffer that forward wrote (the global state held since the
 * forward: Pith review of ZeCO, assumptions: Appendix A.4).  workspace needs
 * zeco_gla_workspace_bytes(shape, 1) bytes and is overwritten.
 */
int zeco_gla_bwd(const zeco_shape *shape, const void *q, const void *k, const void *v,
                 const void *log_alpha, const void *saved, const void *d_o,
                 const float *dS_final, void *dq, void *dk, void *dv, void *dlog_alpha,
                 float *dS0, void *workspace, size_t ws_bytes, zeco_stream_t stream);

/*
 * Backward without a caller-provided workspace (the ZeCO pages have no
 * counterpart: this exists for callers that cannot allocate device memory --
 * code that runs where cudaMalloc is unavailable or forbidden, or inside a
 * host framework that owns all device memory and passes in only the tensors).
 * Same arguments, results and return codes as zeco_gla_bwd, minus workspace
 * and ws_bytes: the scratch is a fixed array of ZECO_NOALLOC_MAX_WS_BYTES in
 * the library's own device memory, which every GPU that loads the library
 * holds until the process exits.  Nothing is allocated or freed by the call.
 *   - Shapes needing more scratch than that (zeco_gla_workspace_bytes(shape, 1)
 *     > ZECO_NOALLOC_MAX_WS_BYTES) return ZECO_ERR_WORKSPACE, after the same
 *     shape and pointer checks as zeco_gla_bwd.
 *   - All calls on one GPU share the array: calls whose GPU work could overlap
 *     (other streams, other host threads) race on it and must be ordered by
 *     the caller.  The array keeps the last call's contents; the backward
 *     writes every scratch byte before reading it.
 *   - The first call on each device looks up the array's device address with
 *     that device current and caches it for the life of the process: make that
 *     first call before any stream capture on the device.  A cudaDeviceReset
 *     frees the array with the rest of the device's memory and leaves the
 *     cached address stale: do not call this entry point on a device after
 *     resetting it in the same process.
 */
#define ZECO_NOALLOC_MAX_WS_BYTES (32u << 20)
int zeco_gla_bwd_noalloc(const zeco_shape *shape, const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *saved, const void *d_o,
                         const float *dS_final, void *dq, void *dk, void *dv,
                         void *dlog_alpha, float *dS0, zeco_stream_t stream);

/*
 * Every wait of the tensor-core kernels on an mbarrier (a copy or an MMA group
 * to complete, a peer CTA's partial sums) gives up after 2 seconds (device
 * %globaltimer) instead of hanging the GPU.  The first wait of a CTA that gives
 * up sets a device flag and an abort word of that CTA: every other wait of the
 * CTA then returns at once, it issues no further copies, MMAs, remote stores
 * or remote arrives, waits (bounded again) for the copies and MMAs it has in
 * flight, frees its tensor memory and exits.  A wait that can never complete
 * therefore costs each CTA that meets it about one time limit.  The outputs of
 * that call are not valid.
 *
 * zeco_check_device_status reads and clears the flags of the current device:
 * ZECO_OK when no wait gave up since the last check, ZECO_ERR_TIMEOUT when one
 * did, ZECO_ERR_CUDA when the flags cannot be read.  The flags are per device,
 * not per stream or per call: a check reports (and clears) a give-up of any
 * call on any stream of this device since the previous check, so two host
 * threads that check the same device at once can clear each other's reports.
 * It copies from device memory and synchronises nothing itself: call it after
 * the streams of the calls it should cover have been synchronised.
 */
int zeco_check_device_status(void);

/*
 * Checked mode: synchronises `stream` (so every call enqueued on it so far has
 * finished), then reads and clears the bounded-wait flags of the current device
 * as zeco_check_device_status does (same codes; ZECO_ERR_CUDA also when the
 * synchronisation fails).  The only entry point that synchronises.  The flags
 * are per device, so a give-up in a call on another stream of the device that
 * finished before the read is reported too.
 */
int zeco_last_device_status(zeco_stream_t stream);

/*
 * Diagnostic of the bounded waits above (the ZeCO pages have no counterpart):
 * launches on `stream` one CTA of four warps whose threads each wait 64 times
 * on mbarriers that can never complete.  The first wait gives up after its
 * time limit (2 s), the CTA's other waits then return at once, the kernel
 * records the timeout and returns: it ends after about one time limit, the
 * next zeco_check_device_status() reports ZECO_ERR_TIMEOUT and the CUDA
 * context stays usable.  Returns ZECO_ERR_CUDA if the launch fails.
 */
int zeco_selftest_bounded_wait(zeco_stream_t stream);

/* Static message for an error code (never NULL). */
const char *zeco_strerror(int code);

/*
 * Optional per-kernel timing (measurement aid; not part of the method).
 * After zeco_set_profile_events(events, n) with n > 0, every zeco_gla_fwd /
 * zeco_gla_bwd call made on this host thread records, for its i-th kernel
 * counted from the set call, events[2i] right before the launch and
 * events[2i + 1] right after it, both on the stream the kernel runs on (the
 * caller's, or one of the auxiliary streams of zeco_set_overlap), until the n events
 * are used; n = 0 (or events = NULL) switches it off.  So the elapsed time from
 * events[2i] to events[2i + 1] is kernel i's duration, and intervals of kernels
 * on the two streams can be compared on one timeline.  `events` are
 * cudaEvent_t handles created (and later destroyed) by the caller.  The calls
 * return ZECO_OK.  zeco_profile_event_count() gives the number of events
 * recorded so far (two per kernel) and zeco_profile_kernel_name(i) the name of
 * kernel i (NULL when i is out of range).
 */
int zeco_set_profile_events(void *const *events, int n);
int zeco_profile_event_count(void);
const char *zeco_profile_kernel_name(int i);

/*
 * Schedule of the work beside the segment scan.  The pages' central claim is
 * that the exchange of segment states (the All-Scan) hides behind work that
 * does not need it (ZeCO, Pith review, "What carries the argument"; Algorithm 1
 * runs the All-Scan and the intra-chunk diagonal attention on two streams,
 * Eq. 11).  On the tensor-core path the passes that build the intra-chunk
 * scores A (forward) and their gradient dA (backward) do not depend on the
 * segment scan.
 *   mode 1: A and dA run on an auxiliary stream as soon as their inputs
 *     exist, concurrently with the segment-state pass and the scan (and,
 *     backward, the dv sweep);
 *   mode 2 (the pages' schedule): the segment scan (forward and reverse) runs
 *     on the auxiliary stream, concurrently with the A (dA) pass on `stream`;
 *   mode 3 (forward; the backward as mode 1): pass 2 of each of up to 8 blocks of
 *     segments starts as soon as the scan has produced that block's incoming
 *     states -- the scan runs block by block on `stream`, pass 2 of each block
 *     on the auxiliary stream after the A pass and after its block's scan;
 *   mode 4 (ZECO_OVERLAP_DEFAULT): mode 1, and in the backward the dq/dk sweeps
 *     run on a second auxiliary stream created at the device's highest stream
 *     priority while the dv sweep runs on `stream`: the two do not depend on
 *     each other, and the dv sweep's CTAs take the SMs that the last waves of
 *     the dq/dk sweeps leave idle.  Shapes whose segments hold fewer than 4
 *     chunks run as mode 0 under this setting (their kernels are bound by the
 *     segment-state traffic, and concurrent streams only contend);
 *   mode 0: everything on `stream`.
 * The call forks from and joins back into its `stream` with events, so all its
 * work stays ordered on `stream` (a zeco_gla_fwd + zeco_gla_bwd pair captured on
 * one stream, after one eager call has created the auxiliary streams, replays as
 * a CUDA graph with the eager results; tested).  Results are identical in every
 * mode.  The
 * auxiliary streams and eleven events are created on the first such call of
 * each host thread on each device and destroyed when the thread exits.
 * Process-wide; returns ZECO_OK, or ZECO_ERR_ARG for a mode outside 0..4.
 */
#define ZECO_OVERLAP_DEFAULT 4
int zeco_set_overlap(int mode);

/* The path zeco_gla_fwd / zeco_gla_bwd would run for this shape
 * (ZECO_PATH_SIMT or ZECO_PATH_TC), or a negative ZECO_ERR_* code. */
int zeco_gla_resolve_path(const zeco_shape *shape);

#ifdef __cplusplus
}
#endif

#endif /* ZECO_GLA_H */
