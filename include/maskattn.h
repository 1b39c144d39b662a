/*
 * maskattn.h -- C ABI of libmaskattn: masked attention forward and backward
 * (GQA/MHA, BHSD, head dim 128, fp16 or bf16, fp32 accumulation) with a
 * per-head attention sink, for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operation (restated from the pages this library follows):
 *   - tilelang-ascend PR #1 "Add GQA Sink Backward BHSD", Summary: online
 *     softmax with an attention sink and a sliding-window mask; commit notes
 *     of the 2-kernel design: Phase0 Delta = sum(O*dO), a KV loop of five
 *     contractions + softmax + dS, Phase5 dSink.  The sink is one logit per
 *     head that joins only the softmax denominator (it has no value row).
 *   - cannbot-knowledge PR #174, BlockSparseAttentionGrad runbook, task
 *     features: a uint8 block mask [B,N,ceil(Sq/bx),ceil(Skv/by)] with bx and
 *     by chosen independently and not required to divide the sequence
 *     lengths; optimisations 1-2: the host only checks shapes and carves
 *     memory, the mask is transposed and compacted into select tables on the
 *     device; optimisation 3: dK/dV are written back contiguously, without
 *     atomics; precision notes: p = exp(s - lse), ds = p * (dp - delta), a row
 *     that sees no key gets zeros.
 *
 * With g = Hq / Hkv, query head h reads key/value head floor(h / g).
 * Visibility of key j to query i (0-based):
 *   ATTN_MASK_NONE     every j
 *   ATTN_MASK_CAUSAL   j <= i                        (requires Sq == Skv)
 *   ATTN_MASK_SLIDING  j <= i and i - j < window     (requires Sq == Skv)
 *   ATTN_MASK_BLOCK    block_mask[b, h, i / bx, j / by] != 0
 *
 * Memory: every tensor argument is a DEVICE pointer owned by the caller,
 * contiguous, 16-byte aligned.  q, o, dO, dq: [B,Hq,Sq,128]; k, v, dk, dv:
 * [B,Hkv,Skv,128], all of `dtype`; lse: float32 [B,Hq,Sq] (natural log);
 * sink, dsink: float32 [Hq]; block_mask: uint8 [B,Hq,ceil(Sq/bx),ceil(Skv/by)].
 * The library allocates no device memory: scratch comes from the caller's
 * workspace `ws` (size from attn_workspace_size, 256-byte aligned).
 * Limits: Sq, Skv <= 2^24 and B * Hq <= 65535.
 *
 * Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 * default stream), returns a status at once, and may be enqueued again on the
 * same stream with the same workspace.  Calls that share a workspace must not
 * overlap in time (use one stream, or one workspace per stream).
 *
 * Errors: arguments are checked on the host before anything is enqueued; on
 * an error nothing is enqueued and the outputs are left untouched.  Device
 * waits inside the kernels are bounded: a wait that runs out records
 * ATTN_ERR_TIMEOUT in the workspace status word, which attn_get_device_status
 * reads back; the outputs of such a call are undefined.  The limit is 2 s per
 * wait, or MASKATTN_WAIT_TIMEOUT_NS nanoseconds from the environment at the
 * time of the call.  Test hooks, off unless set in the environment at the time
 * of a call: MASKATTN_TEST_NO_LOADS=1 makes the kernels' loader warps issue
 * nothing, so the call's waits run out and it ends with ATTN_ERR_TIMEOUT;
 * MASKATTN_DKDV_SCHEDULE=tile or =units forces the per-tile or the persistent
 * form of the dK/dV kernel (otherwise chosen by the walk lengths; the results
 * are the same bit for bit).
 */
#ifndef MASKATTN_H_
#define MASKATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer, bad mask fields */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request the library does not implement (D != 128) */
  ATTN_ERR_WORKSPACE = 3,   /* ws_bytes smaller than attn_workspace_size() */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  ATTN_ERR_TIMEOUT = 5      /* a device-side wait ran out (read back by attn_get_device_status) */
} attn_status_t;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_SLIDING = 2, /* causal with a window of `window` keys including the diagonal */
  ATTN_MASK_BLOCK = 3
} attn_mask_kind_t;

/* Shapes of one call; tensors are contiguous BHSD.  flags: 0, or
 * ATTN_FLAG_COMPENSATED or ATTN_FLAG_SINGLE_PASS (not both). */
typedef struct {
  int B, Hq, Hkv, Sq, Skv, D;
  int dtype; /* attn_dtype_t */
  int flags; /* attn_flag_t bits */
} attn_shape_t;

/* ATTN_FLAG_COMPENSATED (attn_bwd): P and dS enter the 16-bit contractions
 * dV += P^T dO, dK += dS^T Q and dQ += dS K as a 16-bit high part plus a
 * 16-bit remainder (two contractions each), so they are rounded to about 22
 * bits instead of 11 (fp16) or 8 (bf16) before the fp32 accumulation --
 * the compensated ("hi + lo") mode for tighter tolerances.  It costs 1.3x
 * the tensor work and 1.1x to 1.35x the time.  attn_fwd ignores it. */
/* ATTN_FLAG_SINGLE_PASS (attn_bwd): the single-pass design of the backward.
 * The key-stationary kernel also computes, for every visible (key tile,
 * query sub-tile) step, that step's dq partial dS K in fp32 and stores it in
 * the workspace; a second kernel sums each query sub-tile's partials in
 * ascending key-tile order (deterministic) and rounds.  S and dP are then
 * computed once per tile instead of twice (the default split design computes
 * them again in its query-stationary dq kernel), at the price of 32 KB of
 * partials written and read per step: the workspace grows by 32 KB + 1 byte
 * per (query head, key tile, query sub-tile) step the key tiles can take at
 * the full lengths (all of them for block masks).  Same results up to
 * rounding order.  ATTN_ERR_UNSUPPORTED with ATTN_FLAG_COMPENSATED or the
 * packed layout.  attn_fwd ignores it (its workspace need is unchanged). */
typedef enum { ATTN_FLAG_COMPENSATED = 1, ATTN_FLAG_SINGLE_PASS = 2 } attn_flag_t;

/* Mask description.  window is read for ATTN_MASK_SLIDING only; bx, by and
 * block_mask for ATTN_MASK_BLOCK only (block_mask is a device pointer).
 *
 * Variable lengths: seqlen_q and seqlen_k, when not NULL, are device int32
 * arrays [B] of the valid query rows and keys of each batch element (values
 * are clamped to [0, Sq] and [0, Skv]); NULL means all rows / keys.  Rows
 * i >= seqlen_q[b] and keys j >= seqlen_k[b] are outside the problem: no pair
 * with either is visible (the mask rules count i and j from the start of the
 * sequence, as without lengths), such a row has O = 0 and LSE = +inf in the
 * forward, dQ = 0 and no part in dSink in the backward whatever finite values
 * q, O, dO and LSE hold there, and such a key has dK = dV = 0 whatever finite
 * values k and v hold there.  This is the variable-length
 * batch on the padded BHSD layout: each sequence starts at row 0 of its batch
 * element.  4-byte aligned.
 *
 * Packed variable lengths: cu_seqlens_q and cu_seqlens_k, when not NULL (both,
 * with seqlen_q and seqlen_k NULL), are device int32 arrays [B + 1] of
 * cumulative sequence offsets: sequence b owns tokens [cu_seqlens_q[b],
 * cu_seqlens_q[b + 1]) of q, o, dO and dq, which are then token-major
 * [total_q, Hq, 128] tensors, and tokens [cu_seqlens_k[b], cu_seqlens_k[b + 1])
 * of k, v, dk and dv, [total_k, Hkv, 128]; lse is float32 [Hq, total_q].
 * total_q and total_k (>= 1) are the token counts of those tensors, known to
 * the caller; Sq and Skv of the shape are the longest sequence lengths (they
 * size the workspace and the block mask, whose rows and columns count from
 * each sequence's start, as the causal and sliding-window rules do).  Offsets
 * are clamped to [0, total] and lengths to [0, Sq] / [0, Skv]; every write
 * stays inside the sequence's own tokens, and tokens no sequence owns are not
 * written.  4-byte aligned. */
typedef struct {
  int kind; /* attn_mask_kind_t */
  int window;
  int bx, by;
  const uint8_t* block_mask;
  const int* seqlen_q;     /* device [B] or NULL */
  const int* seqlen_k;     /* device [B] or NULL */
  const int* cu_seqlens_q; /* device [B + 1] or NULL: packed layout */
  const int* cu_seqlens_k; /* device [B + 1] or NULL */
  int total_q, total_k;    /* packed layout: tokens in the query / key tensors */
} attn_mask_desc_t;

/* Workspace bytes needed by attn_fwd and attn_bwd for this shape and mask.
 * Host only; never touches the GPU.  Errors: ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED (same checks as attn_bwd, pointers not required). */
attn_status_t attn_workspace_size(const attn_shape_t* shape, const attn_mask_desc_t* mask,
                                  size_t* bytes);

/* Forward: O = softmax_with_sink(scale * q k^T, masked) v, and
 * lse[b,h,i] = log(sum_j exp(scale*s_ij) + exp(sink_h)) over visible j.
 * sink may be NULL (no sink).  A row with no visible key and no sink gets
 * O = 0 and lse = +inf.  Outputs: o (dtype), lse (float32). */
attn_status_t attn_fwd(const attn_shape_t* shape, const void* q, const void* k, const void* v,
                       const float* sink, const attn_mask_desc_t* mask, float scale, void* o,
                       float* lse, void* ws, size_t ws_bytes, void* stream);

/* Backward from the forward's o and lse (taken as given):
 *   Delta_i = sum_d dO_id o_id;  P_ij = exp(scale*s_ij - lse_i);
 *   dS_ij = P_ij (dO_i . v_j - Delta_i);
 *   dq_i = scale sum_j dS_ij k_j;  dk_j = scale sum_{h in group} sum_i dS_ij q_i;
 *   dv_j = sum_{h in group} sum_i P_ij dO_i;
 *   dsink_h = - sum_b sum_i exp(sink_h - lse_i) Delta_i.
 * sink NULL means no sink; dsink is then not written and may be NULL.
 * Every element of dq, dk, dv (and dsink) is written.  Outputs dq, dk, dv
 * have `dtype` (fp32 accumulation, round to nearest even). */
attn_status_t attn_bwd(const attn_shape_t* shape, const void* q, const void* k, const void* v,
                       const void* o, const void* dO, const float* lse, const float* sink,
                       const attn_mask_desc_t* mask, float scale, void* dq, void* dk, void* dv,
                       float* dsink, void* ws, size_t ws_bytes, void* stream);

/* Backward for callers that cannot allocate device memory (operator or plugin
 * interfaces that receive no workspace, services that forbid allocation while
 * running).  The pages describe no such variant; this is an addition of this
 * library.  Same arguments and results as attn_bwd, without ws / ws_bytes:
 * the scratch lives in a fixed 32 MiB device array inside the library, held
 * on every GPU that loads it until the process exits.  The first call on a
 * device looks up that array's address (make that first call before any
 * stream capture on the device).  Errors: those of attn_bwd, and
 * ATTN_ERR_WORKSPACE when attn_workspace_size() for the shape exceeds 32 MiB.
 * All calls on a device share the array: calls whose GPU work overlaps in
 * time race on it and give wrong results, so order them on one stream.
 * `stream` must belong to the current device (ATTN_ERR_INVALID_ARG
 * otherwise).  The array's address is cached per device for the life of the
 * process: after cudaDeviceReset on a device this entry point must not be
 * used on it again.  A device wait that runs out is recorded in the array's
 * status word: read it with attn_noalloc_get_device_status. */
attn_status_t attn_bwd_noalloc(const attn_shape_t* shape, const void* q, const void* k,
                               const void* v, const void* o, const void* dO, const float* lse,
                               const float* sink, const attn_mask_desc_t* mask, float scale,
                               void* dq, void* dk, void* dv, float* dsink, void* stream);

/* Synchronizes `stream`, then reads the status word that the last call which
 * used `ws` left in the workspace: ATTN_OK, or ATTN_ERR_TIMEOUT when a device
 * wait ran out.  ATTN_ERR_CUDA if the synchronization itself fails. */
attn_status_t attn_get_device_status(const void* ws, void* stream);

/* Synchronizes `stream` (which must belong to the current device), then
 * reads the status word that the last attn_bwd_noalloc call on the current
 * device left in the library's scratch array: ATTN_OK or ATTN_ERR_TIMEOUT.
 * ATTN_ERR_INVALID_ARG for a stream of another device, ATTN_ERR_CUDA if the
 * synchronization or the read fails. */
attn_status_t attn_noalloc_get_device_status(void* stream);

/* Per-kernel timing, for diagnostics and benchmarks.  attn_profile_enable(1)
 * makes later attn_fwd / attn_bwd calls on this process bracket every kernel
 * they enqueue with CUDA events (created on first use, on the current device,
 * and kept until the process exits); attn_profile_enable(0) stops it.
 * attn_profile_read waits for the events of the most recent profiled call and
 * writes up to `capacity` kernel names (static strings) and elapsed times in
 * milliseconds, in launch order; *count receives the number of kernels.
 * Errors: ATTN_ERR_INVALID_ARG (null count, or names/ms null with capacity >
 * 0), ATTN_ERR_CUDA (event creation or synchronization failed). */
attn_status_t attn_profile_enable(int on);
attn_status_t attn_profile_read(const char** names, float* ms, int capacity, int* count);

/* Static string naming a status code ("ATTN_OK", ...). Never NULL. */
const char* attn_status_string(attn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MASKATTN_H_ */
