/*
 * attn_varlen.h -- C ABI of the GB300 (sm_103a) ragged GQA attention library.
 *
 * One fused call computes, for packed ragged (cu_seqlens) grouped-query
 * attention with Hq query heads sharing ONE key/value head of dimension 160
 * (the pages' case) or, more generally, Hkv key/value heads each shared by
 * Hq/Hkv consecutive query heads, the forward output and log-sum-exp and the
 * complete vector-Jacobian product (dq, dk, dv) for a given output cotangent
 * dout.
 *
 * Operation ("Noncausal Global Extreme-GQA Ragged Attention Full VJP",
 * sections "Hard Constraints" and "What You Have"):
 *   for sequence b with Lq = cu_q[b+1]-cu_q[b] queries and Lk = cu_k[b+1]-cu_k[b]
 *   keys, head h, local query i and key j:
 *     s   = (scale_multiplier / sqrt(head_dim)) * q[i,h,:] . k[j,g(h),:]
 *     t   = softcap * tanh(s / softcap)        (t = s when softcap <= 0)
 *     z   = t - alibi_slopes[b,h] * |i + Lk - Lq - j|
 *     z   = -inf where the causal/window mask forbids (i, j)
 *     lse = ln sum_j exp(z),  out[i,h,:] = sum_j exp(z - lse) v[j,g(h),:]
 *   with g(h) = h / (Hq / Hkv) (0 for the pages' Hkv = 1), and dq, dk, dv
 *   are the gradients of <dout, out> with respect to q, k, v; dk and dv of
 *   K/V head g are summed over every query head that reads it (same page,
 *   "Hard Constraints": all query heads share the single K/V head).  The
 *   pages fix only Hkv = 1; the consecutive grouping for Hkv > 1 is the
 *   usual grouped-query reading.
 * The softcap acts on the scaled dot product before ALiBi and masking.  A row
 * with no admissible key ("ragged flash attention gradient recompute",
 * section "Root causes addressed", empty rows) gets out = 0, lse = -inf and
 * contributes nothing to any gradient.
 *
 * Mask (the pages accept causal/window arguments without defining them; the
 * library reads them bottom-right aligned like the ALiBi offset): with
 * k0 = i + Lk - Lq, key j is admissible iff
 *   (window_left < 0 or j >= k0 - window_left) and
 *   (wr < 0 or j <= k0 + wr), where wr = 0 if causal else window_right.
 *
 * Layouts.  All strides are in ELEMENTS; the feature axis (head_dim values,
 * 160 in the pages' workload) is contiguous.  q, dout, out, dq are [total_q, Hq, head_dim] at
 *   base + token * tok_stride + head * head_stride + feature;
 * k, v, dk, dv are [total_k, Hkv, head_dim] at
 *   base + token * tok_stride + head * head_stride + feature
 * (the head stride is ignored when Hkv = 1).
 * Token and head strides may be non-dense (padded features, token steps).
 * lse is a dense fp32 [total_q, Hq] array.  cu_q, cu_k are int32 [B+1] with
 * cu[0] = 0, non-decreasing, cu[B] = total.  alibi_slopes is fp32 [B, Hq]
 * with the given batch stride and head stride 1, or NULL for no ALiBi.
 *
 * Ownership and execution.  Every pointer argument except the scalar
 * arguments is a DEVICE pointer owned by the caller (the host-buffer entry
 * point below takes host pointers instead, and creates two streams and a few
 * events per call); the library allocates no memory and keeps no pointer
 * after the call returns.  The call validates
 * its arguments on the host, enqueues its kernels on `stream` and returns
 * without synchronising.  Inputs are read-only; out, dq, dk, dv and lse are
 * fully overwritten (dk/dv rows of keys that no query attends get 0).  For a
 * fixed build, device and input, results are bitwise identical from call to
 * call: no reduction uses atomics.
 *
 * Errors.  Host-detectable problems return a negative attn_status before
 * anything is enqueued.  Problems only visible on the device (inconsistent
 * cu arrays, a bounded wait that ran out) are recorded in the device status
 * word: an int32 at `device_status` if non-NULL, else the first 4 bytes of
 * the workspace.  It is 0 after a clean call; otherwise it holds
 * ATTN_DEV_* bits and the kernels skip their remaining work.  Read it after
 * synchronising the stream.
 */
#ifndef ATTN_VARLEN_H
#define ATTN_VARLEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = -1,     /* a null pointer, negative size, bad cu/total pair,
                                Hkv < 1 or Hq not a multiple of Hkv */
  ATTN_ERR_UNSUPPORTED = -2, /* head_dim not 64, 128 or 160; B too large */
  ATTN_ERR_ALIGNMENT = -3,   /* base not 16-byte aligned, stride not a multiple of 8 */
  ATTN_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
  ATTN_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed */
  ATTN_ERR_DEVICE_STATUS = -6,
  ATTN_ERR_TIMEOUT = -7,
  ATTN_ERR_SCRATCH_LIMIT = -8 /* needs more than the no-allocation entry point's scratch */
} attn_status;

/* Bits of the device status word. */
#define ATTN_DEV_BAD_CU 0x1          /* cu arrays not monotone / not ending at total */
#define ATTN_DEV_TIMEOUT_FWD 0x2     /* a bounded wait in the forward kernel ran out */
#define ATTN_DEV_TIMEOUT_DKDV 0x4    /* ... in the dk/dv kernel */
#define ATTN_DEV_TIMEOUT_DQ 0x8      /* ... in the dq kernel */
#define ATTN_DEV_SMEM_ALIGN 0x10     /* dynamic shared memory base not 1024-byte aligned */
#define ATTN_DEV_MASK_SPACE 0x20     /* keep-mask buffer smaller than the lengths need */

/* Largest batch (number of sequences) accepted. */
#define ATTN_MAX_BATCH 16384
/* The pages' head dimension; 128 and 64 are accepted too. */
#define ATTN_HEAD_DIM 160

/* Bytes of device workspace a call with these sizes needs (256-byte aligned
 * base).  Holds the status word, the tile schedule and the fp32 row term
 * D = rowsum(dout * out) of the backward pass. */
size_t attn_varlen_fvjp_workspace_size(int B, int Hq, int64_t total_q, int64_t total_k);

/* Forward + full VJP, fused into one call on `stream` (a cudaStream_t; NULL
 * is the legacy default stream).  `dtype` is the element type of q, k, v,
 * dout, out, dq, dk, dv.  head_dim must be 160 (the pages' case), 128 or 64
 * (run on the same 160-feature tiles with the features past head_dim read
 * as zeros and never written), and Hq a multiple of Hkv.
 * Every base pointer of a 16-bit tensor must be 16-byte aligned and every
 * token/head stride a multiple of 8 elements (the tensors are staged by
 * TMA).  With Hkv > 1 each K/V head group runs as its own problem, one after
 * the other on `stream` (query heads g*Hq/Hkv .. (g+1)*Hq/Hkv - 1 with K/V
 * head g), so the call enqueues more kernels (attn_varlen_launch_count). */
attn_status attn_varlen_fvjp_fwd_bwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

/* The two halves of the fused call, for training loops that run the forward
 * pass and, later, the backward pass: the steps either side of the fused
 * call of the same page ("Noncausal Global Extreme-GQA Ragged Attention Full
 * VJP", "What You Have": the function returns out and the gradients; the
 * backward recomputes the softmax from the stored lse as in "ragged flash
 * attention gradient recompute", "Root causes addressed").
 *
 * attn_varlen_fwd writes out and lse only (same arguments, layouts and rules
 * as attn_varlen_fvjp_fwd_bwd without dout, dq, dk, dv).
 *
 * attn_varlen_bwd reads out and lse as written by attn_varlen_fwd (or the
 * fused call) for the same q, k, v, cu arrays, slopes, mask, softcap and
 * scale, and writes dq, dk, dv.  out and lse are inputs here and are not
 * modified.  The workspace is the one attn_varlen_fvjp_workspace_size sizes;
 * it need not be the one the forward used.  For the same inputs the three
 * calls give bitwise the same out, lse, dq, dk and dv: they run the same
 * kernels. */
attn_status attn_varlen_fwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

attn_status attn_varlen_bwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    const void *out, int64_t out_tok_stride, int64_t out_head_stride, const float *lse,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    void *workspace, size_t workspace_bytes, int32_t *device_status, void *stream);

/* A static description of an attn_status value. */
const char *attn_status_string(attn_status s);

/* Number of kernel launches one attn_varlen_fvjp_fwd_bwd call enqueues for
 * these sizes with one K/V head (for launch accounting by callers and
 * benchmarks). */
int attn_varlen_fvjp_launch_count(int B, int Hq, int64_t total_q, int64_t total_k);

/* The same for any entry point and K/V head count: mode 1 = attn_varlen_fwd,
 * 2 = attn_varlen_bwd, 3 = the fused call.  0 for an invalid mode or Hkv. */
int attn_varlen_launch_count(int mode, int B, int Hq, int Hkv, int64_t total_q,
                             int64_t total_k);

/* Timing hook: the next attn_varlen_fvjp_fwd_bwd call made by THIS host
 * thread records events[0] before its first kernel and events[i] after its
 * i-th kernel (i = 1..n-1; the five kernels are schedule, forward,
 * preprocess, dk/dv, dq), then forgets the events.  `events` holds
 * cudaEvent_t handles owned by the caller; n must be 6 (or 0 to cancel).
 * Returns ATTN_ERR_INVALID for any other n.  Used by benchmarks to time each
 * kernel on the launching stream.  A call with Hkv > 1 records nothing (and
 * still forgets the events). */
attn_status attn_varlen_fvjp_record_events(void *const *events, int n);

/* The fused, forward and backward calls with counter-based dropout on the
 * attention weights ("ragged flash attention gradient recompute", "Root
 * causes addressed": a splitmix64 hash of (seed, b, h, row, col), independent
 * of tiling, with a scalar or a per-row rate).  Arguments are those of
 * attn_varlen_fvjp_fwd_bwd / attn_varlen_fwd / attn_varlen_bwd plus, after
 * scale_multiplier: dropout_seed, dropout_rate (used when dropout_rates is
 * NULL) and dropout_rates (DEVICE fp32 [total_q]: one rate per query token,
 * shared by its heads, or NULL).
 *
 * Element (sequence b, query head h, local query i, local key j) is kept when
 * the 16-bit field j mod 4 (bits 16 (j mod 4) and up) of
 * splitmix64(splitmix64(seed ^ b) ^ (h << 48 | i << 24 | floor(j / 4))) is at
 * least T = (uint32)(rate * 2^16) (computed in fp32; 2^16, dropping
 * everything, when rate >= 1), and kept weights are scaled by 1 / (1 - rate):
 * one hash per four keys of a row.
 * out = sum_j P_ij keep_ij scale v_j with the undropped softmax P (lse is the
 * undropped one); the backward pass regenerates the same keep bits.  Local
 * positions must stay below 2^24 and head indices below 2^16.  Every head
 * dimension of the dropout-free calls (160, 128, 64) is accepted; a NaN rate is
 * ATTN_ERR_INVALID.  Results are bitwise repeatable for a fixed seed. */
attn_status attn_varlen_fvjp_fwd_bwd_dropout(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    uint64_t dropout_seed, float dropout_rate, const float *dropout_rates,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

attn_status attn_varlen_fwd_dropout(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    uint64_t dropout_seed, float dropout_rate, const float *dropout_rates,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

attn_status attn_varlen_bwd_dropout(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    uint64_t dropout_seed, float dropout_rate, const float *dropout_rates,
    const void *out, int64_t out_tok_stride, int64_t out_head_stride, const float *lse,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    void *workspace, size_t workspace_bytes, int32_t *device_status, void *stream);

/* The dropout calls with the keep bits STORED instead of regenerated: the
 * forward computes each element's keep bit from the hash above once and
 * writes it to `keep_mask`, and the backward kernels read it there instead of
 * hashing again.  The bits, and so every result, are bitwise those of the
 * calls above (the reading of the page is unchanged: a stored copy of the
 * same counter-based bits).  The pages regenerate the mask in the backward;
 * this variant trades device memory (one bit per admissible-tile element) for
 * the backward's hashing.
 *
 * Arguments: those of the matching call above plus, after dropout_rates,
 * `keep_mask` (DEVICE, 256-byte aligned, owned by the caller) and its size
 * `keep_mask_bytes`, at least attn_varlen_dropout_mask_bytes for the call's
 * lengths and heads.  attn_varlen_fwd_dropout_mask writes the mask,
 * attn_varlen_bwd_dropout_mask reads it (it must come from the forward of the
 * same inputs, seed and rates; the backward then uses the rates only for the
 * scale), and the fused call does both.  The mask's layout is private to the
 * library.  A NULL or misaligned keep_mask is ATTN_ERR_INVALID /
 * ATTN_ERR_ALIGNMENT; a buffer smaller than the lengths need (checked on the
 * device, where the lengths are) sets ATTN_DEV_MASK_SPACE in the device
 * status and the kernels then skip their work. */
attn_status attn_varlen_fvjp_fwd_bwd_dropout_mask(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    uint64_t dropout_seed, float dropout_rate, const float *dropout_rates,
    void *keep_mask, size_t keep_mask_bytes,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

attn_status attn_varlen_fwd_dropout_mask(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    uint64_t dropout_seed, float dropout_rate, const float *dropout_rates,
    void *keep_mask, size_t keep_mask_bytes,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

attn_status attn_varlen_bwd_dropout_mask(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    uint64_t dropout_seed, float dropout_rate, const float *dropout_rates,
    const void *keep_mask, size_t keep_mask_bytes,
    const void *out, int64_t out_tok_stride, int64_t out_head_stride, const float *lse,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    void *workspace, size_t workspace_bytes, int32_t *device_status, void *stream);

/* Bytes of keep mask the _mask calls need for these lengths (HOST cu_q,
 * cu_k of B + 1 entries each): a 256-byte-aligned header of 4 (B + 1) bytes,
 * then Hkv times 2 KB per (128-row query tile, 128-key tile) pair of every
 * sequence, that is about Hq * sum_b Lq_b * Lk_b / 8 bytes.  0 for invalid
 * arguments. */
size_t attn_varlen_dropout_mask_bytes(int B, const int32_t *cu_q, const int32_t *cu_k, int Hq,
                                      int Hkv);

/* Forward + full VJP with every input and output in HOST memory, for
 * callers whose data lives on the host (the transfers over the host link are
 * then part of the call).  The pages have no counterpart; it serves the
 * end-to-end path.
 *
 * The batch is cut into `chunks` runs of whole sequences, each of about its
 * share of the sum of Lq*Lk: equal shares, except that with three chunks or
 * more the first and the last take a quarter of the others' (their copies in
 * and out are the ones no computation overlaps).  Each chunk goes through one of up to four slots of the device
 * buffer: its inputs are copied in on one internal stream (once the slot's
 * previous chunk has been copied out), it computes on one of two internal
 * compute streams (chunks alternate between them, so one chunk's first
 * kernels overlap the last kernels of the one before), and its results are
 * copied back on another internal stream.  Sequences are independent, so
 * each sequence's out, lse, dq, dk, dv are bitwise those of
 * attn_varlen_fvjp_fwd_bwd on device copies of the inputs, whatever the
 * chunking.
 *
 * Arguments: those of attn_varlen_fvjp_fwd_bwd with HOST pointers for q, k,
 * v, dout, cu_q, cu_k, alibi_slopes (or NULL), out, dq, dk, dv and lse (same
 * shapes and stride rules; host memory should be page-locked for the copies
 * to run asynchronously), plus `device_buffer` (a DEVICE array of at least
 * attn_varlen_fvjp_host_buffer_size_for bytes, 256-byte aligned, owned by the
 * caller; its slots hold dense device copies of one chunk each and its
 * workspace) and `host_status`
 * (HOST, `chunks` int32 words: the device status word of each chunk, 0 when
 * clean; written when the stream reaches the end of the call).  The call
 * reads the host cu arrays before it returns (to cut the chunks); the other
 * host arrays are read and written asynchronously, so they must stay valid
 * until `stream` has passed the call.  Host rows are copied one token at a
 * time when their heads are dense (head stride = head_dim), else one
 * (token, head) row at a time; feature padding is neither read nor written.
 * Errors as for attn_varlen_fvjp_fwd_bwd; ATTN_ERR_WORKSPACE when the device
 * buffer is too small; ATTN_ERR_INVALID when chunks < 1.  An error found
 * after the first chunk was enqueued (a failed CUDA call) returns with the
 * caller's stream waiting for the work already enqueued: the output host
 * arrays may then hold the results of the earlier chunks, and host_status
 * is not written (its copy is enqueued last). */
attn_status attn_varlen_fvjp_fwd_bwd_host(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    float *lse, void *device_buffer, size_t device_buffer_bytes, int chunks,
    int32_t *host_status, void *stream);

/* The chunking attn_varlen_fvjp_fwd_bwd_host uses: writes the sequence
 * boundaries 0 = cuts[0] < cuts[1] < ... < cuts[n] = B of n <= chunks runs of
 * whole sequences (HOST cu arrays; sequence b weighs Lq*Lk + 1, run c has the
 * share s_c = 1/4 for the first and the last run when chunks >= 3, else 1,
 * and ends at the first sequence where the running weight reaches
 * (s_0 + ... + s_c) / (s_0 + ... + s_{chunks-1}) of the total) and returns n (0 for invalid arguments; 1 when B = 0, with
 * cuts = {0, 0}).  `cuts` holds chunks + 1 entries. */
int attn_varlen_host_chunks(int B, const int32_t *cu_q, const int32_t *cu_k, int chunks,
                            int32_t *cuts);

/* The sigmoid-gated variant ("Pairwise-Gated Attention Engine", "Why it is
 * hard"): each query-key pair also gets a gate from separate projections
 * q_gate [total_q, Hq, gate_dim] and k_gate [total_k, Hkv, gate_dim],
 *   G_ij = sigmoid(q_gate[i,h,:] . k_gate[j,g(h),:] / sqrt(gate_dim)),
 * which scales the normalised attention weight:
 *   out[i,h,:] = sum_j exp(z_ij - lse_ih) G_ij v[j,g(h),:],
 * with z = (scale_multiplier / sqrt(head_dim)) q.k - ALiBi, masked as in
 * the ungated call, and lse the ungated log-sum-exp (the gate sits outside
 * the normalisation).  The page's attention is the plain softmax: there is
 * no softcap argument (the logits are not capped) and no dropout.  The
 * backward pass writes dq, dk, dv and the gate gradients dq_gate
 * [total_q, Hq, gate_dim] and dk_gate [total_k, Hkv, gate_dim] (dk, dv and
 * dk_gate summed over the query heads of each K/V head).
 *
 * head_dim must be 64 or 128 and gate_dim a multiple of 8 up to 64
 * (ATTN_ERR_UNSUPPORTED otherwise); the gate tensors follow the layout and
 * alignment rules of q and k (16-byte base, strides multiples of 8
 * elements).  Other arguments, the workspace (attn_varlen_fvjp_workspace_size)
 * and the error behaviour are those of attn_varlen_fvjp_fwd_bwd; every
 * output, dk_gate rows of keys no query attends included, is fully
 * overwritten, and repeated calls are bitwise identical. */
attn_status attn_varlen_gated_fvjp_fwd_bwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int gate_dim,
    int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const void *q_gate, int64_t qg_tok_stride, int64_t qg_head_stride,
    const void *k_gate, int64_t kg_tok_stride, int64_t kg_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float scale_multiplier,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    void *dq_gate, int64_t dqg_tok_stride, int64_t dqg_head_stride,
    void *dk_gate, int64_t dkg_tok_stride, int64_t dkg_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

/* The forward half of the gated call: out and lse only. */
attn_status attn_varlen_gated_fwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int gate_dim,
    int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *q_gate, int64_t qg_tok_stride, int64_t qg_head_stride,
    const void *k_gate, int64_t kg_tok_stride, int64_t kg_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float scale_multiplier,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    float *lse, void *workspace, size_t workspace_bytes, int32_t *device_status,
    void *stream);

/* Shard plan of one batch over `nranks` processes (1..16), one GPU each.
 * Sequences are independent problems, so the batch shards by sequence with
 * no exchange of data.  Each sequence weighs Hq times its admissible
 * (query, key) pairs under the mask; a sequence weighing more than 1/nranks
 * of the batch is cut into k = min(nranks, ceil(weight / (total/nranks)))
 * parts by query head (one K/V head: heads [e*Hq/k, (e+1)*Hq/k)) or by
 * whole K/V head groups (Hkv > 1: at most Hkv parts), and every unit (a
 * whole sequence or a part) goes, heaviest first, to the least loaded rank
 * (lowest on ties), the parts of one sequence to different ranks.  With one
 * K/V head each part's call yields a partial dk/dv of the sequence's keys
 * (summed over the part's heads only); the rank holding part 0 adds the
 * parts in part order (attn_varlen_sum_partials).  Parts of Hkv > 1 cover
 * disjoint K/V heads and need no sum.  Partitioning follows the sequence
 * independence of "Noncausal Global Extreme-GQA Ragged Attention Full VJP",
 * "Hard Constraints" (each sequence attends only within itself); the pages
 * describe no multi-GPU split, so this plan is this library's own.
 *
 * cu_q, cu_k are HOST int32 [B+1] arrays.  Writes, for units u = 0..n-1 in
 * order of (sequence, first head), unit_seq[u], the head range
 * [unit_h0[u], unit_h1[u]) and unit_rank[u], and the work of each rank in
 * rank_work[nranks].  Returns n (at most B + (nranks - 1)^2, and max_units
 * must be at least n), or -1 for invalid arguments. */
int attn_varlen_shard_plan(int B, const int32_t *cu_q, const int32_t *cu_k, int Hq, int Hkv,
                           int causal, int window_left, int window_right, int nranks,
                           int max_units, int32_t *unit_seq, int32_t *unit_h0,
                           int32_t *unit_h1, int32_t *unit_rank, double *rank_work);

/* Fixed-order sum of partial key gradients (the exchange step of the shard
 * plan above): out[r, :] = part[0][r, :] + part[1][r, :] + ... in part order,
 * accumulated in fp32 and rounded once to `dtype`.  `parts` is a HOST array
 * of nparts (1..16) DEVICE pointers to [rows, d] 16-bit arrays with row
 * stride part_row_stride (elements); out has row stride out_row_stride.  d
 * and both strides must be multiples of 8 elements and every pointer 16-byte
 * aligned (ATTN_ERR_ALIGNMENT otherwise).  Asynchronous on `stream`; the
 * result is the same bits on every call. */
attn_status attn_varlen_sum_partials(attn_dtype dtype, int nparts, const void *const *parts,
                                     int64_t rows, int d, int64_t part_row_stride, void *out,
                                     int64_t out_row_stride, void *stream);

/* Bytes of device buffer attn_varlen_fvjp_fwd_bwd_host needs for these
 * lengths (HOST cu arrays): the status words, cu arrays and slopes, and
 * min(4, number of chunks) slots sized for the largest chunk -- about
 * min(4, chunks)/chunks of the batch's dense copies.  0 for invalid
 * arguments. */
size_t attn_varlen_fvjp_host_buffer_size_for(int B, const int32_t *cu_q, const int32_t *cu_k,
                                              int Hq, int Hkv, int head_dim, int chunks);

/* An upper bound of attn_varlen_fvjp_host_buffer_size_for over every length
 * split with these totals (each slot sized for the whole batch). */
size_t attn_varlen_fvjp_host_buffer_size(int B, int Hq, int Hkv, int head_dim, int64_t total_q,
                                          int64_t total_k, int chunks);

/* Size of the fixed device scratch array used by
 * attn_varlen_fvjp_fwd_bwd_noalloc (64 MiB). */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u << 20)

/* The same fused forward + VJP call for callers that cannot allocate device
 * memory -- for example a plugin inside a host framework that owns every
 * device allocation, or a latency-critical service that forbids allocator
 * calls (which can synchronise the device) while it serves.  The pages have
 * no counterpart; this is a deployment convenience.
 *
 * Arguments are those of attn_varlen_fvjp_fwd_bwd without the workspace: the
 * caller still passes every input and output.  Instead of a workspace the
 * call uses one device array of ATTN_NOALLOC_SCRATCH_BYTES compiled into the
 * library; every GPU that loads the library holds it until the process exits.
 * The call allocates nothing (no cudaMalloc, no allocating library routine).
 *
 * Limits and sharing:
 *  - The call needs A(16 + 12 * max(Hq, 2)) + A(4 * (5 * B + 2)) +
 *    A(4 * total_q * Hq) bytes of the array, A() rounding up to a multiple
 *    of 256 (status word and tile counters, the tile schedule, the fp32 D
 *    term): at most ATTN_NOALLOC_SCRATCH_BYTES, so total_q * Hq up to about
 *    16.7 million query rows.  Larger problems are rejected with
 *    ATTN_ERR_SCRATCH_LIMIT before anything is enqueued.
 *  - Every call on a device uses the same array, which keeps the last call's
 *    contents.  The call resets what must start at zero itself.  Calls whose
 *    work overlaps on the GPU (other streams, other host threads) race on the
 *    array and give wrong results; serialise them.
 *  - The current device must be the one that owns `stream` and every
 *    pointer: the array used is the current device's.
 *  - The first call on each device, and the first after that device's
 *    context was destroyed and created again (cudaDeviceReset), looks up the
 *    array's device address (cudaGetSymbolAddress) with that device current;
 *    make such a call before any stream capture.
 *  - With device_status NULL the status word is the first int32 of the
 *    array, which the caller cannot read; pass a device_status pointer to
 *    see device-side errors. */
attn_status attn_varlen_fvjp_fwd_bwd_noalloc(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void *q, int64_t q_tok_stride, int64_t q_head_stride,
    const void *k, int64_t k_tok_stride, int64_t k_head_stride,
    const void *v, int64_t v_tok_stride, int64_t v_head_stride,
    const void *dout, int64_t do_tok_stride, int64_t do_head_stride,
    const int32_t *cu_q, const int32_t *cu_k,
    const float *alibi_slopes, int64_t slopes_batch_stride,
    int causal, int window_left, int window_right, float softcap, float scale_multiplier,
    void *out, int64_t out_tok_stride, int64_t out_head_stride,
    void *dq, int64_t dq_tok_stride, int64_t dq_head_stride,
    void *dk, int64_t dk_tok_stride, int64_t dk_head_stride,
    void *dv, int64_t dv_tok_stride, int64_t dv_head_stride,
    float *lse, int32_t *device_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_VARLEN_H */
