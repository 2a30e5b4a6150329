/*
 * ring_attn.h -- C ABI of the GB300 (sm_103a) exact ring-attention library
 * (libringattn.so).
 *
 * The method ("Training Long-Context Models Without OOM: Ring Attention",
 * section "Ring Attention Demystified", steps 1-5; "Context Parallelism"
 * guide, section 2 "Ring Attention" / "How It Works"): a sequence of S tokens
 * is split into P equal contiguous chunks of C = S / P tokens.  Query chunk i
 * meets KV chunk j = (i - t) mod P at ring step t = 0 .. P-1 (step 0 is its
 * own chunk; every later step receives the left neighbour's K and V).  Each
 * step's partial attention is folded into running softmax statistics (row
 * maximum and sum of exponentials), so after P - 1 rotations every query has
 * attended to the whole sequence and the result is exactly unchunked
 * attention:
 *     s_rc  = scale * <q_r, k_c>
 *     LSE_r = ln sum_{c in A_r} exp(s_rc)          (natural log)
 *     O_r   = sum_{c in A_r} exp(s_rc - LSE_r) v_c
 * with A_r = { c <= r } when causal, else all keys.  Causal masking is not
 * on the pages; the reading used is global-position masking, which skips
 * chunks j > i and masks key > query inside chunk i.  On one GPU the P ranks
 * are chunks and the rotation is double-buffered on-chip staging of the next
 * K/V tile.
 *
 * Conventions for every entry point:
 *   - Tensors are contiguous, row-major [B, H, S, d], except where an
 *     entry point takes stride arguments (the *_strided calls); LSE and
 *     other per-row vectors are always contiguous [B, H, S].  ra_bf16 holds
 *     raw bfloat16 bits.
 *   - All tensor pointers are DEVICE pointers, 16-byte aligned, owned by the
 *     caller.  The library allocates no device memory per call; it keeps one
 *     4-byte status word per device (static device storage).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream; nothing synchronizes except
 *     ring_attn_check_status.
 *   - Arguments are validated before any launch; a bad argument returns
 *     RA_ERR_INVALID_ARG, a valid but unsupported shape RA_ERR_UNSUPPORTED,
 *     a failed launch RA_ERR_CUDA (see ring_attn_last_error).  Nothing is
 *     launched when an error is returned.
 *   - Shapes with B, H or S equal to 0 are accepted and launch nothing.
 *   - Every wait inside the kernels is bounded in time; a wait that runs out
 *     ends the kernel early and sets the device status word, which
 *     ring_attn_check_status reports as RA_ERR_DEVICE_TIMEOUT.
 */
#ifndef RING_ATTN_H
#define RING_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ra_bf16;

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = -1,
    RA_ERR_UNSUPPORTED = -2,
    RA_ERR_CUDA = -3,
    RA_ERR_DEVICE_TIMEOUT = -4
} ra_status;

/*
 * Forward pass of exact ring attention.
 *   q, k, v  [B, H, S, d] bf16 inputs (read only).
 *   o        [B, H, S, d] bf16 output: O_r rounded to nearest even.
 *   lse      [B, H, S] fp32 output: LSE_r (natural log), kept for the
 *            backward pass.
 *   P        number of ring chunks, P >= 1 and S % P == 0 (the pages split
 *            the sequence "equally"; an unequal split is RA_ERR_INVALID_ARG).
 *   causal   0 or 1.
 *   scale    finite softmax scale (typically 1/sqrt(d)).
 *   d        64 or 128 (other values: RA_ERR_UNSUPPORTED).
 * q, k, v must not alias o or lse.  Chunk lengths need not be multiples of
 * the 128-row tile: ragged tails are masked.
 */
int ring_attn_fwd(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, ra_bf16 *o, float *lse,
                  int B, int H, int S, int d, int P, int causal, float scale, void *stream);

/*
 * Grouped-query forward: H query heads share H_kv key/value heads, query
 * head h reading key/value head h / (H / H_kv) -- the case the pages single
 * out, where ring attention does not depend on the head count ("Training
 * Long-Context Models Without OOM: Ring Attention", section "Ring Attention
 * vs. DeepSpeed Ulysses (All-to-All)").  q, o are [B, H, S, d]; k, v are
 * [B, H_kv, S, d]; lse is [B, H, S].  H_kv >= 1 and H % H_kv == 0, else
 * RA_ERR_INVALID_ARG.  Everything else as ring_attn_fwd, which is this call
 * with H_kv = H.
 */
int ring_attn_fwd_gqa(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, ra_bf16 *o, float *lse,
                      int B, int H, int H_kv, int S, int d, int P, int causal, float scale,
                      void *stream);

/*
 * Bytes of device workspace ring_attn_fwd_f32 needs: bf16 copies of q
 * ([B, H, S, d]) and of k and v ([B, H_kv, S, d]), each 256-byte aligned.
 * 0 for empty or invalid shapes.
 */
size_t ring_attn_fwd_f32_workspace_size(int B, int H, int H_kv, int S, int d);

/*
 * Forward pass from fp32 inputs (the same method as ring_attn_fwd_gqa;
 * H_kv = H for plain multi-head attention).
 *   q        [B, H, S, d] fp32; k, v [B, H_kv, S, d] fp32; contiguous.
 *   o        [B, H, S, d] fp32 output: O_r normalized, not rounded to bf16.
 *   lse      [B, H, S] fp32 output (natural log).
 *   workspace, workspace_bytes  caller-owned device memory of at least
 *            ring_attn_fwd_f32_workspace_size(B, H, H_kv, S, d) bytes,
 *            256-byte aligned; it receives the bf16 copies of the inputs.
 * The inputs are rounded to bf16 (round to nearest even) on the GPU and
 * multiplied on the bf16 tensor cores with fp32 accumulation, so the result
 * equals ring_attn_fwd_gqa on the rounded inputs except that O skips the
 * final bf16 rounding.  o may alias q (q is read before o is written) but
 * not k or v.  Other arguments and errors as ring_attn_fwd.
 */
int ring_attn_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse, int B,
                      int H, int H_kv, int S, int d, int P, int causal, float scale, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * Forward pass over tensors in any row layout ("Training Long-Context Models
 * Without OOM: Ring Attention", section "Ring Attention Demystified", step 1
 * splits the sequence of tokens into equal chunks but fixes no memory
 * layout; sequence-major [B, S, H, d] is the common one in training code).
 * Computes exactly what ring_attn_fwd_gqa computes (H_kv = H for plain
 * multi-head attention).
 *   X_strides  three element strides {batch, head, position} of tensor X:
 *              row (b, h, s) of X starts at element
 *              b * X_strides[0] + h * X_strides[1] + s * X_strides[2], and
 *              its d elements are contiguous.  NULL means the contiguous
 *              [B, heads, S, d] layout.  [B, S, H, d] storage is
 *              {S * H * d, d, H * d}.
 * Every stride of a dimension with more than one index must be a positive
 * multiple of 8 elements (16 bytes) below 2^35, else RA_ERR_INVALID_ARG.
 * lse stays contiguous [B, H, S].  The rows of o must not overlap one
 * another or any input.  The results are bit-identical to the contiguous
 * entry points on the same values: the layout changes only where rows are
 * read and written.
 */
int ring_attn_fwd_strided(const ra_bf16 *q, const long long *q_strides, const ra_bf16 *k,
                          const long long *k_strides, const ra_bf16 *v, const long long *v_strides,
                          ra_bf16 *o, const long long *o_strides, float *lse, int B, int H, int H_kv,
                          int S, int d, int P, int causal, float scale, void *stream);

/*
 * Bytes of device workspace ring_attn_fwd_ulysses_emulated needs: the P
 * ranks' receive buffers for q and O ([B, H, S, d] bf16 in all), k and v
 * ([B, H_kv, S, d] bf16) and LSE ([B, H, S] fp32), each 256-byte aligned.
 * 0 for empty or invalid shapes.
 */
size_t ring_attn_fwd_ulysses_workspace_size(int B, int H, int H_kv, int S, int d);

/*
 * The Ulysses (DeepSpeed) layout path on one GPU, for comparison with the
 * ring ("Context Parallelism" guide, section 3 "Ulysses (DeepSpeed)", steps
 * 1-4; "Training Long-Context Models Without OOM: Ring Attention", section
 * "Ring Attention vs. DeepSpeed Ulysses (All-to-All)").  P logical ranks;
 * rank i starts with tokens [iC, (i+1)C) of every head of q, k, v
 * ([B, H, S, d], [B, H_kv, S, d] bf16, contiguous).
 *   1. all-to-all: rank r receives chunk i of heads [rH/P, (r+1)H/P) (and
 *      key/value heads [rH_kv/P, (r+1)H_kv/P)) from every rank i -- full
 *      sequences of H/P heads -- as P^2 B device-to-device copies per tensor;
 *   2. every rank computes full-sequence attention for its heads (one launch
 *      of the fused kernel over all ranks, a single chunk);
 *   3. all-to-all of O and LSE back to the ranks' token chunks.
 * o, lse as ring_attn_fwd.  Everything runs on `stream` in this order: the
 * all-to-alls block the compute, as the guide notes.  H and H_kv must be
 * multiples of P (a rank holds whole heads; the pages' limit on Ulysses
 * with few key/value heads), else RA_ERR_UNSUPPORTED.  The result equals
 * ring_attn_fwd_gqa with P = 1 bit for bit.
 */
int ring_attn_fwd_ulysses_emulated(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, ra_bf16 *o,
                                   float *lse, int B, int H, int H_kv, int S, int d, int P, int causal,
                                   float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace ring_attn_bwd needs for this shape: an fp32 dQ
 * accumulator [B, H, S, d] plus two fp32 row vectors [B, H, S]
 * (D_r = sum dO_r * O_r and LSE in base 2), each section 256-byte aligned.
 * Returns 0 for an empty or invalid shape.
 */
size_t ring_attn_bwd_workspace_size(int B, int H, int S, int d);

/*
 * Backward pass.  The pages keep activations for the backward pass and trade
 * compute for memory by recomputation ("Training Long-Context Models
 * Without OOM: Ring Attention", sections "Diagnosing the Sequence-Length
 * OOM" and "Why the Parallelism You Already Have Will Not Work"); the
 * attention matrix is recomputed from the saved LSE, tile by tile, in the
 * same ring order.  For the loss L = sum(dO * O):
 *     P_rc = exp(s_rc - LSE_r) on A_r,  dV = P^T dO,  dP = dO V^T,
 *     D_r = sum_c dO_rc O_rc,  dS = P * (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 *   q, k, v, o, dO  [B, H, S, d] bf16 inputs; lse [B, H, S] fp32 from
 *                   ring_attn_fwd with the same arguments.
 *   dq, dk, dv      [B, H, S, d] bf16 outputs (overwritten).
 *   workspace       device buffer of at least
 *                   ring_attn_bwd_workspace_size(B, H, S, d) bytes, 256-byte
 *                   aligned, owned by the caller; its contents on entry do
 *                   not matter and are clobbered.
 * Other arguments as for ring_attn_fwd.  Inputs must not alias outputs.
 */
int ring_attn_bwd(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, const ra_bf16 *o,
                  const float *lse, const ra_bf16 *dO, ra_bf16 *dq, ra_bf16 *dk, ra_bf16 *dv,
                  int B, int H, int S, int d, int P, int causal, float scale, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * Grouped-query backward: shapes as ring_attn_fwd_gqa; dq is [B, H, S, d],
 * dk and dv are [B, H_kv, S, d] and collect the gradients of every query
 * head of their group.  The workspace is ring_attn_bwd_workspace_size(B, H,
 * S, d) (query heads).  ring_attn_bwd is this call with H_kv = H.
 */
int ring_attn_bwd_gqa(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, const ra_bf16 *o,
                      const float *lse, const ra_bf16 *dO, ra_bf16 *dq, ra_bf16 *dk, ra_bf16 *dv,
                      int B, int H, int H_kv, int S, int d, int P, int causal, float scale,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass over tensors in any row layout: the gradients of
 * ring_attn_bwd_gqa, with the stride convention of ring_attn_fwd_strided
 * for each of q, k, v, o, dO, dq, dk and dv (NULL = contiguous).  lse and
 * the workspace (ring_attn_bwd_workspace_size(B, H, S, d) bytes, 256-byte
 * aligned) keep their contiguous layouts.  The rows of dq, dk and dv must
 * not overlap one another or any input.  Results are bit-identical to
 * ring_attn_bwd_gqa on the same values.
 */
int ring_attn_bwd_strided(const ra_bf16 *q, const long long *q_strides, const ra_bf16 *k,
                          const long long *k_strides, const ra_bf16 *v, const long long *v_strides,
                          const ra_bf16 *o, const long long *o_strides, const float *lse,
                          const ra_bf16 *dO, const long long *do_strides, ra_bf16 *dq,
                          const long long *dq_strides, ra_bf16 *dk, const long long *dk_strides,
                          ra_bf16 *dv, const long long *dv_strides, int B, int H, int H_kv, int S,
                          int d, int P, int causal, float scale, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Size of the fixed device scratch used by ring_attn_bwd_noalloc: 64 MiB per
 * device (one copy on every GPU that loads the library, kept until the
 * process exits).
 */
#define RING_ATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Backward pass for callers that cannot allocate device memory -- for
 * example code running inside a host framework that hands out all device
 * memory through its own pool and forbids raw cudaMalloc, or code on a path
 * where cudaMalloc / cudaFree would block or synchronize the device.  The
 * paper has no counterpart to this entry point.
 *
 * Same arguments, results and errors as ring_attn_bwd, without the
 * workspace: the fp32 dQ accumulator and the two row vectors live in a
 * fixed static device array inside the library
 * (RING_ATTN_NOALLOC_SCRATCH_BYTES).  The caller still passes every input
 * and output.  Shapes whose workspace (ring_attn_bwd_workspace_size) is
 * larger than that array return RA_ERR_UNSUPPORTED before any launch; with
 * d = 128 the limit is about 129,000 rows of B * H * S (16 heads of 8,064
 * tokens fit; 32 heads of 4,096 tokens do not).  The call allocates no device memory and calls
 * no allocating library routine; it clears on `stream` the part of the
 * scratch that must start at zero.
 *
 * Every call on a device shares the one array, and the array keeps the last
 * call's contents.  Calls whose work can overlap on the GPU (for example on
 * two streams with no ordering between them) race on it and give wrong
 * results; order them, e.g. on one stream.  The first call on each device
 * looks up the array's device address (with that device current); make that
 * first call before any stream capture.
 */
int ring_attn_bwd_noalloc(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, const ra_bf16 *o,
                          const float *lse, const ra_bf16 *dO, ra_bf16 *dq, ra_bf16 *dk,
                          ra_bf16 *dv, int B, int H, int S, int d, int P, int causal, float scale,
                          void *stream);

/*
 * Bytes of device workspace ring_attn_fwd_emulated needs: two receive
 * buffers of K and V for the P logical ranks (4 x B*H*S*d bf16), the running
 * and the per-step fp32 O (2 x B*H*S*d fp32) and the per-step LSE, each
 * 256-byte aligned.  0 for an empty or invalid shape.
 */
size_t ring_attn_fwd_emulated_workspace_size(int B, int H, int S, int d);

/*
 * The pages' ring protocol emulated literally with P logical ranks on one
 * GPU ("Training Long-Context Models Without OOM: Ring Attention", "Ring
 * Attention Demystified", steps 2-5; "Context Parallelism" guide, section 2,
 * "How It Works" and "Communication").  Rank i owns query chunk Q_i and a
 * private K/V receive buffer that starts with K_i, V_i.  At ring step t each
 * rank computes the partial attention of Q_i against the chunk it holds
 * (KV chunk (i - t) mod P; nothing for j > i when causal) and folds it into
 * its running (O, LSE) with attn_merge_partials.  Meanwhile every rank sends
 * its chunk to rank (i + 1) % P: device-to-device copies into the other
 * receive buffer on a separate copy stream ("the interconnect"), ordered by
 * events, so the rotation overlaps the step's compute (overlap = 1).  With
 * overlap = 0 the copies run on `stream` between the steps instead, which
 * measures the rotation's cost.  The result equals ring_attn_fwd (O bf16,
 * LSE fp32); P is merged in fp32 and rounded to bf16 once at the end.
 * Arguments as ring_attn_fwd, plus the caller-owned workspace (256-byte
 * aligned, ring_attn_fwd_emulated_workspace_size bytes).  The copy stream
 * and its events are created on the first call on a device and kept.
 * Concurrent calls on one device share them and must be ordered.
 */
int ring_attn_fwd_emulated(const ra_bf16 *q, const ra_bf16 *k, const ra_bf16 *v, ra_bf16 *o,
                           float *lse, int B, int H, int S, int d, int P, int causal, float scale,
                           void *workspace, size_t workspace_bytes, int overlap, void *stream);

/*
 * Log-sum-exp merge of two partial attention results of the same query rows
 * (the merge each ring step performs; "Context Parallelism" guide, section
 * 2: partial results are merged with the online-softmax statistics):
 *     m = max(lse_a, lse_b),  w_a = exp(lse_a - m),  w_b = exp(lse_b - m),
 *     o_out = (w_a o_a + w_b o_b) / (w_a + w_b),  lse_out = m + ln(w_a + w_b).
 * (o = 0, lse = -inf) is the identity; two -inf rows give (0, -inf).
 *   o_a, o_b, o_out      [B, H, S, d] fp32 (any d >= 1; 16-byte aligned).
 *   lse_a, lse_b, lse_out [B, H, S] fp32, natural log (4-byte aligned).
 * In-place use is allowed: o_out == o_a and lse_out == lse_a.  No other
 * aliasing.
 */
int attn_merge_partials(const float *o_a, const float *lse_a, const float *o_b, const float *lse_b,
                        float *o_out, float *lse_out, int B, int H, int S, int d, void *stream);

/*
 * The chunk-level ring schedule the kernels follow, on the host.  For query
 * chunk i (0 <= i < P) writes, in ring order t = 0, 1, ..., the visited KV
 * chunks out_j[n] = (i - t) mod P and their kind out_kind[n]: 0 = the query
 * chunk's own chunk (lower-triangular mask when causal), 1 = a whole chunk.
 * Causal skips j > i.  Returns the number of visits (P, or i + 1 when
 * causal), or RA_ERR_INVALID_ARG (bad P or i, or cap too small; null
 * out_j / out_kind with cap = 0 just returns the count).  Host memory only.
 */
int ring_attn_schedule(int P, int causal, int i, int *out_j, int *out_kind, int cap);

/*
 * Synchronizes `stream`, then reads and clears the current device's status
 * word.  RA_OK if no kernel reported a problem since the last check,
 * RA_ERR_DEVICE_TIMEOUT if a bounded wait ran out, RA_ERR_CUDA if the
 * stream reported an error.
 */
int ring_attn_check_status(void *stream);

/* Static, human-readable name of a status code. */
const char *ring_attn_status_string(int status);

/* Last CUDA error message recorded by this thread (static storage). */
const char *ring_attn_last_error(void);

/*
 * Time limit, in nanoseconds, of every bounded wait inside the kernels
 * launched after this call (default 4e9, i.e. 4 s; 0 restores the default).
 * A small limit makes a valid run end early with RA_ERR_DEVICE_TIMEOUT
 * instead of completing; it exists to test that path.  Returns RA_OK.
 */
int ring_attn_set_wait_limit_ns(unsigned long long ns);

/*
 * Record of the ring order the kernels follow (testing and tracing).
 *   buf       DEVICE buffer of `capacity` ints, 16-byte aligned, owned by
 *             the caller; NULL (with capacity 0) turns recording off, which
 *             is the state at load.
 * While a buffer is set, every CTA of the forward (ring_fwd_kernel) and
 * backward (ring_bwd_kernel) kernels launched afterwards on the current
 * device writes, from its TMA producer thread, the ring visits its tile
 * stream makes -- one entry each time it enters a new chunk -- into its own
 * slot of (P + 1) x 8 ints at buf + blockIdx * (P + 1) * 8:
 *   slot[0..7]        header.  Forward: {b*H + h, query chunk i, first query
 *                     row of the CTA, number of visits, ring step of a
 *                     one-step launch or -1, tiles in total, 0, 0}.
 *                     Backward: {b*H_kv + key/value head, key chunk j, key
 *                     tile in the chunk, number of visits, query tiles in
 *                     total, query heads per key/value head, 0, 0}.
 *   slot[8e .. 8e+7]  visit e = 1 .. visits, in the order made.  Forward:
 *                     {ring step t, key chunk j, kind, tiles, first key,
 *                     first key of the last tile, 0, 0}.  Backward: {query
 *                     chunk i, ring step t = (i - j) mod P, kind, tiles,
 *                     first query, first query of the last tile, 0, 0}
 *                     (the tiles of the first query head of a group; the
 *                     other heads repeat them).
 *   kind is 0 for the CTA's own chunk (i == j) and 1 for any other.
 * The order is the one the "Context Parallelism" guide, section 2 "How It
 * Works", gives: at step t query chunk i meets KV chunk (i - t) mod P, and
 * causal attention skips chunks j > i.  Slots past `capacity` are not
 * written.  The setting is per device and process-wide; change it only
 * while no kernel of this library is running.  Returns RA_ERR_INVALID_ARG
 * for a misaligned buffer or a NULL/capacity mismatch.
 */
int ring_attn_trace_visits(int *buf, long long capacity);

/*
 * Kernel timing.  While enabled, every kernel the library launches is
 * bracketed by a pair of CUDA events on its launch stream.
 * ring_attn_profile_read synchronizes on the recorded events and returns,
 * for the kernel named (one of "ring_fwd_kernel", "ring_bwd_kernel",
 * "bwd_prep_kernel", "dq_convert_kernel", "merge_partials_kernel"), the
 * number of launches and their summed device time in milliseconds since
 * the last ring_attn_profile_reset.  Host-side state, process-wide; not for
 * use inside CUDA graph capture.  RA_ERR_INVALID_ARG for an unknown name.
 */
int ring_attn_profile_enable(int on);
int ring_attn_profile_reset(void);
int ring_attn_profile_read(const char *kernel, double *total_ms, long long *launches);

#ifdef __cplusplus
}
#endif

#endif /* RING_ATTN_H */
