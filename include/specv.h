/*
 * specv.h -- C ABI of the batched speculative-decoding verify step on one
 * GB300 (sm_103a).
 *
 * For every sequence b of a batch the library scores k draft tokens against
 * the target model's k+1 output distributions and emits between 1 and k+1
 * tokens whose distribution is exactly the target's:
 *
 *   1. p_i = softmax(target_logits[b,i,:] / T_b) at each position i = 0..k
 *      ("Speculative decoding." lesson, "First: what an output distribution
 *      is": softmax of the logits, temperature divides them first);
 *   2. draft token x_i is kept iff U[b,i,0] < min(1, p_i(x_i) / q_i(x_i)),
 *      q_i(x_i) clamped below at 1e-12 ("LLM Inference & Speculative
 *      Decoding: From Roofline Physics to Lossless Acceleration", s.2,
 *      acceptance rule and its PyTorch verification step);
 *   3. the walk stops at the first rejected position j ("Speculative
 *      Decoding: Mathematical Foundations, ...", "The Modified Rejection
 *      Sampling Algorithm": later drafts are discarded);
 *   4. at j < k one token is drawn from max(0, p_j - q_j) normalised, by
 *      inverse CDF with U[b,j,1]; if all k drafts are kept, the bonus token is
 *      drawn from p_k with U[b,k,1] (same sources, residual distribution and
 *      bonus token).  If the residual has zero mass, p_j is sampled instead
 *      ("Speculative Decoding: Draft, Verify, Accept", demo script part B).
 *   Rows with T_b == 0 use the greedy rule: keep x_i while it equals
 *   argmax p_i (lowest index on ties), emit the argmax at the first mismatch
 *   or at position k ("LLM Inference & Speculative Decoding ...", s.4 fix for
 *   T -> 0; "Speculative Decoding: Mathematical Foundations, ...", "Greedy
 *   Decoding Equivalence").
 *
 * Inverse CDF: the emitted token is the smallest v (vocabulary order) with
 *   u * W < w(0) + ... + w(v), W the total weight ("Speculative decoding."
 *   lesson: lay the probabilities end to end and take the slice u lands in).
 *
 * Layouts (all row-major, contiguous, device memory unless stated):
 *   target_logits [B, k+1, V]  bf16 (SPECV_BF16) or fp32 (SPECV_F32)
 *   draft_probs   [B, k, V]    fp32, the distribution the drafts were drawn
 *                              from, used as given (never re-tempered); or
 *                              NULL for one-hot drafts (prompt lookup, n-gram
 *                              or greedy drafting: q is the point mass at the
 *                              draft token, so a draft is kept with
 *                              probability p(x) and a rejection samples p with
 *                              x removed -- "Speculative decoding." lesson,
 *                              "One guess (lookup)", "N-gram and prompt
 *                              lookup"; no page gives a separate call for it)
 *   draft_tokens  [B, k]       int32
 *   uniforms      [B, k+1, 2]  fp32 in [0,1); [b,i,0] drives the accept test
 *                              at i < k, [b,j,1] the residual/bonus draw at
 *                              the stop position j; [b,k,0] is unused
 *   temperature   [B]          fp32; 0 = greedy row; otherwise a finite
 *                              normal positive float
 *   num_accepted  [B]          int32 out, j in [0, k]; the row emits j+1 tokens
 *   out_tokens    [B, k+1]     int32 out: x_0..x_{j-1}, then the fixed or
 *                              bonus token at index j, then -1
 *   row_status    [B]          int32 out (nullable), bit mask:
 *                                1  non-finite logits at an examined position
 *                                   (a NaN or +inf, or all -inf; greedy rows:
 *                                   a NaN)
 *                                2  draft token outside [0, V)
 *                                4  uniform outside [0, 1)
 *                                8  temperature negative, NaN, infinite or
 *                                   subnormal
 *                               16  (information) residual mass was zero, the
 *                                   token was drawn from p_j
 *                               32  draft probability NaN, negative or
 *                                   infinite at an examined entry
 *                               64  an internal wait timed out (the result of
 *                                   this row is not valid)
 *                              512  (tree verification) a parent index
 *                                   outside [-1, node)
 *                             1024  (top-k / top-p verification) top_k
 *                                   outside [1, 4096] or top_p outside (0, 1]
 *                              The walk checks position 0, 1, ... in order and
 *                              stops at the first position with an error; a
 *                              row with any of the bits 1, 2, 4, 8, 32, 64, 512, 1024 set
 *                              reports num_accepted = 0 and out_tokens = -1.
 *
 * Ownership and execution: the caller owns every buffer.  Calls are
 * asynchronous on the given CUDA stream (a cudaStream_t passed as void*;
 * NULL is the legacy default stream) and allocate nothing; argument errors
 * are reported synchronously before anything is launched.  A handle may be
 * used from one host thread at a time.  Pointers need no particular
 * alignment; sizes are limited by the handle (batch <= max_batch,
 * 1 <= k <= max_k, V <= vocab).
 */
#ifndef SPECV_H
#define SPECV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct specv_ctx *specv_handle;

typedef enum {
    SPECV_OK = 0,
    SPECV_ERR_INVALID_ARGUMENT = 1, /* bad pointer, size or dtype; nothing launched */
    SPECV_ERR_UNSUPPORTED = 2,      /* device is not sm_103 or lacks a needed feature */
    SPECV_ERR_CUDA = 3,             /* a CUDA runtime call failed (see specv_last_cuda_error) */
    SPECV_ERR_TIMEOUT = 4           /* reserved: reported per row as row_status bit 64 */
} specv_status;

typedef enum { SPECV_F32 = 0, SPECV_BF16 = 1 } specv_dtype;

/* Optional intermediates, all device pointers, each nullable.  For greedy
 * rows row_sumexp, p_at_draft, q_at_draft and residual_mass are 0. */
typedef struct {
    float *p_at_draft;    /* [B, k]   p_i(x_i) (0 if x_i is out of range) */
    float *q_at_draft;    /* [B, k]   q_i(x_i) as read, 1 for one-hot drafts (0 if out of range) */
    float *row_max;       /* [B, k+1] max_v logits[b,i,v] */
    float *row_sumexp;    /* [B, k+1] sum_v exp((logits[b,i,v] - row_max) / T) */
    float *residual_mass; /* [B]      sum_v max(0, p_j(v) - q_j(v)) at a rejected
                                      position (1 - p_j(x_j) for one-hot drafts),
                                      else 0 */
} specv_debug;

/* Create a handle on CUDA device `device` for batches up to max_batch rows,
 * 1 <= k <= max_k (1 <= max_k <= 31: positions 0..k fit one warp) and
 * vocabularies up to `vocab` entries (1 <= vocab <= 262144: at most 16 CTAs
 * of 16384 entries a position).  Other values: SPECV_ERR_INVALID_ARGUMENT.
 * Queries the device; allocates no device memory.  Returns
 * SPECV_ERR_UNSUPPORTED if the device is not compute capability 10.3.
 * Two environment variables, read at every call, override the launch plan
 * (for tests and tuning; the results do not depend on them):
 * SPECV_CLUSTER=C (V > 2048: C CTAs per row, from the fewest the slice limit
 * allows up to 16) and SPECV_SMALLV=row|warp (V <= 2048: one CTA of eight
 * warps per row, or one warp per row; by default the first while the batch
 * is at most twice the SM count). */
specv_status specv_create(specv_handle *out, int device, int max_batch, int max_k, int64_t vocab);

/* Sampled verification (rows with temperature 0 take the greedy rule).
 * target_logits: dtype logits_dtype; every other pointer as in the layout
 * table above; dbg may be NULL.  V = vocabulary size of this call. */
specv_status specv_verify_sample(specv_handle h, specv_dtype logits_dtype, const void *target_logits,
                                 const float *draft_probs, const int32_t *draft_tokens,
                                 const float *uniforms, const float *temperature, int batch, int k,
                                 int64_t V, int32_t *num_accepted, int32_t *out_tokens,
                                 int32_t *row_status, const specv_debug *dbg, void *stream);

/* Sampled verification with top-k / top-p applied to each target row before
 * the rule ("Speculative decoding." lesson, "Why the output is exactly p":
 * temperature, top-k and top-p have to be applied to p before the rule, and
 * to q before drafting -- q is used as given).  The pages name the filters
 * without defining them; the readings here:
 *   top_k [B] int32, 1..4096: keep the top_k largest logits (all V if
 *         top_k >= V), the lower index first among equal logits;
 *   top_p [B] fp32, (0, 1]: within those, in the same order, keep the
 *         shortest prefix whose mass (renormalised over the top_k) reaches
 *         top_p (at least one entry; 1 keeps all top_k).
 * p' = exp((l - max) / T) on the kept set, renormalised; the accept test,
 * the residual max(0, p' - q) and the bonus use p'.  The residual and the
 * bonus are drawn over the kept set in vocabulary order; q is read (and
 * checked, bit 32) only there and at the draft tokens.  draft_probs may be
 * NULL (one-hot drafts), device memory, or page-locked host memory, read in
 * place (pageable host memory: SPECV_ERR_INVALID_ARGUMENT).  A row whose
 * top_k or top_p is out of range gets row_status bit 1024 and emits
 * nothing.  Rows with temperature 0 take the greedy rule (the filters keep
 * the argmax).  Other arguments and bits as for specv_verify_sample; no
 * debug outputs.  Two launches on the stream: rows with top_k up to 64 (and
 * greedy or refused rows) take one thread-block cluster of min(k + 1, 8)
 * CTAs per row that keeps each position's best 64 in registers; rows with
 * top_k above 64 take a cluster of min(k + 1, 16) CTAs per row that selects
 * each position's kept set exactly by a radix select on the logits' keys. */
specv_status specv_verify_sample_filtered(specv_handle h, specv_dtype logits_dtype, const void *target_logits,
                                          const float *draft_probs, const int32_t *draft_tokens,
                                          const float *uniforms, const float *temperature, const int32_t *top_k,
                                          const float *top_p, int batch, int k, int64_t V, int32_t *num_accepted,
                                          int32_t *out_tokens, int32_t *row_status, void *stream);

/* Greedy verification of every row (no draft probabilities, uniforms or
 * temperatures): keep x_i while it equals the target argmax. */
specv_status specv_verify_greedy(specv_handle h, specv_dtype logits_dtype, const void *target_logits,
                                 const int32_t *draft_tokens, int batch, int k, int64_t V,
                                 int32_t *num_accepted, int32_t *out_tokens, int32_t *row_status,
                                 void *stream);

/* Greedy verification of draft trees ("LLM Inference & Speculative Decoding:
 * From Roofline Physics to Lossless Acceleration", s.3 "Multi-Draft Tree
 * Speculation"; "Speculative Decoding: Mathematical Foundations, ...",
 * "SpecInfer and Tree-Based Verification": the target scores every node in
 * one pass and the longest accepted path is kept).  Device pointers:
 *   target_logits [B, M+1, V]  row 0: the prediction after the prefix;
 *                              row 1+i: the prediction after node i
 *   tokens        [B, M]       int32, the draft token of each node
 *   parents       [B, M]       int32, parent node of each node, in [-1, i)
 *                              (-1: a child of the prefix)
 *   num_accepted  [B]          out: length of the kept path
 *   out_tokens    [B, M+1]     out: the path's tokens from the prefix down,
 *                              then the bonus (argmax after the path's last
 *                              node, or of row 0), -1 after
 *   path          [B, M]       out (nullable): the path's node indices, -1 after
 *   row_status    [B]          out (nullable): 0, or bits 1 (a NaN logit in
 *                              any row), 2 (a token outside [0, V)), 512 (a
 *                              parent outside [-1, i)); such rows emit nothing
 * A node is kept iff its parent is kept (the prefix always is) and its
 * token is the argmax (lowest index on ties) of its parent's row; the
 * deepest kept node wins, the lowest index among equally deep ones.  The
 * pages define the path only in words; this is the plain reading.  A chain
 * (parent i-1) gives exactly specv_verify_greedy.  1 <= M <= max_k. */
specv_status specv_verify_tree_greedy(specv_handle h, specv_dtype logits_dtype, const void *target_logits,
                                      const int32_t *tokens, const int32_t *parents, int batch, int M, int64_t V,
                                      int32_t *num_accepted, int32_t *out_tokens, int32_t *path,
                                      int32_t *row_status, void *stream);

/* Same as specv_verify_sample, but every pointer is HOST memory (pinned
 * memory gives the fastest copies).  The handle copies the inputs to device
 * buffers it owns (allocated on the first call, grown when a larger call
 * comes; this is the one call that may allocate), verifies, copies the three
 * outputs back and synchronises `stream` before returning.  draft_probs in
 * page-locked host memory (cudaHostAlloc / cudaHostRegister) is not copied:
 * the kernel reads in place the entries the rule needs (q at the draft
 * tokens and the stop rows), with plain loads; pageable draft_probs is
 * copied like the other inputs. */
specv_status specv_verify_sample_host(specv_handle h, specv_dtype logits_dtype, const void *target_logits,
                                      const float *draft_probs, const int32_t *draft_tokens,
                                      const float *uniforms, const float *temperature, int batch,
                                      int k, int64_t V, int32_t *num_accepted, int32_t *out_tokens,
                                      int32_t *row_status, void *stream);

/* Paged KV-cache bookkeeping after a verification ("LLM Inference &
 * Speculative Decoding: From Roofline Physics to Lossless Acceleration", s.1,
 * PagedKVCacheManager.rollback_to), all pointers device memory:
 *   num_accepted [B]               int32, as returned by a verify call
 *   seq_lens     [B]               int32 in/out: positions held in the cache,
 *                                  the last k of them the drafts; becomes
 *                                  seq_len - (k - num_accepted)
 *   block_tables [B, max_blocks]   int32 in/out: physical block of each
 *                                  logical block; popped entries become -1
 *   num_blocks   [B]               int32 in/out: blocks in use; becomes
 *                                  ceil(new seq_len / block_size)
 *   free_list    [free_capacity]   int32: freed blocks are appended
 *   free_count   [1]               int32 in/out: entries used in free_list
 *   row_status   [B]               int32 out (nullable): 0; 128 if the row's
 *                                  num_accepted is outside [0, k], its new
 *                                  length would be negative or num_blocks is
 *                                  outside [0, max_blocks] (the row is left
 *                                  as it is); 256 on every row if the free
 *                                  list has no room for all freed blocks
 *                                  (then nothing changes)
 * The result equals rolling the rows back one at a time in batch order,
 * each row's blocks popped last-first.  Asynchronous on `stream`; argument
 * errors are returned before launch (SPECV_ERR_INVALID_ARGUMENT, among them
 * free_capacity outside [0, INT32_MAX]: free_count is an int32). */
specv_status specv_rollback(specv_handle h, const int32_t *num_accepted, int batch, int k, int32_t *seq_lens,
                            int32_t *block_tables, int max_blocks, int32_t *num_blocks, int block_size,
                            int32_t *free_list, int64_t free_capacity, int32_t *free_count, int32_t *row_status,
                            void *stream);

/* Number of CTAs per sequence (thread-block cluster size, 1..16) that the
 * next call with these sizes would use; 0 if the sizes are invalid. */
int specv_plan_cluster(specv_handle h, specv_dtype logits_dtype, int batch, int k, int64_t V);

/* Test hook, off unless called: arms the next launch of the split-vocabulary
 * kernel (V > 2048) on this handle so that CTA 0 of the grid never issues
 * the bulk copy of its pass-1 stage use number `stage_use` (counted from 0
 * in issue order) nor signals it, and every wait of that launch gives up
 * after `polls` polls.  The waits that run out end the row's work: it
 * reports row_status bit 64 (num_accepted 0, out_tokens -1) and the call
 * still returns SPECV_OK; the other rows and the next call run normally.  No
 * copy is in flight when a CTA exits (it waits, bounded, for every copy it
 * issued).  SPECV_ERR_INVALID_ARGUMENT for stage_use < 0 or polls < 1. */
specv_status specv_test_withhold_stage(specv_handle h, int stage_use, int polls);

/* Kernel launches issued by this handle since it was created. */
int64_t specv_launch_count(specv_handle h);

/* Release the handle and any buffers it owns.  NULL is ignored. */
void specv_destroy(specv_handle h);

/* Static description of a status code. */
const char *specv_status_string(specv_status s);

/* Text of the last CUDA error seen by this library on the calling thread. */
const char *specv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECV_H */
