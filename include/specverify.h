/*
 * specverify.h -- C ABI of the GB300 (sm_103a) library for the data-parallel
 * hot path of batch speculative decoding: per-round verification of k draft
 * tokens against k+1 target logit rows, and the ragged-to-rectangular
 * realignment of a contiguous left-padded KV cache, position IDs and
 * attention mask that variable acceptance forces.
 *
 * Pages the operations are defined on (cited by title and section):
 *   "Correctness Forensics for Batch Speculative Decoding: Diagnosing the
 *    Ragged Tensor Problem" (summary of arXiv 2510.22876v4)     -- [CF]
 *   "Chapter 10 Speculative Decoding (Code Walkthrough)" (zero-to-sglang)
 *                                                                -- [ZS]
 *   "Design Document -- speculative-decoding-real"               -- [SDR]
 *   "Speculative decoding: proposals and verified output" (Atlas lesson)
 *                                                                -- [AL]
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless stated; the
 *     library allocates nothing and keeps no state between calls.
 *   - Every call is asynchronous on `cuda_stream` (a cudaStream_t, NULL =
 *     the legacy default stream) and returns once its kernels are enqueued.
 *   - Return value: SPEC_OK, or a negative SPEC_E* code for an argument error
 *     found on the host (nothing is launched then) or a failed launch.
 *     Errors that depend on device data never trap: they go to per-sequence
 *     flag words or an error word in device memory.
 *   - Sizes are int; a batch of 0 sequences is a valid no-op.
 *   - `workspace` is caller-owned device scratch of at least
 *     spec_workspace_bytes(B, k, V) bytes, 256-byte aligned.  It must be
 *     zero-filled before its first use (spec_workspace_init does that); every
 *     call that completes leaves its counters at zero again, so later calls
 *     need no re-zeroing.  Calls that share one workspace must be ordered
 *     (the same stream, or events); concurrent calls need separate
 *     workspaces.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of target logits (and of KV elements for realignment). */
typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1, SPEC_F16 = 2 } spec_dtype;

enum {
    SPEC_OK = 0,
    SPEC_EINVAL = -1,     /* null pointer, negative size, k out of range */
    SPEC_EDTYPE = -2,     /* unknown spec_dtype */
    SPEC_EWORKSPACE = -3, /* workspace NULL, misaligned or too small */
    SPEC_ECUDA = -4,      /* a CUDA launch failed (see cudaGetLastError) */
    SPEC_EALIGN = -5,     /* a pointer lacks the alignment its type needs */
    SPEC_ESCRATCH = -6    /* sizes need more than SPEC_STATIC_SCRATCH_BYTES */
};

/* Per-sequence flag bits of spec_verify_sample. */
#define SPEC_FLAG_Q_ZERO 1u        /* q(y) = 0 for a tested proposal y        */
#define SPEC_FLAG_ZERO_RESIDUAL 2u /* rejection left no positive residual     */
#define SPEC_FLAG_NONFINITE 4u     /* a used logits row held inf / NaN        */
#define SPEC_FLAG_BAD_TOKEN 8u     /* a proposal outside [0, V)               */

/* Values of the realignment error word. */
#define SPEC_REALIGN_OK 0
#define SPEC_REALIGN_CAPACITY 1 /* new width W' > S: nothing was moved     */
#define SPEC_REALIGN_LAYOUT 2   /* input breaks rectangular alignment       */
#define SPEC_REALIGN_EMIT 3     /* a committed count would run past S       */
#define SPEC_REALIGN_TIMEOUT 4  /* a bounded wait gave up (never expected)  */

/* Most caches one spec_realign_kv_multi call moves. */
#define SPEC_MAX_CACHES 4

/* Largest vocabulary of spec_verify_sample_filtered. */
#define SPEC_MAX_FILTER_V (1 << 18)

/* Largest pool (sequences) of the ragged-pool entry points. */
#define SPEC_MAX_POOL 65536

/* Largest k (proposals per sequence) accepted by the verify entry points. */
#define SPEC_MAX_K 31
/* Largest pool accepted by spec_group_by_length. */
#define SPEC_MAX_GROUP_N 4096

/* Bytes of workspace that any call with these sizes needs (B sequences, k
 * proposals, vocabulary V).  Never fails; returns 0 only for B <= 0. */
SPEC_API size_t spec_workspace_bytes(int B, int k, int V);

/* Zero-fill `bytes` of workspace on the stream (a cudaMemsetAsync). */
SPEC_API int spec_workspace_init(void *workspace, size_t bytes, void *cuda_stream);

/* Text for a SPEC_* return code. */
SPEC_API const char *spec_status_str(int status);

/*
 * Greedy verification of one round for every sequence of a batch.
 * Definition ([ZS] §4.1 greedy_commit; [SDR] "Standard Greedy Algorithm"
 * steps 4-6; [CF] App. D): for j < k_b the argmax t_j of target row j (lowest
 * index among equal maxima; a NaN counts as larger than any number) is
 * committed; the round stops after t_j when t_j == eos_id, when the number
 * committed reaches remaining[b], or when t_j != draft_tokens[b, j] (t_j is
 * then the correction).  If all k_b proposals are accepted, the argmax of row
 * k_b is the bonus.  Row alignment ([ZS] §3.3): row j of sequence b is the
 * target's prediction after the confirmed prefix plus proposals 0..j-1.
 *
 * target_logits [B, k+1, V] row-major in `dt` (16-byte alignment preferred)
 * draft_tokens  [B, k] int32
 * draft_len     [B] int32 proposals per sequence, each in [0, k], or NULL (= k)
 * eos_id        end-of-sequence token, or negative for none
 * remaining     [B] int32 output budget (<= 0 commits nothing) or NULL
 * out_tokens    [B, k+1] int32 committed tokens, -1 after the last
 * n_accept      [B] int32 committed tokens that are accepted proposals
 * n_emit        [B] int32 committed tokens (n_accept plus 0 or 1)
 * 1 <= V, 0 <= k <= SPEC_MAX_K.  Rows after the first stop are not needed and
 * may not be read.
 */
SPEC_API int spec_verify_greedy(const void *target_logits, spec_dtype dt, int B, int k, int V,
                       const int32_t *draft_tokens, const int32_t *draft_len, int32_t eos_id,
                       const int32_t *remaining, int32_t *out_tokens, int32_t *n_accept,
                       int32_t *n_emit, void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Stochastic verification of one round ([ZS] §5.1; [AL] "The mechanism"
 * steps 2-4 and "Acceptance and rejection correction").
 * p_j = softmax(target row j / temperature), computed in fp32 as
 * x * (1/temperature); q_j = draft_probs[b, j, :] (already processed by any
 * sampling transform).  Proposal y = draft_tokens[b, j] is accepted iff
 * uniforms[b, j] < p_j(y) / q_j(y).  At the first rejection the correction is
 * drawn from the normalised positive residual max(0, p_j - q_j) and the round
 * stops; if that residual sums to 0 the draw is from p_j and
 * SPEC_FLAG_ZERO_RESIDUAL is set.  After k_b acceptances the bonus is drawn
 * from p_{k_b}, the target ([CF] App. D).  Each draw is an inverse-CDF draw at
 * uniforms[b, k]: the smallest index whose prefix sum exceeds u * total (the
 * last positive-weight index if rounding leaves none).  EOS and the budget
 * stop the round as in spec_verify_greedy.
 *
 * draft_probs  [B, k, V] fp32; uniforms [B, k+1] fp32 in [0, 1)
 * out_residual [B, V] fp32 or NULL: the normalised distribution of the round's
 *              draw; rows of sequences that drew nothing are not written
 * flags        [B] uint32 SPEC_FLAG_* bits, or NULL
 * Other arguments as in spec_verify_greedy; temperature > 0.
 */
SPEC_API int spec_verify_sample(const void *target_logits, spec_dtype dt, float temperature,
                       const float *draft_probs, const int32_t *draft_tokens,
                       const float *uniforms, int B, int k, int V, const int32_t *draft_len,
                       int32_t eos_id, const int32_t *remaining, int32_t *out_tokens,
                       int32_t *n_accept, int32_t *n_emit, float *out_residual, uint32_t *flags,
                       void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Stochastic verification with top-k / top-p applied to the target
 * distribution: the ratio test, the residual and the bonus use the processed
 * distribution ([ZS] §5.1: with temperature, Top-k or Top-p, keep the
 * processed probabilities; [AL] "The mechanism" step 1).  Order: temperature,
 * top-k, top-p.  Per sequence b:
 *   top_k[b] in (0, V): keep the logits >= the k-th largest (ties kept);
 *     <= 0 or >= V: off.  top_k == NULL: off for every sequence.
 *   top_p[b] < 1: among those, keep v iff the mass of strictly larger logits
 *     is below top_p[b] times their total (the smallest set of top values
 *     reaching top_p, ties kept; the largest value is always kept, so
 *     top_p <= 0 keeps only it); >= 1 or NaN: off.  top_p == NULL: off.
 *   p = softmax(x / T) renormalised over the kept tokens.
 * The top-p boundary is decided on exact integer sums of fixed-point weights
 * Q = floor(2^40 * 2^t), t = fp32(fp32(x - x_max) * fp32(log2(e) / T)), 2^t by
 * range reduction and the degree-7 Taylor polynomial of 2^f evaluated in fp32
 * with fused multiply-adds, so the kept set does not depend on summation
 * order.  The draft probabilities are taken as given: they must already be
 * the draft's processed distribution.
 * Everything else -- arguments, layouts, flags, outputs, errors -- is as in
 * spec_verify_sample; top_k [B] int32 and top_p [B] fp32 are device arrays
 * (4-byte aligned).  With both NULL this is spec_verify_sample.  With either
 * given, V > SPEC_MAX_FILTER_V returns SPEC_EINVAL.
 */
SPEC_API int spec_verify_sample_filtered(const void *target_logits, spec_dtype dt, float temperature,
                                const int32_t *top_k, const float *top_p, const float *draft_probs,
                                const int32_t *draft_tokens, const float *uniforms, int B, int k, int V,
                                const int32_t *draft_len, int32_t eos_id, const int32_t *remaining,
                                int32_t *out_tokens, int32_t *n_accept, int32_t *n_emit, float *out_residual,
                                uint32_t *flags, void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Realignment of a contiguous left-padded KV cache after a round
 * ("unpad-append-repad", [CF] §3.2 and App. B).
 * Layout: kv [L, 2, B, H, S, D] of `dt` elements; the (layer, K/V, sequence,
 * head) slab is a contiguous run of S rows of D elements.  On input sequence b
 * holds len[b] confirmed tokens at slots pad[b] .. pad[b] + len[b] - 1 of the
 * common width W = pad[b] + len[b], min pad = 0, and the verification forward
 * wrote the KV of the last token and the proposals at slots W-1 .. W+k-1.
 * With n = n_emit[b]: len' = len + n, W' = max len', pad' = W' - len'.  The run
 * of len' - 1 rows at slot pad[b] (everything that has target-computed KV: the
 * old prefix, the last token, the accepted proposals) moves to slot pad'[b]
 * with memmove semantics; the committed correction/bonus has no KV yet.  Only
 * sequences with pad' != pad move, and no other byte of kv is written.
 *
 * len, pad, n_emit [B] int32 (inputs); len_new, pad_new [B] int32 and
 * width_new [1] int32 (outputs; len_new / pad_new may alias len / pad).
 * err [1] int32: SPEC_REALIGN_* -- on any value but OK, kv and the outputs are
 * left untouched.  kv must be 16-byte aligned when D * sizeof(dt) is a
 * multiple of 16 (the bulk-copy path); other row sizes take a plain path.
 */
SPEC_API int spec_realign_kv(void *kv, spec_dtype dt, int L, int B, int H, int S, int D,
                    const int32_t *len, const int32_t *pad, const int32_t *n_emit,
                    int32_t *len_new, int32_t *pad_new, int32_t *width_new, int32_t *err,
                    void *workspace, size_t workspace_bytes, void *cuda_stream);

/* One contiguous left-padded KV cache [L, 2, B, H, S, D] of `dt` elements
 * (B and S are given to the call; every cache of one call shares them). */
typedef struct {
    void *kv;
    spec_dtype dt;
    int L, H, D;
} spec_kv_cache;

/*
 * The realignment of spec_realign_kv applied to several caches that share the
 * batch and its slot geometry -- typically the target model's cache and the
 * draft model's, which both must follow the accepted prefix ("Design Document
 * -- speculative-decoding-real", "KV Cache Synchronization": the draft cache
 * is re-synchronised to the accepted prefix by copying the accepted cache
 * entries).  One plan is computed and one shift launch moves the slabs of
 * every cache, balanced across them.
 *
 * caches [n_caches] (host array, 1 <= n_caches <= SPEC_MAX_CACHES); the other
 * arguments as in spec_realign_kv.  A draft cache that holds KV for the last
 * token and proposals 0..k-2 (the draft consumed them while proposing) lacks
 * the row of proposal k-1; when a sequence accepts all k proposals that row
 * is moved like the others but holds no computed KV -- the drafter must
 * recompute it (it re-feeds that token) before reading it.
 */
SPEC_API int spec_realign_kv_multi(const spec_kv_cache *caches, int n_caches, int B, int S,
                          const int32_t *len, const int32_t *pad, const int32_t *n_emit,
                          int32_t *len_new, int32_t *pad_new, int32_t *width_new, int32_t *err,
                          void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Position IDs and attention mask recomputed from the new padding ([CF]
 * App. B: positions are recomputed from the mask after repadding), in one
 * pass: mask[b, s] = (s >= pad_new[b]); pos[b, s] = s - pad_new[b] for
 * s >= pad_new[b], 0 in the padding (cumsum(mask) - 1, clamped at 0).
 * pad_old [B] or NULL: rows with pad_old[b] == pad_new[b] are skipped (their
 * buffers must already hold that state); NULL rewrites every row.  pad_old
 * must not alias pad_new.
 * pos [B, S] int32, mask [B, S] uint8.
 */
SPEC_API int spec_rebuild_pos_mask(int B, int S, const int32_t *pad_old, const int32_t *pad_new,
                          int32_t *pos, uint8_t *mask, void *cuda_stream);

/*
 * Same-length grouping (EXSPEC, [CF] §3.2): from a pool of N sequences with
 * current lengths len [N] (active [N] uint8 or NULL = all active), pick B
 * sequences.  L* = the most frequent active length (ties to the smaller);
 * members of length L* in ascending index, at most B, come first
 * (count_equal of them); remaining slots take other active sequences in
 * ascending (|len - L*|, index); slots beyond the active count are -1.
 * group_len = L* (-1 if nothing is active).  When count_equal == B the group
 * is rectangular in a pool kept left-aligned and realignment can be skipped.
 * The pages give no algorithm for this step: the policy is this library's.
 * out_idx [B], out_count_equal [1], out_group_len [1] int32.
 * 0 <= N <= SPEC_MAX_GROUP_N.
 */
SPEC_API int spec_group_by_length(int N, const int32_t *len, const uint8_t *active, int B,
                         int32_t *out_idx, int32_t *out_count_equal, int32_t *out_group_len,
                         void *cuda_stream);

/* Size of the device scratch built into the library for
 * spec_verify_greedy_static (held by every GPU that loads the library). */
#define SPEC_STATIC_SCRATCH_BYTES (4u << 20)

/*
 * spec_verify_greedy_static -- spec_verify_greedy without a workspace
 * argument.  The pages have no counterpart: this entry point exists for
 * callers that cannot allocate device memory when they call in, for example
 * a serving loop that allows no allocation after start-up so that its memory
 * use stays fixed, or a plugin whose host framework hands it only its input
 * and output buffers and no scratch.  It allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library call): its scratch is a file-scope
 * device array of SPEC_STATIC_SCRATCH_BYTES in the library itself.
 *
 * Same arguments, results and definition as spec_verify_greedy.  Sizes whose
 * scratch (spec_workspace_bytes(B, k, V)) exceeds SPEC_STATIC_SCRATCH_BYTES
 * are rejected with SPEC_ESCRATCH before anything is launched.
 *
 * The array used is the current device's: cuda_stream must belong to the
 * current device (or be a default stream), else SPEC_EINVAL is returned and
 * nothing is enqueued.  The first call on each device looks up the device
 * address of the array (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.  Every call also clears the array's counters
 * with an asynchronous memset on the caller's stream.  All calls on a device
 * share the one array and it keeps the last call's contents, so calls that
 * overlap on the GPU (different streams without ordering) race: order them.
 */
SPEC_API int spec_verify_greedy_static(const void *target_logits, spec_dtype dt, int B, int k, int V,
                              const int32_t *draft_tokens, const int32_t *draft_len, int32_t eos_id,
                              const int32_t *remaining, int32_t *out_tokens, int32_t *n_accept,
                              int32_t *n_emit, void *cuda_stream);

/*
 * Ragged pool of EXSPEC ([CF] §3.2: keep sequences ragged and batch
 * identical-length sequences so realignment is bypassed; when grouping fails,
 * fall back to unpad-append-repad).  Pool cache pool[L, 2, N, H, S, D]:
 * sequence n is left-aligned at slot 0, positions 0 .. pool_len[n] - 2 have
 * KV (the last token has none), and a position ID is its slot index.  A group
 * of equal lengths is rectangular as it is; after a round on it the commit
 * below is the whole "rollback of rejected tokens" a variable-length layout
 * needs ([CF] §2): their KV rows lie past the new length.
 * The pages give no algorithm for EXSPEC's scheduler; the selection policy
 * (spec_group_by_length over a window) and these operations are this
 * library's.
 */

/* pool_len[idx[b]] += n_emit[b] for the B sequences of a round (idx [B] pool
 * indices, distinct).  err [1]: SPEC_REALIGN_OK, SPEC_REALIGN_LAYOUT (an index
 * outside [0, N) or repeated, or a negative count) or SPEC_REALIGN_CAPACITY (a
 * length past S); on an error nothing changes.  0 <= N <= SPEC_MAX_POOL. */
SPEC_API int spec_commit_ragged(int N, int32_t *pool_len, int B, const int32_t *idx, const int32_t *n_emit,
                       int S, int32_t *err, void *cuda_stream);

/* Repad: batch[L, 2, B, H, S, D] row b receives pool sequence idx[b]'s rows
 * 0 .. pool_len[idx[b]] - 2 at slot pad_b = W - pool_len[idx[b]], W = the
 * longest of them; no other batch byte changes.  len_out, pad_out [B] and
 * width_out [1] describe the batch (rectangular alignment holds; the caller
 * rebuilds positions and the mask with spec_rebuild_pos_mask).  err [1]:
 * SPEC_REALIGN_OK or SPEC_REALIGN_LAYOUT (bad or repeated index, a length
 * outside [1, S]; nothing written).  pool and batch must not overlap. */
SPEC_API int spec_repad_gather(const void *pool, void *batch, spec_dtype dt, int L, int N, int B, int H, int S,
                      int D, const int32_t *idx, const int32_t *pool_len, int32_t *len_out,
                      int32_t *pad_out, int32_t *width_out, int32_t *err, void *workspace,
                      size_t workspace_bytes, void *cuda_stream);

/* Unpad: batch row b's rows pad[b] .. pad[b] + len[b] - 2 go back to slot 0 of
 * pool sequence idx[b], and pool_len[idx[b]] = len[b]; no other pool byte
 * changes.  err [1]: SPEC_REALIGN_OK or SPEC_REALIGN_LAYOUT (bad or repeated
 * index, len < 1, pad < 0, n_emit < 0 or a run past S; nothing written).
 * n_emit [B] int32 or NULL: when given, the lengths written back are
 * len + n_emit, read from a batch that a round has just extended without
 * realigning it.  After a round on a left-padded batch of width W the
 * verification forward wrote the last token and the proposals at slots
 * W - 1 .. = pad + len - 1 .., so rows pad .. pad + len + n_emit - 2 hold
 * positions 0 .. len + n_emit - 2: unpadding them needs no realignment first
 * (the pool ends byte for byte as after spec_realign_kv and an unpad with the
 * new lengths and paddings). */
SPEC_API int spec_unpad_scatter(const void *batch, void *pool, spec_dtype dt, int L, int N, int B, int H, int S,
                       int D, const int32_t *idx, const int32_t *len, const int32_t *pad,
                       const int32_t *n_emit, int32_t *pool_len, int32_t *err, void *workspace,
                       size_t workspace_bytes, void *cuda_stream);

/*
 * One whole round in one call: spec_verify_greedy (or spec_verify_sample /
 * spec_verify_sample_filtered), then spec_realign_kv_multi over `caches` with
 * the n_emit the verification produced, then spec_rebuild_pos_mask with
 * pad_old = pad.  The definitions, layouts, outputs and errors are those of
 * the three calls; each argument means what it means there.  Every argument
 * is checked before anything is launched (a non-zero return launches
 * nothing); the launches follow one another on the stream, so the
 * realignment reads n_emit on the device and the caller needs no
 * synchronisation inside a round (the whole round can be captured in a CUDA
 * graph).  pad_new must not alias pad.  One workspace serves all three
 * stages: spec_workspace_bytes(B, k, V).
 */
SPEC_API int spec_round_greedy(const void *target_logits, spec_dtype dt, int B, int k, int V,
                      const int32_t *draft_tokens, const int32_t *draft_len, int32_t eos_id,
                      const int32_t *remaining, const spec_kv_cache *caches, int n_caches, int S,
                      const int32_t *len, const int32_t *pad, int32_t *pos, uint8_t *mask,
                      int32_t *out_tokens, int32_t *n_accept, int32_t *n_emit, int32_t *len_new,
                      int32_t *pad_new, int32_t *width_new, int32_t *err, void *workspace,
                      size_t workspace_bytes, void *cuda_stream);

/* The stochastic round; top_k / top_p may be NULL (see
 * spec_verify_sample_filtered). */
SPEC_API int spec_round_sample(const void *target_logits, spec_dtype dt, float temperature,
                      const int32_t *top_k, const float *top_p, const float *draft_probs,
                      const int32_t *draft_tokens, const float *uniforms, int B, int k, int V,
                      const int32_t *draft_len, int32_t eos_id, const int32_t *remaining,
                      const spec_kv_cache *caches, int n_caches, int S, const int32_t *len,
                      const int32_t *pad, int32_t *pos, uint8_t *mask, int32_t *out_tokens,
                      int32_t *n_accept, int32_t *n_emit, float *out_residual, uint32_t *flags,
                      int32_t *len_new, int32_t *pad_new, int32_t *width_new, int32_t *err,
                      void *workspace, size_t workspace_bytes, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
