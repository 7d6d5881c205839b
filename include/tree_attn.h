/*
 * tree_attn.h -- C ABI of the split tree attention library (libtreeattn.so).
 *
 * Split tree attention is the verification attention of EAGLE-style
 * speculative decoding described in "Efficient Speculative Decoding for Llama
 * at Scale: Challenges and Solutions" (arXiv 2508.08192; pith.science review,
 * section "What carries the argument"): the draft tree is flattened into one
 * sequence of T tokens; attention is computed in two pieces -- every tree
 * token against the committed prefix with no mask, and the tree tokens among
 * themselves under the tree mask -- and the two partial results are merged by
 * log-sum-exp ("merge_attentions", the combination of attention over disjoint
 * KV chunks named in the review's supporting citations).  The prefix lives in
 * a paged KV cache (the review's Referee Report summary counts paged,
 * persistent KV handling among what tree attention needs) and is processed
 * split over its length in
 * the manner of flash-decoding (Dao, Haziza, Massa, Sizov, cited in the
 * review's reference list).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     owned by the caller.  The library never allocates, frees or
 *     synchronises; every call only enqueues work on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and returns.
 *   - bf16 tensors are passed as `const uint16_t *` holding raw bfloat16 bit
 *     patterns.  All layouts are dense row-major in the order written.
 *   - `status` (nullable) is a device int32 the caller zeroes beforehand.
 *     Kernels that detect bad DATA (which the host cannot see without a
 *     synchronisation) store the first such code there (TREE_ATTN_STATUS_*)
 *     and leave the outputs unspecified; they never trap.
 *   - A negative return value means nothing was enqueued.
 */
#ifndef TREE_ATTN_H
#define TREE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TREE_ATTN_API __attribute__((visibility("default")))
#else
#define TREE_ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side return codes. */
#define TREE_ATTN_OK 0
#define TREE_ATTN_ERR_NULL (-1)       /* a required pointer is NULL                */
#define TREE_ATTN_ERR_SHAPE (-2)      /* unsupported or inconsistent sizes         */
#define TREE_ATTN_ERR_ALIGN (-3)      /* a pointer is not suitably aligned         */
#define TREE_ATTN_ERR_WORKSPACE (-4)  /* workspace NULL, too small or misaligned   */
#define TREE_ATTN_ERR_CUDA (-5)       /* a CUDA runtime/driver call failed         */

/* Device-side status codes (written to *status). */
#define TREE_ATTN_STATUS_BAD_PARENT 1   /* parents[i] outside [-1, i)                 */
#define TREE_ATTN_STATUS_BAD_PAGE 2     /* block_table entry outside [0, num_pages)   */
#define TREE_ATTN_STATUS_BAD_SEQ_LEN 3  /* seq_lens[b] < 0 or > max_pages_per_seq*P   */
#define TREE_ATTN_STATUS_TIMEOUT 4      /* an internal pipeline wait gave up           */
#define TREE_ATTN_STATUS_BAD_PATH 5     /* accept_len outside [0, T] or a path node     */
                                        /* outside [0, T) (tree_kv_commit)              */

/* Limits. */
#define TREE_ATTN_MAX_T 64

/*
 * tree_mask_build -- ancestor bitmask of every node of a flattened draft tree.
 *
 * Source: "tree mask" of split tree attention (pith.science review,
 * "What carries the argument"); flattened-draft verification after SpecInfer
 * (Miao et al., verdict record supporting_citations).
 *
 *   parents   int32 [T], parents[i] in {-1} U [0, i): the tree in topological
 *             order; -1 marks a root (several roots form a forest).
 *   T         1 .. 64.
 *   mask_out  uint64 [T]: bit j of mask_out[i] is set iff j == i or node j is
 *             an ancestor of node i; bits >= T are zero.
 *   status    nullable; TREE_ATTN_STATUS_BAD_PARENT if a parent is invalid
 *             (mask_out then unspecified).
 *
 * One warp, pointer jumping over log2(T) rounds.  Returns TREE_ATTN_OK,
 * TREE_ATTN_ERR_NULL, TREE_ATTN_ERR_SHAPE, TREE_ATTN_ERR_ALIGN (mask_out not
 * 8-byte aligned) or TREE_ATTN_ERR_CUDA.
 */
TREE_ATTN_API int tree_mask_build(const int32_t *parents, int T, uint64_t *mask_out,
                                  int32_t *status, void *stream);

/*
 * tree_mask_build_batched -- tree_mask_build for n_trees trees at once
 * (one warp each): parents int32 [n_trees][T] -> mask_out uint64
 * [n_trees][T].  Used with per-sequence draft trees (the pages' tree
 * dispatcher picks trees per batch; sequences may also carry their own).
 * n_trees = 0 enqueues nothing.  Return codes as tree_mask_build.
 */
TREE_ATTN_API int tree_mask_build_batched(const int32_t *parents, int T, int n_trees,
                                          uint64_t *mask_out, int32_t *status, void *stream);

/*
 * tree_attn_workspace_size -- bytes of device scratch tree_attn_verify needs
 * for these sizes on the CURRENT device (the count depends on its SM count).
 * Holds the per-split partial results (m, l, acc) of the prefix pass.
 * max_seq_len is accepted for interface stability and does not change the
 * result.  Returns 0 for unsupported sizes.
 */
TREE_ATTN_API size_t tree_attn_workspace_size(int B, int Hq, int Hkv, int d, int T,
                                              int max_seq_len, int page_size);

/*
 * tree_attn_verify -- split tree attention for one layer.
 *
 * For every sequence b, tree node i and query head h (KV head hk = h / G,
 * G = Hq / Hkv):
 *   keys  = the seq_lens[b] committed prefix tokens (no mask) plus the tree
 *           tokens j with bit j of mask[i] set,
 *   s     = softmax_scale * <q[b][i][h], key>,
 *   out[b][i][h] = softmax(s) . values   (bf16, round to nearest even),
 *   lse[b][i][h] = natural-log log-sum-exp of s (fp32).
 * Computed as (1) a prefix pass split over the KV length, (2) a suffix pass
 * over the tree keys under the mask, (3) a log-sum-exp merge of all partial
 * results.
 *
 *   q            bf16 [B][T][Hq][d]
 *   k_pages,
 *   v_pages      bf16 [num_pages][Hkv][page_size][d]; the slots of a page
 *                beyond a sequence's length are never used in results.
 *   block_table  int32 [B][max_pages_per_seq]: physical page of logical page
 *                p/page_size of sequence b; entries past the sequence's
 *                last page are ignored.
 *   seq_lens     int32 [B]: committed prefix length (0 allowed).
 *   tree_k,
 *   tree_v       bf16 [B][T][Hkv][d]: the draft tokens' keys and values.
 *   mask         uint64 [T] (as built by tree_mask_build), shared by all B.
 *   out          bf16 [B][T][Hq][d];  lse  fp32 [B][T][Hq].
 *   Sizes: B >= 0 (B = 0 enqueues nothing), 1 <= T <= 64, Hq % Hkv == 0,
 *          d in {64, 128}, page_size in {16, 32, 64, 128},
 *          max_pages_per_seq >= 1, num_pages >= 1,
 *          num_pages*Hkv*page_size < 2^31.
 *   workspace    device scratch of at least tree_attn_workspace_size(...)
 *                bytes, 256-byte aligned; contents need no initialisation and
 *                are garbage afterwards.  Calls that share a workspace must
 *                not overlap in time.
 *   status       nullable device int32 (see above).
 *
 * Alignment: q, k_pages, v_pages, tree_k, tree_v, out must be 16-byte
 * aligned; block_table, seq_lens, lse 4-byte; mask 8-byte.
 * Returns TREE_ATTN_OK or a negative TREE_ATTN_ERR_* code.
 */
TREE_ATTN_API int tree_attn_verify(const uint16_t *q, const uint16_t *k_pages,
                                   const uint16_t *v_pages, const int32_t *block_table,
                                   int max_pages_per_seq, const int32_t *seq_lens,
                                   const uint16_t *tree_k, const uint16_t *tree_v,
                                   const uint64_t *mask, uint16_t *out, float *lse, int B, int Hq,
                                   int Hkv, int d, int T, int page_size, int num_pages,
                                   float softmax_scale, void *workspace, size_t workspace_bytes,
                                   int32_t *status, void *stream);

/*
 * tree_attn_verify_ctas -- tree_attn_verify with an explicit number of
 * prefix-pass CTAs (each CTA takes an equal share of the prefix work, so this
 * is the split count).  n_ctas <= 0 selects the default (one per SM).  The
 * workspace must then be sized by tree_attn_workspace_size_ctas with the same
 * n_ctas.  Results differ from the default only by fp32 reassociation.
 */
TREE_ATTN_API int tree_attn_verify_ctas(const uint16_t *q, const uint16_t *k_pages,
                                        const uint16_t *v_pages, const int32_t *block_table,
                                        int max_pages_per_seq, const int32_t *seq_lens,
                                        const uint16_t *tree_k, const uint16_t *tree_v,
                                        const uint64_t *mask, uint16_t *out, float *lse, int B,
                                        int Hq, int Hkv, int d, int T, int page_size,
                                        int num_pages, float softmax_scale, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream,
                                        int n_ctas);

TREE_ATTN_API size_t tree_attn_workspace_size_ctas(int B, int Hq, int Hkv, int d, int T,
                                                   int page_size, int n_ctas);

/*
 * tree_attn_verify_batched -- tree_attn_verify with one draft tree per
 * sequence: masks is uint64 [B][T] (tree b at masks[b * T], e.g. from
 * tree_mask_build_batched).  Everything else as tree_attn_verify.
 */
TREE_ATTN_API int tree_attn_verify_batched(const uint16_t *q, const uint16_t *k_pages,
                                           const uint16_t *v_pages, const int32_t *block_table,
                                           int max_pages_per_seq, const int32_t *seq_lens,
                                           const uint16_t *tree_k, const uint16_t *tree_v,
                                           const uint64_t *masks, uint16_t *out, float *lse,
                                           int B, int Hq, int Hkv, int d, int T, int page_size,
                                           int num_pages, float softmax_scale, void *workspace,
                                           size_t workspace_bytes, int32_t *status, void *stream);

/*
 * tree_attn_verify_tree -- tree_mask_build and tree_attn_verify in one call:
 * the ancestor masks are built inside the suffix/merge kernel from the
 * parent array (one warp's pointer jumping per row, the same algorithm as
 * tree_mask_build), which removes a kernel and its dependency hop from the
 * step.
 *
 *   parents         int32 [T] (parents_stride 0, one tree) or [B][T]
 *                   (parents_stride T, one tree per sequence)
 *   mask_out        nullable uint64 [T] / [B][T]: the masks, for later use
 *                   (e.g. tree_greedy_accept)
 *   status          also receives TREE_ATTN_STATUS_BAD_PARENT
 *
 * Everything else as tree_attn_verify.
 */
TREE_ATTN_API int tree_attn_verify_tree(const uint16_t *q, const uint16_t *k_pages,
                                        const uint16_t *v_pages, const int32_t *block_table,
                                        int max_pages_per_seq, const int32_t *seq_lens,
                                        const uint16_t *tree_k, const uint16_t *tree_v,
                                        const int32_t *parents, int parents_stride,
                                        uint64_t *mask_out, uint16_t *out, float *lse, int B,
                                        int Hq, int Hkv, int d, int T, int page_size,
                                        int num_pages, float softmax_scale, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream);

/*
 * tree_attn_verify_paged_tree -- split tree attention with the draft tokens
 * padded into the paged KV cache (the padded layout named in the pith.science
 * verdict record, desk editor's note): tree token j of sequence b has its
 * K/V at logical position seq_lens[b] + j of that sequence's pages, so the
 * block table must cover seq_lens[b] + T tokens (else status
 * TREE_ATTN_STATUS_BAD_SEQ_LEN).  The prefix pass covers positions
 * [0, seq_lens[b]) unmasked; the suffix pass reads the T tree positions
 * through the block table under the mask.  mask is uint64 [T]
 * (mask_stride 0) or [B][T] (mask_stride T).  No tree_k / tree_v.  Other
 * arguments, layouts and return codes as tree_attn_verify.
 */
TREE_ATTN_API int tree_attn_verify_paged_tree(const uint16_t *q, const uint16_t *k_pages,
                                              const uint16_t *v_pages, const int32_t *block_table,
                                              int max_pages_per_seq, const int32_t *seq_lens,
                                              const uint64_t *mask, int mask_stride, uint16_t *out,
                                              float *lse, int B, int Hq, int Hkv, int d, int T,
                                              int page_size, int num_pages, float softmax_scale,
                                              void *workspace, size_t workspace_bytes,
                                              int32_t *status, void *stream);

/*
 * tree_accept_commit -- tree_greedy_accept and tree_kv_commit in one launch
 * (each commit CTA finds its sequence's path itself).  Arguments as the two
 * calls; accept_len, accept_path and bonus_token are nullable here.  The
 * result is the same as calling the two in turn.
 */
TREE_ATTN_API int tree_accept_commit(const uint64_t *mask, int mask_stride,
                                     const int32_t *draft_tokens, const int32_t *target_tokens,
                                     uint16_t *k_pages, uint16_t *v_pages,
                                     const int32_t *block_table, int max_pages_per_seq,
                                     const int32_t *seq_lens, const uint16_t *tree_k,
                                     const uint16_t *tree_v, int32_t *accept_len,
                                     int32_t *accept_path, int32_t *bonus_token,
                                     int32_t *seq_lens_out, int B, int Hkv, int d, int T,
                                     int page_size, int num_pages, int32_t *status, void *stream);

/*
 * tree_dense_mask_build / tree_attn_verify_dense -- the one-pass form of tree
 * attention under an explicit mask: the very large explicit mask that split
 * tree attention replaces (pith.science review of arXiv 2508.08192, "What carries
 * the argument").  Kept as an ablation of the split form; both compute the
 * same attention.  The tree tokens must sit in the paged cache after each
 * prefix (tree_attn_verify_paged_tree layout).
 *
 * tree_dense_mask_build writes dense_mask uint8 [B][T][dense_cols]:
 *   dense_mask[b][t][p] = 1 for p < seq_lens[b] (the committed prefix),
 *                       = bit (p - seq_lens[b]) of mask[t] for the tree tokens,
 *                       = 0 beyond;
 * and key_lens[b] = seq_lens[b] + T.  dense_cols must be a multiple of 16
 * and at least max_b seq_lens[b] + T (else status TREE_ATTN_STATUS_BAD_SEQ_LEN).
 * mask: uint64 [T] (mask_stride 0) or [B][T] (mask_stride T).
 *
 * tree_attn_verify_dense attends, for query (b, t, h), every cache position
 * p < key_lens[b] with dense_mask[b][t][p] != 0, in one pass (the prefix
 * kernel's split over the key range and the LSE merge still apply; there is
 * no separate tree pass).  Arguments otherwise as tree_attn_verify; the
 * workspace size is tree_attn_workspace_size's.  Returns as tree_attn_verify.
 */
TREE_ATTN_API int tree_dense_mask_build(const uint64_t *mask, int mask_stride,
                                        const int32_t *seq_lens, int B, int T, int dense_cols,
                                        uint8_t *dense_mask, int32_t *key_lens, int32_t *status,
                                        void *stream);

TREE_ATTN_API int tree_attn_verify_dense(const uint16_t *q, const uint16_t *k_pages,
                                         const uint16_t *v_pages, const int32_t *block_table,
                                         int max_pages_per_seq, const int32_t *key_lens,
                                         const uint8_t *dense_mask, int dense_cols, uint16_t *out,
                                         float *lse, int B, int Hq, int Hkv, int d, int T,
                                         int page_size, int num_pages, float softmax_scale,
                                         void *workspace, size_t workspace_bytes, int32_t *status,
                                         void *stream);

/*
 * tree_greedy_accept -- greedy acceptance of the verified draft tree
 * ("Efficient Speculative Decoding for Llama at Scale", fdeinterviews.com
 * summary, opening paragraph: the service commits one accepted path; greedy
 * drafting and verification per the mlsanity.com referee report, Summary).
 *
 *   mask           uint64 [T] (mask_stride 0, one tree) or [B][T] (mask_stride
 *                  T): ancestor-or-self bits as tree_mask_build writes them
 *   draft_tokens   int32 [B][T]: token of tree node i
 *   target_tokens  int32 [B][T]: the target's greedy (argmax) token after
 *                  node i, i.e. its prediction for node i's children
 *   accept_len     int32 [B] out: nodes on the committed path (root included)
 *   accept_path    int32 [B][T] out: the path's nodes root first, then -1
 *   bonus_token    int32 [B] out: target_tokens at the path's last node
 *
 * A root is accepted; node i is accepted when its parent is and
 * draft_tokens[i] == target_tokens[parent].  The path ends at the deepest
 * accepted node, the lowest index among equally deep ones.  Integer work:
 * results are exact.  All pointers device memory owned by the caller; async
 * on `stream`.  Returns 0, -1 (NULL), -2 (T outside [1, 64], B < 0, stride
 * neither 0 nor T), -3 (misaligned), -5 (launch failed).
 */
TREE_ATTN_API int tree_greedy_accept(const uint64_t *mask, int mask_stride,
                                     const int32_t *draft_tokens, const int32_t *target_tokens,
                                     int B, int T, int32_t *accept_len, int32_t *accept_path,
                                     int32_t *bonus_token, void *stream);

/*
 * tree_kv_commit -- write the accepted path's K/V into the paged cache so
 * that it holds the committed history only (fdeinterviews.com summary,
 * paragraph on hidden correctness obligations; mlsanity.com referee report,
 * minor comment on Section 3.3).  For sequence b, path node accept_path[b][k]
 * (k < accept_len[b]) goes to logical position seq_lens[b] + k.
 *
 *   tree_k, tree_v  bf16 [B][T][Hkv][d] sources, or both NULL when the tree
 *                   tokens already sit in the cache at seq_lens[b] + j
 *                   (tree_attn_verify_paged_tree layout); that compaction is
 *                   done in place, every row read before any is written
 *   seq_lens_out    nullable int32 [B]: seq_lens[b] + accept_len[b]; must not
 *                   be seq_lens itself (-2)
 *   status          nullable: TREE_ATTN_STATUS_BAD_PATH, _BAD_PAGE (a target
 *                   position's page outside [0, num_pages)), _BAD_SEQ_LEN (a
 *                   position past max_pages_per_seq * page_size); rows that
 *                   fail are skipped
 *
 * The pages that positions [seq_lens[b], seq_lens[b] + T) map to must be
 * mapped by the caller and not shared with another sequence of the batch.
 * Shapes as tree_attn_verify.  Returns 0, -1, -2, -3, -5.
 */
TREE_ATTN_API int tree_kv_commit(uint16_t *k_pages, uint16_t *v_pages, const int32_t *block_table,
                                 int max_pages_per_seq, const int32_t *seq_lens,
                                 const uint16_t *tree_k, const uint16_t *tree_v,
                                 const int32_t *accept_path, const int32_t *accept_len,
                                 int32_t *seq_lens_out, int B, int Hkv, int d, int T,
                                 int page_size, int num_pages, int32_t *status, void *stream);

/*
 * tree_attn_plan -- the kernel selector's choices for a call of these shapes
 * (the split-count heuristic of flash-decoding, Dao et al., cited in the
 * pith.science verdict record's supporting_citations; here it sizes a
 * persistent stream-K grid instead of a split count).  Host only; the
 * verify entry points make the same choices.  Inputs as tree_attn_verify;
 * sm_count_hint > 0 replaces the current device's SM count (no CUDA call is
 * then made).  Returns 0, -1 (out NULL), -2 (shapes), -5 (no device).
 */
typedef struct tree_attn_plan_info {
    int units;               /* B * Hkv * row_blocks work units                      */
    int row_blocks;          /* ceil(T * Hq / Hkv / 128) query-row blocks per unit   */
    int replicas;            /* query-row copies per 128-row tile (1, 2 or 4)         */
    int n_ctas;              /* persistent prefix-pass CTAs                           */
    int merge_warps_per_row; /* warps that merge one query row (1, 2 or 4)            */
    long long max_steps;     /* 64-token work-line steps if every sequence were full */
                             /* (+1 per unit when the tree rides on the prefix pass) */
    size_t workspace_bytes;  /* partial-result slots for this n_ctas                 */
    int tree_in_prefix;      /* 1: the prefix pass attends the tree tokens too (one   */
                             /* masked chunk per unit: calls of at most 32 steps per  */
                             /* CTA, or with no more units than CTAs and 2 or more    */
                             /* row copies); 0: the suffix/merge kernel attends them  */
    int merge_rows_per_warp; /* query rows each merge warp takes in turn (> 1 only    */
                             /* when the tree is on the prefix pass and one row per   */
                             /* warp would need more merge CTAs than the SMs hold)    */
} tree_attn_plan_info;

TREE_ATTN_API int tree_attn_plan(int B, int Hq, int Hkv, int d, int T, int page_size,
                                 int max_pages_per_seq, int sm_count_hint,
                                 tree_attn_plan_info *out);

/*
 * tree_attn_prefix_pass / tree_attn_suffix_merge -- the two passes of
 * tree_attn_verify as separate calls (tree_attn_verify_ctas == prefix pass
 * then suffix merge, same arguments).  The prefix pass (the tree tokens
 * against the committed prefix, which needs no mask: pith.science review,
 * "What carries the argument") writes one partial result (running max m,
 * sum l, unnormalised accumulator acc, base-2 exponent domain) per split of
 * the prefix into `workspace`.  The suffix merge computes the tree part under
 * `mask` and merges it with every partial (merge_attentions over disjoint KV
 * chunks, verdict record supporting_citations) into out / lse.
 *
 * Both calls must see the same B, Hq, Hkv, d, T, page_size,
 * max_pages_per_seq, seq_lens contents, softmax_scale, n_ctas (<= 0: one per
 * SM) and workspace, in stream order.  Arguments, layouts, alignment and
 * return codes as for tree_attn_verify; the merge reads no K/V pages.
 */
TREE_ATTN_API int tree_attn_prefix_pass(const uint16_t *q, const uint16_t *k_pages,
                                        const uint16_t *v_pages, const int32_t *block_table,
                                        int max_pages_per_seq, const int32_t *seq_lens, int B,
                                        int Hq, int Hkv, int d, int T, int page_size,
                                        int num_pages, float softmax_scale, void *workspace,
                                        size_t workspace_bytes, int n_ctas, int32_t *status,
                                        void *stream);

TREE_ATTN_API int tree_attn_suffix_merge(const uint16_t *q, const int32_t *seq_lens,
                                         int max_pages_per_seq, const uint16_t *tree_k,
                                         const uint16_t *tree_v, const uint64_t *mask,
                                         uint16_t *out, float *lse, int B, int Hq, int Hkv, int d,
                                         int T, int page_size, float softmax_scale,
                                         const void *workspace, size_t workspace_bytes,
                                         int n_ctas, void *stream);

/*
 * tree_attn_verify_noalloc -- tree_attn_verify for callers that cannot
 * allocate device memory.  (The paper has no counterpart: this is a
 * deployment convenience of this library.)
 *
 * Some callers cannot call cudaMalloc at the point where they run attention:
 * code that runs inside a caller-managed memory pool with a fixed budget,
 * plug-ins of a host engine that forbids allocations after start-up, or
 * tools that must not grow the process's device footprint.  This entry point
 * takes the same inputs and outputs as tree_attn_verify but no workspace: the
 * per-split partial results go to a scratch array that is part of the
 * library itself (TREE_ATTN_NOALLOC_SCRATCH_BYTES, 16 MiB, reserved on every
 * GPU that loads the library until the process exits).
 *
 *   - Sizes whose partial results do not fit in the array are rejected with
 *     TREE_ATTN_ERR_SCRATCH_LIMIT (nothing is enqueued).  The need is
 *     (B*Hkv*ceil(T*Hq/Hkv/128) + SM count) * (256 + 128*d) * 4 bytes, e.g.
 *     a batch of 1 with 8 KV heads and d = 128 on 152 SMs needs 10.6 MB.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.  A cudaDeviceReset destroys the array's address
 *     with the context: the first call after a reset looks it up again, so
 *     make that call outside a capture too.  No call allocates or frees
 *     memory.
 *   - All calls share the one array and it keeps the previous call's
 *     contents; nothing in it needs to start at zero.  Calls that overlap on
 *     the GPU (e.g. on two streams at once) race on it and give wrong
 *     results: serialise them.
 * Arguments, layouts, alignment, status and other return codes as for
 * tree_attn_verify.
 */
#define TREE_ATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
#define TREE_ATTN_ERR_SCRATCH_LIMIT (-6) /* sizes exceed the built-in scratch array */

TREE_ATTN_API int tree_attn_verify_noalloc(const uint16_t *q, const uint16_t *k_pages,
                                           const uint16_t *v_pages, const int32_t *block_table,
                                           int max_pages_per_seq, const int32_t *seq_lens,
                                           const uint16_t *tree_k, const uint16_t *tree_v,
                                           const uint64_t *mask, uint16_t *out, float *lse,
                                           int B, int Hq, int Hkv, int d, int T, int page_size,
                                           int num_pages, float softmax_scale, int32_t *status,
                                           void *stream);

/*
 * tree_attn_set_wait_limit_ns -- limit of the prefix pass's internal waits.
 *
 * The prefix pass is a warp-specialised pipeline: a copy warp, an MMA warp
 * and softmax warps hand tiles to one another through shared-memory
 * barriers.  Every such wait is bounded: one that lasts longer than this
 * limit (nanoseconds of the GPU's global timer) makes the kernel store
 * TREE_ATTN_STATUS_TIMEOUT in *status, let its own copies and MMAs in flight
 * finish, free its tensor memory and return, so the CUDA context stays
 * usable (the call's out / lse are then unspecified).  The failure detection
 * this supports is a status word read on the host, never a trap.
 *
 *   ns   the new limit; 0 restores TREE_ATTN_DEFAULT_WAIT_NS (2 s).
 *
 * Returns the previous limit.  Process-wide; read when a call is enqueued,
 * so a CUDA graph keeps the value in force when it was captured.  A healthy
 * pipeline wait lasts microseconds: a short limit serves watchdogs and tests
 * of the timeout path (a call under a limit shorter than its waits reports
 * the timeout).  Host only; makes no CUDA call.
 */
#define TREE_ATTN_DEFAULT_WAIT_NS 2000000000ull

TREE_ATTN_API unsigned long long tree_attn_set_wait_limit_ns(unsigned long long ns);

/* Early start of the prefix pass (an opt-in promise about the stream).
 *
 * Every kernel of this library is launched with programmatic dependent
 * launch: its CTAs may start while the kernel before it in the stream is
 * still running, and wait for that kernel (griddepcontrol.wait) before they
 * read an input it may write.  By default the prefix pass waits before it
 * reads anything.
 *
 * Enabling this setting is the caller's promise that the kernel directly
 * before each later call in its stream writes none of seq_lens,
 * block_table and the committed-prefix rows of k_pages / v_pages (the
 * usual case: that kernel produces q and the tree tokens' K/V).  The prefix
 * pass then plans its work and issues the loads of its first ring stages of
 * committed-prefix K/V before that wait, overlapping them with the previous
 * kernel's tail; q, the tree K/V (also when padded into the paged cache),
 * the parent array and the masks are still read after the wait, and the
 * workspace is written only after it.  The one-pass explicit-mask form
 * (tree_attn_verify_dense) ignores the setting.  Results are the same
 * either way; a call whose promise does not hold may read stale prefix
 * data.  (Copies and memsets before a kernel complete before it starts
 * whatever the setting.  This library's kernels let their successor start
 * only after their own wait for the kernel before them; a kernel of the
 * caller's that signals its successor before its own wait extends the
 * promise to the kernels it may overlap.)
 *
 *   enable   non-zero to enable, 0 to disable (the default).
 *
 * Returns the previous setting (0 or 1).  Process-wide; read when a call is
 * enqueued, so a CUDA graph keeps the value in force when it was captured.
 * Host only; makes no CUDA call.
 */
TREE_ATTN_API int tree_attn_set_early_prefix_loads(int enable);

/* Library version, as major*10000 + minor*100 + patch. */
TREE_ATTN_API int tree_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TREE_ATTN_H */
