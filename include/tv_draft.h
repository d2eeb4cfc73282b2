/*
 * tv_draft.h -- draft-side companions of the verify step in libtv.so: the
 * vocab-wide top-k of logits rows and the best-first construction of the draft
 * tree that the verify step then checks.
 *
 *   tv_topk        -> per-depth candidate lists (or top-W per spine position)
 *   tv_build_tree  -> tokens[N], parent[N], depth[N] in the verify layout
 *
 * Source pages (cited by title and section):
 *   [SPEC]   "Tree spec-decode -> vLLM serve integration spec": "1. Proposer:
 *            emit top-K, not top-1" (top-W candidates per spine position),
 *            "Layout contract".
 *   [DDTREE] "From Linear to Tree-Walk: Validating DDTree's Core Algorithm in
 *            vLLM": "The Failed First Attempt", "The Thinking Process"
 *            (best-first expansion on cumulative log-probability with a
 *            priority queue, a node budget, top_k and a draft horizon).
 *   [TFM]    "Technische Samenvatting: Trees from Marginals (DFlash-TfM)":
 *            "2. Boomconstructie" (pop the top w candidates per round, so a
 *            tree of B nodes takes ceil(B / w) rounds).
 *
 * Conventions are those of tv.h: device pointers owned by the caller, nothing
 * allocated, every call only enqueues work on `stream`, the return value covers
 * host-side validation and launch errors.
 */
#ifndef TV_DRAFT_H_
#define TV_DRAFT_H_

#include "tv.h"

#ifdef __cplusplus
extern "C" {
#endif

#define TV_TOPK_MAX 16        /* largest k of tv_topk */

/*
 * Bytes of scratch tv_topk needs for `rows` rows of `V` values of `dtype` and
 * this k (0 when every row is reduced by one thread block).
 */
size_t tv_topk_workspace_size(int64_t rows, int64_t V, int k, int dtype);

/*
 * tv_topk -- the k largest values of every row and their indices.
 * [SPEC] item 1 (top-W per spine position); [DDTREE] "The Thinking Process"
 * (top_k candidates per draft position).
 *
 *   x          dtype [rows, row_stride] (TV_BF16 or TV_F32), first V used
 *   out_vals   float32 [rows, k]  the values, non-increasing along the row
 *                                 (bf16 widened exactly; a NaN reads -inf)
 *   out_idx    int32   [rows, k]  their indices: equal values keep the lower
 *                                 index first, and a NaN counts as -inf, so
 *                                 out_idx[r][0] is tv_argmax's answer
 *   workspace  >= tv_topk_workspace_size(rows, V, k, dtype) bytes, 16-aligned
 * Errors: TV_ERR_ARG (NULL pointers, k < 1, k > V, k > TV_TOPK_MAX,
 * row_stride < V, rows or V beyond int32 indexing, small workspace),
 * TV_ERR_UNSUPPORTED (other dtypes), TV_ERR_CUDA (launch failure).
 */
tv_status tv_topk(const void *x, int dtype, int64_t rows, int64_t V, int64_t row_stride, int k,
                  float *out_vals, int32_t *out_idx, void *workspace, size_t workspace_bytes,
                  tv_stream stream);

/*
 * tv_build_tree -- best-first draft tree of `budget` nodes from per-depth
 * candidate lists.  [DDTREE] "The Failed First Attempt"; [TFM] item 2.
 *
 * Depth d (1-based) of the draft has candidate tokens cand_idx[b][d-1][0..K-1]
 * with log-probabilities cand_lp[b][d-1][0..K-1], each list non-increasing (as
 * tv_topk returns them): one marginal per draft position.  A node's score is
 * the float32 sum of the log-probabilities along its path, added in depth order.
 * The candidate heap starts with the K depth-1 candidates (the roots); each
 * round pops the min(w, budget - n) best candidates (higher score first, equal
 * scores in push order; -0 and +0 are equal) and appends them as nodes in pop
 * order; after the round every popped node of depth < L pushes its K children
 * (the depth-(d+1) list), in pop order, each node's children in list order.  With w = 1 this is
 * the plain best-first (priority-queue) construction, and the tree is the
 * `budget` best-scoring nodes of the K-ary tree of depth L.
 *
 *   cand_lp    float32 [B, L, K]  log-probabilities, rows non-increasing, no NaN
 *   cand_idx   int32   [B, L, K]  token ids
 *   tokens     int32   [B, budget] out: node tokens in pop order
 *   parent     int32   [B, budget] out: parent node index (< the node's index),
 *                                  -1 for a depth-1 node (the [SPEC] "Layout
 *                                  contract": a child of the last accepted token)
 *   depth      int32   [B, budget] out: 1 + the parent's depth
 *   score      float32 [B, budget] out: cumulative log-probability
 *   n_nodes    int32   [B]        out: nodes built, budget unless the K-ary tree
 *                                  of depth L has fewer nodes; the slots past it
 *                                  hold token -1, parent -1, depth 1, score -inf
 * 1 <= budget <= TV_MAX_NODES, 1 <= K <= 64, 1 <= L <= 64, w >= 1.
 * Errors: TV_ERR_ARG (NULL pointers, sizes out of range), TV_ERR_CUDA.
 */
tv_status tv_build_tree(const float *cand_lp, const int32_t *cand_idx, int B, int L, int K,
                        int budget, int w, int32_t *tokens, int32_t *parent, int32_t *depth,
                        float *score, int32_t *n_nodes, tv_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TV_DRAFT_H_ */
