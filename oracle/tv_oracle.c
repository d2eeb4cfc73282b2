/*
 * CPU oracle for the tree speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: it is used by tests/, by __graft_entry__.smoke() and by bench.py's
 * CPU-baseline leg, to check and time the CUDA path against a plain, slow,
 * obviously correct restatement of what the verify step computes.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Source pages (cited by page title and section):
 *   [SPEC]   "Tree spec-decode -> vLLM serve integration spec":
 *            "What's proven", "2. Verify: tree attention mask",
 *            "3. Rejection sampler: tree walk", "Layout contract".
 *   [DDTREE] "From Linear to Tree-Walk: Validating DDTree's Core Algorithm in
 *            vLLM": "The Successful Test" (printed tree, mask shape).
 *
 * Precision: every floating-point step is fp64; bf16 inputs are widened
 * exactly (a bf16 value is the top 16 bits of an IEEE binary32).
 *
 * Pins (all in tests/, run with -m "not gpu"): ancestor masks against an
 * exhaustive transitive-closure enumeration for N <= 6 and the DDTree printed
 * tree; attention against a float64 library SDPA on chain / star / random
 * trees and windows; argmax against numpy's first-occurrence argmax and planted
 * ties; the walk against greedy decoding of a hash-defined target (the
 * greedy-identity property of [SPEC] "What's proven") and brute-force
 * maximality; the commit against a dense per-position gather of the cache.
 * No function here is "parity unpinned".
 *
 * Status codes (same numbering as the library's public header, restated here on
 * purpose so the two share nothing): 0 ok, 2 malformed tree, 3 bad block.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_TREE 2
#define OR_ERR_BLOCK 3

static double bf16_value(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Ancestor-or-self mask and position ids.
 * [SPEC] "2. Verify": node t may attend tree node a iff a is an ancestor of t
 * or t itself (additive bias 0, else -inf); position_ids[t] = ctx_len-1+depth(t).
 * [SPEC] "Layout contract": parent[t] is a node index, -1 meaning a child of
 * the last accepted token.  Reading taken: depth(t) = 1 when parent is -1,
 * else depth(parent)+1; parents precede children (parent[t] < t).
 *
 * mask  : uint8 [B, N, N], mask[b][t][a] = 1 iff a is ancestor-or-self of t
 * pos   : int32 [B, N]
 * status: int32 [B], 0 or OR_ERR_TREE (bad parent index or inconsistent depth)
 */
void oracle_ancestors(int B, int N, const int32_t *parent, const int32_t *depth,
                      const int32_t *ctx_len, uint8_t *mask, int32_t *pos,
                      int32_t *status) {
  for (int b = 0; b < B; ++b) {
    const int32_t *par = parent + (size_t)b * N;
    const int32_t *dep = depth + (size_t)b * N;
    int bad = 0;
    for (int t = 0; t < N; ++t) {
      int p = par[t];
      if (p < -1 || p >= t) { bad = 1; continue; }
      int want = (p < 0) ? 1 : dep[p] + 1;
      if (dep[t] != want) bad = 1;
    }
    status[b] = bad ? OR_ERR_TREE : OR_OK;
    for (int t = 0; t < N; ++t) {
      uint8_t *row = mask + ((size_t)b * N + t) * N;
      memset(row, 0, (size_t)N);
      row[t] = 1;
      /* follow parent pointers up to the last accepted token; at most N hops */
      int a = par[t];
      for (int hop = 0; hop < N && a >= 0 && a < N; ++hop) {
        row[a] = 1;
        a = par[a];
      }
      pos[(size_t)b * N + t] = ctx_len[b] - 1 + dep[t];
    }
  }
}

/*
 * Masked softmax attention of every tree node, by brute force.
 * [SPEC] "2. Verify": each node attends (a) all context keys of its sequence
 * (paged KV) and (b) its tree ancestors and itself; the mask composes with a
 * per-layer sliding window (left, right).
 *
 * Readings taken: scores are sm_scale * <q, k>; a key at position pk is inside
 * the window of a query at position pq iff pq - left <= pk (right side is
 * always satisfied, every allowed key precedes or equals the query); left < 0
 * means no window.  Head h reads KV head h / (Hq/Hkv).  Context key j sits in
 * cache block block_table[b][j / BS], row j % BS.
 *
 * Layouts (bf16 as raw uint16 bits):
 *   q        [B, N, Hq, D]
 *   k_tree   [B, N, Hkv, D], v_tree likewise
 *   k_cache  [num_blocks, Hkv, BS, D], v_cache likewise
 *   block_table int32 [B, max_blocks], ctx_len int32 [B]
 *   mask uint8 [B, N, N] and pos int32 [B, N] as from oracle_ancestors
 *   row_sel  uint8 [B * Hq] or NULL: compute only selected (b, h) rows
 *   out      fp64 [B, N, Hq, D] (rows not selected are left untouched)
 */
void oracle_attention(int B, int N, int Hq, int Hkv, int D, int BS, int max_blocks,
                      const uint16_t *q, const uint16_t *k_tree, const uint16_t *v_tree,
                      const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_table, const int32_t *ctx_len,
                      const uint8_t *mask, const int32_t *pos, int window_left,
                      double sm_scale, const uint8_t *row_sel, double *out) {
  const int G = Hq / Hkv;
  long long pairs = (long long)B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long bh = 0; bh < pairs; ++bh) {
    int b = (int)(bh / Hq), h = (int)(bh % Hq), kvh = h / G;
    if (row_sel && !row_sel[bh]) continue;
    int ctx = ctx_len[b];
    double *score = (double *)malloc(sizeof(double) * (size_t)(ctx + N + 1));
    const uint16_t **vrow = (const uint16_t **)malloc(sizeof(void *) * (size_t)(ctx + N + 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    for (int t = 0; t < N; ++t) {
      const uint16_t *qt = q + (((size_t)b * N + t) * Hq + h) * D;
      int pq = pos[(size_t)b * N + t];
      int nk = 0;
      /* (a) context keys, inside the window */
      for (int j = 0; j < ctx; ++j) {
        if (window_left >= 0 && j < pq - window_left) continue;
        int blk = block_table[(size_t)b * max_blocks + j / BS];
        size_t off = (((size_t)blk * Hkv + kvh) * BS + (size_t)(j % BS)) * D;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += bf16_value(qt[d]) * bf16_value(k_cache[off + d]);
        score[nk] = s * sm_scale;
        vrow[nk] = v_cache + off;
        ++nk;
      }
      /* (b) ancestor-or-self tree nodes, inside the window */
      const uint8_t *mrow = mask + ((size_t)b * N + t) * N;
      for (int a = 0; a < N; ++a) {
        if (!mrow[a]) continue;
        if (window_left >= 0 && pos[(size_t)b * N + a] < pq - window_left) continue;
        size_t off = (((size_t)b * N + a) * Hkv + kvh) * D;
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += bf16_value(qt[d]) * bf16_value(k_tree[off + d]);
        score[nk] = s * sm_scale;
        vrow[nk] = v_tree + off;
        ++nk;
      }
      /* softmax over the allowed keys, then the weighted sum of values */
      double m = -INFINITY;
      for (int i = 0; i < nk; ++i) if (score[i] > m) m = score[i];
      double l = 0.0;
      for (int d = 0; d < D; ++d) acc[d] = 0.0;
      for (int i = 0; i < nk; ++i) {
        double w = exp(score[i] - m);
        l += w;
        for (int d = 0; d < D; ++d) acc[d] += w * bf16_value(vrow[i][d]);
      }
      double *o = out + (((size_t)b * N + t) * Hq + h) * D;
      for (int d = 0; d < D; ++d) o[d] = (nk > 0) ? acc[d] / l : 0.0;
    }
    free(score);
    free(vrow);
    free(acc);
  }
}

/*
 * Row argmax with the lowest index winning ties.
 * [SPEC] "3. Rejection sampler": the walk consumes argmax(target_logits[t]).
 * Readings taken: ties go to the lowest index; +0 and -0 compare equal; a NaN
 * counts as -inf.  dtype 0 = float32, 1 = bf16.  row_stride in elements.
 */
void oracle_argmax(const void *x, int dtype, long long rows, long long V,
                   long long row_stride, int32_t *idx) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < rows; ++r) {
    double best = 0.0;
    long long bi = 0;
    for (long long i = 0; i < V; ++i) {
      double v;
      if (dtype == 0) v = (double)((const float *)x)[r * row_stride + i];
      else v = bf16_value(((const uint16_t *)x)[r * row_stride + i]);
      if (isnan(v)) v = -INFINITY;
      if (i == 0 || v > best) { best = v; bi = i; }
    }
    idx[r] = (int32_t)bi;
  }
}

/*
 * Greedy tree walk.
 * [SPEC] "What's proven" and "3. Rejection sampler": start at the root with
 * pred = the target's argmax there; while some child c of cur has token(c) ==
 * pred, emit token(c), move to c and take pred = argmax(logits[c]); finally
 * emit pred (the bonus token).
 * Readings taken: the root is the last accepted token, already in the cache;
 * its argmax is the input root_pred[b].  When several children carry pred the
 * lowest node index is taken.  A sequence whose status is non-zero emits only
 * root_pred.
 *
 * out_tokens [B, N+1] (unused tail = -1), n_emit [B], acc_nodes [B, N] (unused
 * tail = -1), n_acc [B].
 */
void oracle_walk(int B, int N, const int32_t *tokens, const int32_t *parent,
                 const int32_t *argmax, const int32_t *root_pred, const int32_t *status,
                 int32_t *out_tokens, int32_t *n_emit, int32_t *acc_nodes, int32_t *n_acc) {
  for (int b = 0; b < B; ++b) {
    const int32_t *tok = tokens + (size_t)b * N;
    const int32_t *par = parent + (size_t)b * N;
    const int32_t *am = argmax + (size_t)b * N;
    int32_t *ot = out_tokens + (size_t)b * (N + 1);
    int32_t *an = acc_nodes + (size_t)b * N;
    for (int i = 0; i <= N; ++i) ot[i] = -1;
    for (int i = 0; i < N; ++i) an[i] = -1;
    int k = 0;
    int cur = -1;
    int pred = root_pred[b];
    int ok = (status == NULL) || status[b] == 0;
    while (ok) {
      int child = -1;
      for (int c = 0; c < N; ++c) {
        if (par[c] == cur && tok[c] == pred) { child = c; break; }
      }
      if (child < 0) break;
      ot[k] = tok[child];
      an[k] = child;
      ++k;
      cur = child;
      pred = am[child];
      if (k >= N) break; /* a valid tree never gets here with a child left */
    }
    ot[k] = pred;
    n_acc[b] = k;
    n_emit[b] = k + 1;
  }
}

/*
 * Commit the accepted nodes' K/V into the paged cache.
 * [SPEC] "3. Rejection sampler": the accepted tokens and their KV are kept,
 * rejected branches are discarded.  Reading taken: the i-th accepted node (at
 * depth i+1) goes to position ctx_len[b] + i, i.e. its own position id; nothing
 * else is written; ctx_len_out = ctx_len + n_acc.  A sequence whose positions
 * need a block-table slot beyond max_blocks or a block id outside
 * [0, num_blocks) commits nothing and gets status OR_ERR_BLOCK.
 *
 * k_cache/v_cache are modified in place (raw uint16 bf16 bits).
 */
void oracle_commit(int B, int N, int Hkv, int D, int BS, int max_blocks, int num_blocks,
                   const uint16_t *k_tree, const uint16_t *v_tree,
                   const int32_t *acc_nodes, const int32_t *n_acc,
                   const int32_t *ctx_len_in, const int32_t *block_table,
                   uint16_t *k_cache, uint16_t *v_cache, int32_t *ctx_len_out,
                   int32_t *status) {
  for (int b = 0; b < B; ++b) {
    int n = n_acc[b];
    int ok = 1;
    for (int i = 0; i < n; ++i) {
      int p = ctx_len_in[b] + i;
      int slot = p / BS;
      if (slot >= max_blocks) { ok = 0; break; }
      int blk = block_table[(size_t)b * max_blocks + slot];
      if (blk < 0 || blk >= num_blocks) { ok = 0; break; }
    }
    if (!ok) {
      if (status) status[b] = OR_ERR_BLOCK;
      ctx_len_out[b] = ctx_len_in[b];
      continue;
    }
    for (int i = 0; i < n; ++i) {
      int c = acc_nodes[(size_t)b * N + i];
      int p = ctx_len_in[b] + i;
      int blk = block_table[(size_t)b * max_blocks + p / BS];
      for (int h = 0; h < Hkv; ++h) {
        size_t src = (((size_t)b * N + c) * Hkv + h) * D;
        size_t dst = (((size_t)blk * Hkv + h) * BS + (size_t)(p % BS)) * D;
        memcpy(k_cache + dst, k_tree + src, sizeof(uint16_t) * (size_t)D);
        memcpy(v_cache + dst, v_tree + src, sizeof(uint16_t) * (size_t)D);
      }
    }
    ctx_len_out[b] = ctx_len_in[b] + n;
  }
}
