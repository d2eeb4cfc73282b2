/*
 * tv_graph.h -- the whole verify step of an L-layer model as one unit, eager
 * or captured once into a CUDA graph and replayed.
 *
 * One step is
 *   tv_build_ancestors
 *   -> tv_tree_attention for every layer (its own q / k_tree / v_tree / caches)
 *   -> tv_argmax over the final logits -> tv_tree_walk
 *   -> tv_commit_kv for every layer (the same accepted nodes into every cache).
 * The commit is part of the step: in the graph form nothing runs eagerly
 * between two replays, which is what the GDN parity page, "Follow-up
 * (2026-06-22): ReplaySSM + XPU graph was fast but not valid", shows to be
 * needed -- there an eager state restore between captured decode replays
 * raced them and intermittently failed to take.  Sources for the step itself:
 * "Tree spec-decode -> vLLM serve integration spec", items 2 and 3 and
 * "Layout contract".
 *
 * Conventions are those of tv.h.  A graph records the pointers and sizes it
 * was created with: each replay reads and writes exactly those buffers, so the
 * caller refills the input buffers in place (on the replay stream, or with
 * ordering to it) between replays.  ctx_len and ctx_len_out are distinct
 * arrays, so replaying a step with unchanged inputs is idempotent.
 */
#ifndef TV_GRAPH_H_
#define TV_GRAPH_H_

#include "tv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One attention layer's buffers (layouts as in tv.h). */
typedef struct tv_layer {
  const void *q;        /* bf16 [B, N, Hq, D]  */
  const void *k_tree;   /* bf16 [B, N, Hkv, D] */
  const void *v_tree;   /* bf16 [B, N, Hkv, D] */
  void *k_cache;        /* bf16 [num_blocks, Hkv, 16, D], read, then committed into */
  void *v_cache;        /* bf16 [num_blocks, Hkv, 16, D]                             */
  void *out;            /* bf16 [B, N, Hq, D]  attention output                      */
} tv_layer;

typedef struct tv_step_args {
  /* tree and sequence state ([SPEC] "Layout contract") */
  const int32_t *tokens;       /* int32 [B, N] */
  const int32_t *parent;       /* int32 [B, N] */
  const int32_t *depth;        /* int32 [B, N] */
  const int32_t *ctx_len;      /* int32 [B]    */
  const int32_t *root_pred;    /* int32 [B]    */
  const int32_t *block_table;  /* int32 [B, max_blocks] */
  int B, N, Hq, Hkv, D, max_blocks, num_blocks;
  int window_left;             /* -1: global attention */
  float sm_scale;              /* 0: 1 / sqrt(D)       */
  /* the layers, attention scratch shared by all of them (they run in order) */
  int num_layers;
  const tv_layer *layers;      /* host array of num_layers entries, read at the call */
  void *attn_workspace;        /* >= tv_tree_attention_workspace_size of one layer */
  size_t attn_workspace_bytes;
  /* final logits and their argmax */
  const void *logits;          /* dtype [B * N, V], dense rows */
  int logits_dtype;            /* TV_BF16 or TV_F32 */
  int64_t V;
  void *argmax_workspace;      /* >= tv_argmax_workspace_size(B * N, V, dtype) */
  size_t argmax_workspace_bytes;
  /* outputs */
  uint64_t *anc;               /* [B, N] */
  int32_t *pos;                /* [B, N] */
  int32_t *status;             /* [B]    */
  int32_t *argmax;             /* [B, N] */
  int32_t *out_tokens;         /* [B, N + 1] */
  int32_t *n_emit;             /* [B] */
  int32_t *acc_nodes;          /* [B, N] */
  int32_t *n_acc;              /* [B] */
  int32_t *ctx_len_out;        /* [B] */
} tv_step_args;

/*
 * tv_verify_step -- enqueue one whole step on `stream` (eager launches).
 * Errors: those of the five calls (the first one that fails is returned and
 * nothing after it is enqueued); TV_ERR_ARG for num_layers < 1, NULL layers,
 * or ctx_len and ctx_len_out being the same array when num_layers > 1 (every
 * layer's commit reads ctx_len after the first has written ctx_len_out).
 */
tv_status tv_verify_step(const tv_step_args *a, tv_stream stream);

typedef struct tv_graph_s *tv_graph;

/*
 * tv_verify_graph_create -- capture one step (the same launches tv_verify_step
 * makes) into a CUDA graph on a private stream and instantiate it.  Nothing
 * runs.  The arguments are copied; `layers` need not outlive the call.
 * Errors: as tv_verify_step, or TV_ERR_CUDA if capture or instantiation fails
 * (then *out is NULL).
 */
tv_status tv_verify_graph_create(const tv_step_args *a, tv_graph *out);

/* Replay the captured step on `stream`.  TV_ERR_ARG for a NULL graph. */
tv_status tv_verify_graph_launch(tv_graph g, tv_stream stream);

/* Kernel launches one replay makes (what tv_verify_step enqueues). */
int tv_verify_graph_launches(tv_graph g);

/* Free the graph (after the replays that use it have completed). */
void tv_verify_graph_destroy(tv_graph g);

#ifdef __cplusplus
}
#endif

#endif /* TV_GRAPH_H_ */
