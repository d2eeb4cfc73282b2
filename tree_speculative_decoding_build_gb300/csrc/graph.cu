// The whole verify step of an L-layer model: enqueued eagerly, or captured
// once into a CUDA graph (stream capture on a private stream) and replayed.
//
// Sources: "Tree spec-decode -> vLLM serve integration spec", items 2 and 3
// and "Layout contract" (the step); "Codex GDN Spec Parity Fix", "Follow-up
// (2026-06-22): ReplaySSM + XPU graph was fast but not valid" (eager work
// between graph replays raced them: here the commit is inside the graph).
#include <cuda_runtime.h>
#include <stdint.h>

#include <new>
#include <vector>

#include "common.cuh"
#include "tv_graph.h"

struct tv_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int launches = 0;
};

namespace tv {
namespace {

// Host checks of the step's own arguments (each call checks its own too).
tv_status check_step(const tv_step_args *a) {
  if (!a || a->num_layers < 1 || !a->layers) return TV_ERR_ARG;
  // every layer's commit reads ctx_len and writes ctx_len_out: one array for
  // both would make layer 2 onward commit its rows n_acc positions too far
  if (a->num_layers > 1 && a->ctx_len != nullptr &&
      static_cast<const void *>(a->ctx_len) == static_cast<const void *>(a->ctx_len_out))
    return TV_ERR_ARG;
  return TV_OK;
}

tv_status enqueue_step(const tv_step_args *a, cudaStream_t s) {
  const tv_status c = check_step(a);
  if (c != TV_OK) return c;
  const tv_stream st = reinterpret_cast<tv_stream>(s);
  tv_status r = tv_build_ancestors(a->parent, a->depth, a->ctx_len, a->B, a->N, a->anc, a->pos,
                                   a->status, st);
  if (r != TV_OK) return r;
  for (int l = 0; l < a->num_layers; ++l) {
    const tv_layer &ly = a->layers[l];
    tv_attn_args g = {};
    g.q = ly.q;
    g.k_tree = ly.k_tree;
    g.v_tree = ly.v_tree;
    g.k_cache = ly.k_cache;
    g.v_cache = ly.v_cache;
    g.block_table = a->block_table;
    g.ctx_len = a->ctx_len;
    g.pos = a->pos;
    g.anc = a->anc;
    g.B = a->B;
    g.N = a->N;
    g.Hq = a->Hq;
    g.Hkv = a->Hkv;
    g.D = a->D;
    g.block_size = TV_BLOCK_SIZE;
    g.max_blocks = a->max_blocks;
    g.num_blocks = a->num_blocks;
    g.window_left = a->window_left;
    g.window_right = 0;
    g.sm_scale = a->sm_scale;
    g.num_splits = 0;
    g.kernel = 0;
    g.out = ly.out;
    g.status = a->status;
    r = tv_tree_attention(&g, a->attn_workspace, a->attn_workspace_bytes, st);
    if (r != TV_OK) return r;
  }
  r = tv_argmax(a->logits, a->logits_dtype, (int64_t)a->B * a->N, a->V, a->V, a->argmax,
                a->argmax_workspace, a->argmax_workspace_bytes, st);
  if (r != TV_OK) return r;
  r = tv_tree_walk(a->tokens, a->parent, a->argmax, a->root_pred, a->status, a->B, a->N,
                   a->out_tokens, a->n_emit, a->acc_nodes, a->n_acc, st);
  if (r != TV_OK) return r;
  for (int l = 0; l < a->num_layers; ++l) {
    const tv_layer &ly = a->layers[l];
    r = tv_commit_kv(ly.k_tree, ly.v_tree, a->acc_nodes, a->n_acc, a->ctx_len, a->block_table,
                     a->B, a->N, a->Hkv, a->D, a->max_blocks, a->num_blocks, ly.k_cache, ly.v_cache,
                     a->ctx_len_out, a->status, st);
    if (r != TV_OK) return r;
  }
  return TV_OK;
}

int count_kernels(cudaGraph_t g) {
  size_t n = 0;
  if (cudaGraphGetNodes(g, nullptr, &n) != cudaSuccess || n == 0) return 0;
  std::vector<cudaGraphNode_t> nodes(n);
  if (cudaGraphGetNodes(g, nodes.data(), &n) != cudaSuccess) return 0;
  int k = 0;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++k;
  }
  return k;
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" tv_status tv_verify_step(const tv_step_args *a, tv_stream stream) {
  return enqueue_step(a, as_stream(stream));
}

extern "C" tv_status tv_verify_graph_create(const tv_step_args *a, tv_graph *out) {
  if (!out) return TV_ERR_ARG;
  *out = nullptr;
  const tv_status c = check_step(a);
  if (c != TV_OK) return c;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return TV_ERR_CUDA;
  tv_graph_s *g = new (std::nothrow) tv_graph_s;
  if (!g) {
    cudaStreamDestroy(cs);
    return TV_ERR_CUDA;
  }
  tv_status r = TV_OK;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    r = TV_ERR_CUDA;
  } else {
    r = enqueue_step(a, cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t e = cudaStreamEndCapture(cs, &graph);
    if (r == TV_OK && (e != cudaSuccess || !graph)) r = TV_ERR_CUDA;
    if (r == TV_OK) {
      g->graph = graph;
      g->launches = count_kernels(graph);
      if (cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) r = TV_ERR_CUDA;
    } else if (graph) {
      cudaGraphDestroy(graph);
    }
  }
  cudaGetLastError();  // a failed capture leaves its error here; it is reported as r
  cudaStreamDestroy(cs);
  if (r != TV_OK) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    return r;
  }
  *out = g;
  return TV_OK;
}

extern "C" tv_status tv_verify_graph_launch(tv_graph g, tv_stream stream) {
  if (!g || !g->exec) return TV_ERR_ARG;
  return cudaGraphLaunch(g->exec, as_stream(stream)) == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

extern "C" int tv_verify_graph_launches(tv_graph g) { return g ? g->launches : 0; }

extern "C" void tv_verify_graph_destroy(tv_graph g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}
