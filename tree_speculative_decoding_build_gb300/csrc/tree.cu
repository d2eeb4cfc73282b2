// Tree bookkeeping kernels: ancestor masks / position ids, the greedy walk and
// the KV commit.  All three are latency-bound (a few KB per sequence), so each
// sequence gets one warp (mask, walk) or one thread block (commit), with the
// per-sequence data kept in registers or shared memory.
//
// Source: "Tree spec-decode -> vLLM serve integration spec", sections
// "2. Verify: tree attention mask" (mask, position ids), "3. Rejection
// sampler: tree walk" (walk, commit) and "Layout contract" (tokens / parent /
// depth arrays, parent -1 = child of the last accepted token).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include <atomic>

#include "common.cuh"
#include "tv_debug.h"

TV_DEBUG_RECORD(tree)

namespace tv {

namespace {
std::atomic<int> g_withheld_cta{-1};
}  // namespace

int debug_withheld_cta() { return g_withheld_cta.load(std::memory_order_relaxed); }

int sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// One warp per sequence; lane l owns nodes l and l + 32.  anc[t] is built by
// following parent pointers, each hop strictly decreasing the node index, so
// the chase ends within N hops even on malformed input.
__global__ void build_ancestors_kernel(const int32_t *__restrict__ parent,
                                       const int32_t *__restrict__ depth,
                                       const int32_t *__restrict__ ctx_len, int B, int N,
                                       uint64_t *__restrict__ anc, int32_t *__restrict__ pos,
                                       int32_t *__restrict__ status) {
  // the tree-attention grids launched after this one may start at once: they
  // wait for this grid's completion before reading anc / pos / status
  pdl_launch_dependents();
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int32_t *par = parent + (size_t)b * N;
  const int32_t *dep = depth + (size_t)b * N;
  const int ctx = ctx_len[b];
  bool bad = false;
  for (int t = lane; t < N; t += 32) {
    const int p = par[t];
    bool ok = (p >= -1) && (p < t);
    if (ok) ok = dep[t] == (p < 0 ? 1 : dep[p] + 1);
    uint64_t m = 1ull << t;
    int cur = t, a = p;
    for (int hop = 0; hop < N && a >= 0 && a < cur; ++hop) {
      m |= 1ull << a;
      cur = a;
      a = par[a];
    }
    if (!ok) {
      bad = true;
      m = 1ull << t;
    }
    if (TV_CHECK(t >= 0 && t < N)) {
      anc[(size_t)b * N + t] = m;
      pos[(size_t)b * N + t] = ctx - 1 + dep[t];
    }
  }
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) status[b] = bad ? TV_ERR_TREE : TV_OK;
}

// One warp per sequence.  Each step is a ballot over the N nodes for
// "parent == cur && token == pred"; the lowest set bit is the child followed.
__global__ void tree_walk_kernel(const int32_t *__restrict__ tokens,
                                 const int32_t *__restrict__ parent,
                                 const int32_t *__restrict__ argmax,
                                 const int32_t *__restrict__ root_pred,
                                 const int32_t *__restrict__ status, int B, int N,
                                 int32_t *__restrict__ out_tokens, int32_t *__restrict__ n_emit,
                                 int32_t *__restrict__ acc_nodes, int32_t *__restrict__ n_acc) {
  // launched as a programmatic dependent: the commit grid after it may be
  // scheduled now; this grid's inputs are read after the wait
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int32_t path[4][kMaxNodes + 1];
  const int w = threadIdx.x >> 5;
  const int b = blockIdx.x * (blockDim.x >> 5) + w;
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const size_t base = (size_t)b * N;
  const int t0 = lane, t1 = lane + 32;
  const int par0 = t0 < N ? parent[base + t0] : -2;
  const int par1 = t1 < N ? parent[base + t1] : -2;
  const int tok0 = t0 < N ? tokens[base + t0] : 0;
  const int tok1 = t1 < N ? tokens[base + t1] : 0;
  const bool ok = (status == nullptr) || status[b] == 0;
  int cur = -1;
  int pred = root_pred[b];
  int k = 0;
  if (ok) {
    for (int it = 0; it < N; ++it) {
      const unsigned m0 = __ballot_sync(0xffffffffu, t0 < N && par0 == cur && tok0 == pred);
      const unsigned m1 = __ballot_sync(0xffffffffu, t1 < N && par1 == cur && tok1 == pred);
      const int c = m0 ? __ffs(m0) - 1 : (m1 ? 31 + __ffs(m1) : -1);
      if (c < 0) break;
      if (!TV_CHECK(c < N && k < N)) break;
      if (lane == 0) path[w][k] = c;
      ++k;
      cur = c;
      pred = argmax[base + c];
    }
  }
  __syncwarp();
  int32_t *ot = out_tokens + (size_t)b * (N + 1);
  int32_t *an = acc_nodes + base;
  for (int i = lane; i <= N; i += 32) {
    int v = -1;
    if (i < k && TV_CHECK(path[w][i] >= 0 && path[w][i] < N)) v = tokens[base + path[w][i]];
    else if (i == k) v = pred;
    ot[i] = v;
    if (i < N) an[i] = i < k ? path[w][i] : -1;
  }
  if (lane == 0) {
    n_acc[b] = k;
    n_emit[b] = k + 1;
  }
}

// One thread block per sequence: validate every destination slot first (a
// sequence commits all of its accepted rows or none), then copy 16-byte words.
__global__ void commit_kv_kernel(const uint4 *__restrict__ k_tree, const uint4 *__restrict__ v_tree,
                                 const int32_t *__restrict__ acc_nodes,
                                 const int32_t *__restrict__ n_acc,
                                 const int32_t *__restrict__ ctx_len_in,
                                 const int32_t *__restrict__ block_table, int N, int Hkv,
                                 int D, int max_blocks, int num_blocks, uint4 *__restrict__ k_cache,
                                 uint4 *__restrict__ v_cache, int32_t *__restrict__ ctx_len_out,
                                 int32_t *__restrict__ status) {
  // this grid's inputs are read after the wait.  It releases no dependent
  // early: a tree-attention grid launched after it reads the KV cache (which
  // this grid writes) before its own wait.
  pdl_wait();
  const int b = blockIdx.x;
  __shared__ int32_t s_blk[kMaxNodes];
  __shared__ int32_t s_node[kMaxNodes];
  const int n = n_acc[b];
  const int ctx = ctx_len_in[b];
  int bad = (n < 0 || n > N) ? 1 : 0;
  if (!bad) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const long long p = (long long)ctx + i;
      const long long slot = p >= 0 ? p / kBlock : -1;
      int blk = -1;
      if (slot >= 0 && slot < max_blocks) blk = block_table[(size_t)b * max_blocks + slot];
      const int c = acc_nodes[(size_t)b * N + i];
      if (blk < 0 || blk >= num_blocks || c < 0 || c >= N) bad = 1;
      s_blk[i] = blk;
      s_node[i] = c;
    }
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) {
      atomicCAS(status + b, 0, TV_ERR_BLOCK);
      ctx_len_out[b] = ctx;
    }
    return;
  }
  const int words = D / 8;                       // 16-byte words per head row
  const int per_row = Hkv * words;
  const int total = n * per_row;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int r = i / per_row;
    const int rem = i - r * per_row;
    const int h = rem / words;
    const int wd = rem - h * words;
    const int p = ctx + r;
    const size_t src = (((size_t)b * N + s_node[r]) * Hkv + h) * words + wd;
    const size_t dst = (((size_t)s_blk[r] * Hkv + h) * kBlock + (p % kBlock)) * words + wd;
    if (!TV_CHECK(src < (size_t)gridDim.x * N * Hkv * words &&
                  dst < (size_t)num_blocks * Hkv * kBlock * words && p >= 0))
      continue;
    k_cache[dst] = k_tree[src];
    v_cache[dst] = v_tree[src];
  }
  if (threadIdx.x == 0) ctx_len_out[b] = ctx + n;
}

}  // namespace tv

using namespace tv;

extern "C" const char *tv_status_string(tv_status s) {
  switch (s) {
    case TV_OK: return "ok";
    case TV_ERR_ARG: return "invalid argument";
    case TV_ERR_TREE: return "malformed tree (parent/depth)";
    case TV_ERR_BLOCK: return "block id or block-table slot out of range";
    case TV_ERR_CUDA: return "CUDA error";
    case TV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case TV_ERR_SCRATCH_LIMIT: return "size exceeds the fixed scratch of a no-allocation entry point";
    default: return "unknown status";
  }
}

extern "C" tv_status tv_build_ancestors(const int32_t *parent, const int32_t *depth,
                                        const int32_t *ctx_len, int B, int N, uint64_t *anc,
                                        int32_t *pos, int32_t *status, tv_stream stream) {
  if (B < 0 || N < 0 || N > kMaxNodes) return TV_ERR_ARG;
  if (B == 0) return TV_OK;
  if (!ctx_len || !status || (N > 0 && (!parent || !depth || !anc || !pos))) return TV_ERR_ARG;
  const int threads = 128;
  const int blocks = (B * 32 + threads - 1) / threads;
  build_ancestors_kernel<<<blocks, threads, 0, as_stream(stream)>>>(parent, depth, ctx_len, B, N,
                                                                   anc, pos, status);
  return launch_status();
}

extern "C" tv_status tv_tree_walk(const int32_t *tokens, const int32_t *parent,
                                  const int32_t *argmax, const int32_t *root_pred,
                                  const int32_t *status, int B, int N, int32_t *out_tokens,
                                  int32_t *n_emit, int32_t *acc_nodes, int32_t *n_acc,
                                  tv_stream stream) {
  if (B < 0 || N < 0 || N > kMaxNodes) return TV_ERR_ARG;
  if (B == 0) return TV_OK;
  if (!root_pred || !out_tokens || !n_emit || !n_acc) return TV_ERR_ARG;
  if (N > 0 && (!tokens || !parent || !argmax || !acc_nodes)) return TV_ERR_ARG;
  const int warps = 4;
  if (launch_pdl(tree_walk_kernel, dim3((B + warps - 1) / warps), dim3(warps * 32), 0,
                 as_stream(stream), tokens, parent, argmax, root_pred, status, B, N, out_tokens,
                 n_emit, acc_nodes, n_acc) != cudaSuccess)
    return TV_ERR_CUDA;
  return launch_status();
}

extern "C" tv_status tv_commit_kv(const void *k_tree, const void *v_tree, const int32_t *acc_nodes,
                                  const int32_t *n_acc, const int32_t *ctx_len_in,
                                  const int32_t *block_table, int B, int N, int Hkv, int D,
                                  int max_blocks, int num_blocks, void *k_cache, void *v_cache,
                                  int32_t *ctx_len_out, int32_t *status, tv_stream stream) {
  if (B < 0 || N < 0 || N > kMaxNodes || Hkv <= 0 || D <= 0 || max_blocks < 0 || num_blocks < 0)
    return TV_ERR_ARG;
  if (D % 8 != 0) return TV_ERR_UNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!n_acc || !ctx_len_in || !ctx_len_out || !status || !k_cache || !v_cache) return TV_ERR_ARG;
  if (N > 0 && (!k_tree || !v_tree || !acc_nodes)) return TV_ERR_ARG;
  if (max_blocks > 0 && !block_table) return TV_ERR_ARG;
  // 16-byte copies need 16-byte aligned bases (row strides are D*2 bytes, a multiple of 16)
  if ((reinterpret_cast<uintptr_t>(k_tree) | reinterpret_cast<uintptr_t>(v_tree) |
       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return TV_ERR_ARG;
  if (launch_pdl(commit_kv_kernel, dim3(B), dim3(256), 0, as_stream(stream),
                 static_cast<const uint4 *>(k_tree), static_cast<const uint4 *>(v_tree), acc_nodes,
                 n_acc, ctx_len_in, block_table, N, Hkv, D, max_blocks, num_blocks,
                 static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), ctx_len_out,
                 status) != cudaSuccess)
    return TV_ERR_CUDA;
  return launch_status();
}

extern "C" void tv_debug_withhold_arrival(int cta) {
  tv::g_withheld_cta.store(cta < 0 ? -1 : cta, std::memory_order_relaxed);
}

namespace tv {
unsigned debug_record_argmax(unsigned *, bool);
unsigned debug_record_attention(unsigned *, bool);
unsigned debug_record_attention_tc(unsigned *, bool);
unsigned debug_record_attention_tc256(unsigned *, bool);
unsigned debug_record_draft(unsigned *, bool);
unsigned debug_record_gdn(unsigned *, bool);
}  // namespace tv

extern "C" int tv_debug_checks_enabled(void) {
#ifdef TV_DEBUG
  return 1;
#else
  return 0;
#endif
}

extern "C" unsigned tv_debug_check_failures(unsigned *first_line, int *first_file, int clear) {
  unsigned (*const rec[])(unsigned *, bool) = {
      tv::debug_record_tree, tv::debug_record_argmax, tv::debug_record_attention,
      tv::debug_record_attention_tc, tv::debug_record_attention_tc256, tv::debug_record_draft,
      tv::debug_record_gdn};
  unsigned total = 0, line = 0;
  int file = -1;
  for (int i = 0; i < (int)(sizeof(rec) / sizeof(rec[0])); ++i) {
    unsigned l = 0;
    const unsigned n = rec[i](&l, clear != 0);
    if (n == ~0u) return ~0u;
    if (n > 0 && file < 0) {
      file = i;
      line = l;
    }
    total += n;
  }
  if (first_line) *first_line = line;
  if (first_file) *first_file = file;
  return total;
}
