// Draft-side kernels: vocab-wide top-k of logits rows and best-first draft
// tree construction.
//
// Sources: "Tree spec-decode -> vLLM serve integration spec", "1. Proposer:
// emit top-K, not top-1" (top-W candidates per spine position); "From Linear to
// Tree-Walk: Validating DDTree's Core Algorithm in vLLM", "The Failed First
// Attempt" and "The Thinking Process" (best-first expansion on cumulative
// log-probability, node budget, top_k, draft horizon); "Technische
// Samenvatting: Trees from Marginals (DFlash-TfM)", "2. Boomconstructie" (pop
// the top w candidates per round).
//
// tv_topk: one thread block per row chunk (chunks only when there are too few
// rows to fill the GPU).  Every thread keeps its own sorted list of the 16 best
// (value, index) pairs it has seen in registers; a 16-byte vector is looked at
// element by element only when its packed maximum beats the list's last entry.
// The block then pulls its k best out of the thread lists in k rounds of a
// block-wide arg-max, and a second kernel merges the chunk lists of a row the
// same way.  Order: larger value first, equal values lower index first, NaN as
// -inf; an empty list slot is (-inf, INT32_MAX), which every real element of
// the row beats, so rows with fewer than k finite values still list real
// indices.
//
// tv_build_tree: one warp per sequence, all state in shared memory.  The
// candidate heap of the construction holds, for every expanded node, all K of
// its children; since each node's children come in non-increasing score order
// with increasing push counters, the best candidate among one node's children
// is always the first one not yet popped.  So the heap is kept as one cursor
// per expanded node (plus one for the roots), and a pop is a warp-wide arg-max
// over the cursors' current candidates (higher score, then lower push
// counter).  Scores are float32 sums added in depth order (__fadd_rn), the
// same additions the construction defines, so the tree is exact.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tv_draft.h"

namespace tv {

namespace {

constexpr int kTopThreads = 256;
constexpr int kTopList = TV_TOPK_MAX;  // entries per thread list
constexpr int kTopUnroll = 4;          // 16-byte loads in flight per thread

// a beats b: larger value, or equal value and lower index
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

struct TopList {
  float v[kTopList];
  int i[kTopList];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int j = 0; j < kTopList; ++j) {
      v[j] = -INFINITY;
      i[j] = INT32_MAX;
    }
  }
  // insert (x, xi) in order; NaN is -inf
  __device__ __forceinline__ void push(float x, int xi) {
    x = (x != x) ? -INFINITY : x;
    if (!beats(x, xi, v[kTopList - 1], i[kTopList - 1])) return;
    bool moved = false;
#pragma unroll
    for (int j = 0; j < kTopList; ++j) {
      const bool take = moved || beats(x, xi, v[j], i[j]);
      if (take) {
        const float tv = v[j];
        const int ti = i[j];
        v[j] = x;
        i[j] = xi;
        x = tv;
        xi = ti;
      }
      moved = take;
    }
  }
  // drop the head (after it won a round)
  __device__ __forceinline__ void pop_head() {
#pragma unroll
    for (int j = 0; j < kTopList - 1; ++j) {
      v[j] = v[j + 1];
      i[j] = i[j + 1];
    }
    v[kTopList - 1] = -INFINITY;
    i[kTopList - 1] = INT32_MAX;
  }
  // smallest entry that still matters: a candidate must beat it
  __device__ __forceinline__ bool full_above(float m) const {
    return !(m > v[kTopList - 1]) && i[kTopList - 1] != INT32_MAX;
  }
};

// One block-wide arg-max round over the thread lists' heads; every thread gets
// the winner.  Two barriers per round (kTopThreads threads).
__device__ __forceinline__ void block_best(const TopList &l, float &wv, int &wi) {
  __shared__ float sv[kTopThreads / 32];
  __shared__ int si[kTopThreads / 32];
  __shared__ float bv;
  __shared__ int bi;
  float v = l.v[0];
  int i = l.i[0];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (beats(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[w] = v;
    si[w] = i;
  }
  __syncthreads();
  if (w == 0) {
    v = lane < kTopThreads / 32 ? sv[lane] : -INFINITY;
    i = lane < kTopThreads / 32 ? si[lane] : INT32_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i, o);
      if (beats(ov, oi, v, i)) {
        v = ov;
        i = oi;
      }
    }
    if (lane == 0) {
      bv = v;
      bi = i;
    }
  }
  __syncthreads();
  wv = bv;
  wi = bi;
  __syncthreads();  // bv / bi are rewritten by the next round
}

__device__ __forceinline__ float elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float elem(const float *p) { return *p; }

template <typename T>
__device__ __forceinline__ float vec_max(const uint4 &w);
template <>
__device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4 &w) {
  uint32_t m2, n2;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(w.x), "r"(w.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(n2) : "r"(w.z), "r"(w.w));
  asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(n2));
  return fmaxf(bf16_lo(m2), bf16_hi(m2));
}
template <>
__device__ __forceinline__ float vec_max<float>(const uint4 &w) {
  return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
               fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
}

template <typename T>
__device__ __forceinline__ void push_vec(TopList &l, const uint4 &w, int i0);
template <>
__device__ __forceinline__ void push_vec<__nv_bfloat16>(TopList &l, const uint4 &w, int i0) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) l.push((k & 1) ? bf16_hi(ws[k >> 1]) : bf16_lo(ws[k >> 1]), i0 + k);
}
template <>
__device__ __forceinline__ void push_vec<float>(TopList &l, const uint4 &w, int i0) {
  l.push(__uint_as_float(w.x), i0);
  l.push(__uint_as_float(w.y), i0 + 1);
  l.push(__uint_as_float(w.z), i0 + 2);
  l.push(__uint_as_float(w.w), i0 + 3);
}

// grid.x = rows * chunks.  Writes the chunk's k best, in order, to
// (out_v, out_i) + blockIdx.x * k: the final answer when chunks == 1.
template <typename T>
__global__ void __launch_bounds__(kTopThreads)
topk_chunk_kernel(const T *__restrict__ x, int V, long long row_stride, int chunks, int chunk_len,
                  bool vec, int k, float *__restrict__ out_v, int32_t *__restrict__ out_i) {
  constexpr int E = 16 / sizeof(T);
  const long long row = blockIdx.x / chunks;
  const int c = blockIdx.x - (int)(row * chunks);
  const int begin = c * chunk_len;
  const int end = min(V, begin + chunk_len);
  const T *xr = x + row * row_stride;
  TopList l;
  l.init();
  int tail = begin;
  if (vec) {
    const int nvec = (end - begin) / E;
    const uint4 *xv = reinterpret_cast<const uint4 *>(xr + begin);
    for (int j0 = threadIdx.x; j0 < nvec; j0 += kTopThreads * kTopUnroll) {
      uint4 w[kTopUnroll];
#pragma unroll
      for (int u = 0; u < kTopUnroll; ++u) {
        const int j = j0 + u * kTopThreads;
        if (j < nvec) w[u] = __ldcs(xv + j);
      }
#pragma unroll
      for (int u = 0; u < kTopUnroll; ++u) {
        const int j = j0 + u * kTopThreads;
        if (j < nvec && !l.full_above(vec_max<T>(w[u]))) push_vec<T>(l, w[u], begin + j * E);
      }
    }
    tail = begin + nvec * E;
  }
  for (int i = tail + threadIdx.x; i < end; i += kTopThreads) l.push(elem(xr + i), i);
  for (int r = 0; r < k; ++r) {
    float wv;
    int wi;
    block_best(l, wv, wi);
    if (l.i[0] == wi && wi != INT32_MAX) l.pop_head();
    if (threadIdx.x == 0) {
      out_v[(size_t)blockIdx.x * k + r] = wv;
      out_i[(size_t)blockIdx.x * k + r] = wi;
    }
  }
}

// One block per row: merge the row's chunks * k candidates.
__global__ void __launch_bounds__(kTopThreads)
topk_merge_kernel(const float *__restrict__ part_v, const int32_t *__restrict__ part_i, int chunks,
                  int k, float *__restrict__ out_v, int32_t *__restrict__ out_i) {
  const long long row = blockIdx.x;
  const int n = chunks * k;
  TopList l;
  l.init();
  for (int j = threadIdx.x; j < n; j += kTopThreads)
    l.push(part_v[row * n + j], part_i[row * n + j]);
  for (int r = 0; r < k; ++r) {
    float wv;
    int wi;
    block_best(l, wv, wi);
    if (l.i[0] == wi && wi != INT32_MAX) l.pop_head();
    if (threadIdx.x == 0) {
      out_v[row * k + r] = wv;
      out_i[row * k + r] = wi;
    }
  }
}

struct TopkPlan {
  int chunks;
  int chunk_len;
};

TopkPlan plan_topk(long long rows, long long V, int esize) {
  const int E = 16 / esize;
  // a few thread blocks per SM; never cut a row below 32K elements
  const long long want = 8LL * sm_count();
  long long chunks = 1;
  if (rows < want) chunks = (want + rows - 1) / rows;
  const long long max_chunks = (V + 32767) / 32768;
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  long long len = (V + chunks - 1) / chunks;
  len = (len + E - 1) / E * E;
  chunks = (V + len - 1) / len;
  return TopkPlan{(int)chunks, (int)len};
}

// ------------------------------------------------------------------ build_tree

constexpr int kBtWarps = 4;
constexpr int kBtStreams = TV_MAX_NODES + 1;  // the roots' cursor + one per node
constexpr int kBtSlots = (kBtStreams + 31) / 32;

struct BtWarp {
  float node_score[TV_MAX_NODES];
  int node_tok[TV_MAX_NODES];
  int node_par[TV_MAX_NODES];
  int node_dep[TV_MAX_NODES];
  int next[kBtStreams];   // next child rank of the cursor, -1 while closed
  int cbase[kBtStreams];  // push counter of the cursor's rank-0 candidate
};

__global__ void __launch_bounds__(32 * kBtWarps)
build_tree_kernel(const float *__restrict__ cand_lp, const int32_t *__restrict__ cand_idx, int B,
                  int L, int K, int budget, int w, int32_t *__restrict__ tokens,
                  int32_t *__restrict__ parent, int32_t *__restrict__ depth,
                  float *__restrict__ score, int32_t *__restrict__ n_nodes) {
  __shared__ BtWarp sh[kBtWarps];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kBtWarps + wid;
  if (b >= B) return;
  BtWarp &s = sh[wid];
  const float *lp = cand_lp + (size_t)b * L * K;
  const int32_t *tk = cand_idx + (size_t)b * L * K;
  for (int j = lane; j < kBtStreams; j += 32) {
    s.next[j] = j == 0 ? 0 : -1;
    s.cbase[j] = 0;
  }
  __syncwarp();
  int counter = K;  // the K roots took counters 0 .. K-1
  int n = 0;
  while (n < budget) {
    const int start = n;
    const int take = min(w, budget - n);
    for (int q = 0; q < take; ++q) {
      // every lane evaluates its cursors; then a warp-wide arg-max
      float bs = -INFINITY;
      int bc = INT32_MAX, bstream = -1;
#pragma unroll
      for (int u = 0; u < kBtSlots; ++u) {
        const int st = lane + 32 * u;
        if (st >= kBtStreams) break;
        const int r = s.next[st];
        if (r < 0 || r >= K) continue;
        const int d = st == 0 ? 1 : s.node_dep[st - 1] + 1;  // candidate depth
        const float sc = st == 0 ? lp[r] : __fadd_rn(s.node_score[st - 1], lp[(size_t)(d - 1) * K + r]);
        const int cn = s.cbase[st] + r;
        if (bstream < 0 || sc > bs || (sc == bs && cn < bc)) {
          bs = sc;
          bc = cn;
          bstream = st;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, bs, o);
        const int oc = __shfl_xor_sync(0xffffffffu, bc, o);
        const int ost = __shfl_xor_sync(0xffffffffu, bstream, o);
        if (ost >= 0 && (bstream < 0 || os > bs || (os == bs && oc < bc))) {
          bs = os;
          bc = oc;
          bstream = ost;
        }
      }
      if (bstream < 0) break;  // the heap ran empty: the round ends early
      if (lane == 0) {
        const int r = s.next[bstream];
        const int d = bstream == 0 ? 1 : s.node_dep[bstream - 1] + 1;
        s.node_score[n] = bs;
        s.node_tok[n] = tk[(size_t)(d - 1) * K + r];
        s.node_par[n] = bstream - 1;
        s.node_dep[n] = d;
        s.next[bstream] = r + 1;
      }
      __syncwarp();
      ++n;
    }
    if (n == start) break;  // nothing left to pop: the K-ary tree of depth L is complete
    // after the round, the round's nodes push their children, in pop order
    if (lane == 0) {
      for (int t = start; t < n; ++t) {
        if (s.node_dep[t] < L) {
          s.next[t + 1] = 0;
          s.cbase[t + 1] = counter;
          counter += K;
        }
      }
    }
    counter = __shfl_sync(0xffffffffu, counter, 0);
    __syncwarp();
  }
  for (int t = lane; t < budget; t += 32) {
    const size_t o = (size_t)b * budget + t;
    const bool real = t < n;
    tokens[o] = real ? s.node_tok[t] : -1;
    parent[o] = real ? s.node_par[t] : -1;
    depth[o] = real ? s.node_dep[t] : 1;
    score[o] = real ? s.node_score[t] : -INFINITY;
  }
  if (lane == 0) n_nodes[b] = n;
}

}  // namespace

}  // namespace tv

using namespace tv;

extern "C" size_t tv_topk_workspace_size(int64_t rows, int64_t V, int k, int dtype) {
  if (rows <= 0 || V <= 0 || k < 1 || k > TV_TOPK_MAX) return 0;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const TopkPlan p = plan_topk(rows, V, esize);
  if (p.chunks == 1) return 0;
  const size_t n = (size_t)rows * p.chunks * k;
  return ((n * sizeof(float) + 255) / 256) * 256 + n * sizeof(int32_t);
}

extern "C" tv_status tv_topk(const void *x, int dtype, int64_t rows, int64_t V, int64_t row_stride,
                             int k, float *out_vals, int32_t *out_idx, void *workspace,
                             size_t workspace_bytes, tv_stream stream) {
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  if (rows < 0 || V < 1 || row_stride < V || V > INT32_MAX - 1024) return TV_ERR_ARG;
  if (k < 1 || k > TV_TOPK_MAX || k > V) return TV_ERR_ARG;
  if (rows == 0) return TV_OK;
  if (rows > (int64_t)INT32_MAX) return TV_ERR_ARG;
  if (!x || !out_vals || !out_idx) return TV_ERR_ARG;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const TopkPlan p = plan_topk(rows, V, esize);
  if ((long long)rows * p.chunks > (long long)INT32_MAX) return TV_ERR_ARG;
  float *pv = out_vals;
  int32_t *pi = out_idx;
  if (p.chunks > 1) {
    if (!workspace || workspace_bytes < tv_topk_workspace_size(rows, V, k, dtype)) return TV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return TV_ERR_ARG;
    const size_t n = (size_t)rows * p.chunks * k;
    pv = static_cast<float *>(workspace);
    pi = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                     ((n * sizeof(float) + 255) / 256) * 256);
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && ((row_stride * esize) % 16 == 0);
  const unsigned grid = (unsigned)(rows * p.chunks);
  cudaStream_t s = as_stream(stream);
  if (dtype == TV_BF16)
    topk_chunk_kernel<__nv_bfloat16><<<grid, kTopThreads, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(x), (int)V, row_stride, p.chunks, p.chunk_len, vec, k, pv,
        pi);
  else
    topk_chunk_kernel<float><<<grid, kTopThreads, 0, s>>>(static_cast<const float *>(x), (int)V,
                                                          row_stride, p.chunks, p.chunk_len, vec, k,
                                                          pv, pi);
  if (p.chunks > 1)
    topk_merge_kernel<<<(unsigned)rows, kTopThreads, 0, s>>>(pv, pi, p.chunks, k, out_vals, out_idx);
  return launch_status();
}

extern "C" tv_status tv_build_tree(const float *cand_lp, const int32_t *cand_idx, int B, int L, int K,
                                   int budget, int w, int32_t *tokens, int32_t *parent,
                                   int32_t *depth, float *score, int32_t *n_nodes,
                                   tv_stream stream) {
  if (B < 0 || L < 1 || L > 64 || K < 1 || K > 64 || budget < 1 || budget > TV_MAX_NODES || w < 1)
    return TV_ERR_ARG;
  if (B == 0) return TV_OK;
  if (!cand_lp || !cand_idx || !tokens || !parent || !depth || !score || !n_nodes)
    return TV_ERR_ARG;
  build_tree_kernel<<<(B + kBtWarps - 1) / kBtWarps, 32 * kBtWarps, 0, as_stream(stream)>>>(
      cand_lp, cand_idx, B, L, K, budget, w, tokens, parent, depth, score, n_nodes);
  return launch_status();
}
