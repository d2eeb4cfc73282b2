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
// tv_topk: every warp keeps a sorted list of its 32 best (value, index) pairs
// spread over its lanes.  A lane's 16-byte vector is looked at element by
// element only when its packed maximum beats the list's k-th entry, so after
// the first few hundred elements almost no vector is examined and the scan
// runs at memory speed.  Two plans:
//  - chunk plan (strided or unaligned rows, small inputs): one thread block
//    per row chunk, each warp a contiguous eighth of it; a ballot hands a
//    passing vector to the whole warp, which inserts its winning elements;
//    warp 0 folds the block's lists and a one-warp-per-row kernel the chunks'.
//  - stream plan (dense aligned rows): one contiguous range per warp of a
//    one-CTA-per-SM grid (below).
// Order: larger value first, equal values lower index first, NaN as -inf; an
// empty slot is (-inf, INT32_MAX), which every real element of the row beats,
// so rows with fewer than k finite values still list real indices.
//
// tv_build_tree: one warp per sequence.  The candidate heap of the
// construction holds, for every expanded node, all K of its children; since
// each node's children come in non-increasing score order with increasing push
// counters, the best candidate among one node's children is always the first
// one not yet popped.  So the heap is kept as one cursor per expanded node
// (plus one for the roots), spread over the lanes with each cursor's current
// candidate in registers, and a pop is a warp-wide arg-max: one redux.max over
// an order-preserving key of the score, one redux.min over the push counters
// of the lanes that hold that score.  Scores are float32 sums added in depth
// order (__fadd_rn), the same additions the construction defines, so the tree
// is exact.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tv_draft.h"

TV_DEBUG_RECORD(draft)

namespace tv {

namespace {

constexpr int kTopWarps = 8;
constexpr int kTopThreads = 32 * kTopWarps;
constexpr int kTopUnroll = 4;  // 16-byte loads in flight per lane

// a beats b: larger value, or equal value and lower index
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// A warp's sorted list of its 32 best (value, index) pairs, lane j holding the
// j-th; an empty slot is (-inf, INT32_MAX).  Insertion is warp-wide: x / xi
// must be the same in every lane.
__device__ __forceinline__ void wl_insert(float &lv, int &li, float x, int xi) {
  const bool gt = beats(x, xi, lv, li);
  const unsigned m = __ballot_sync(0xffffffffu, gt);
  if (m == 0) return;
  const int p = __ffs(m) - 1;  // the list is sorted: every lane from p on is beaten
  const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
  const int ui = __shfl_up_sync(0xffffffffu, li, 1);
  const int lane = threadIdx.x & 31;
  if (lane > p) {
    lv = uv;
    li = ui;
  } else if (lane == p) {
    lv = x;
    li = xi;
  }
}

__device__ __forceinline__ float elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float elem(const float *p) { return *p; }

// Packed maximum of a 16-byte vector (a NaN operand is ignored).
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

// Element e of a 16-byte vector.
template <typename T>
__device__ __forceinline__ float vec_elem(const uint4 &w, int e);
template <>
__device__ __forceinline__ float vec_elem<__nv_bfloat16>(const uint4 &w, int e) {
  const uint32_t h = (e >> 1) == 0 ? w.x : (e >> 1) == 1 ? w.y : (e >> 1) == 2 ? w.z : w.w;
  return (e & 1) ? bf16_hi(h) : bf16_lo(h);
}
template <>
__device__ __forceinline__ float vec_elem<float>(const uint4 &w, int e) {
  return __uint_as_float(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
}

// Order-preserving int key of a non-NaN float (for a block-wide atomicMax).
__device__ __forceinline__ int fkey(float f) {
  const int b = __float_as_int(f);
  return b ^ ((b >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float fkey_inv(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7fffffff)); }

// Lanes flagged in `ballot` hand their vector to the whole warp, one lane at a
// time in lane order, and its elements that beat the k-th entry go in.
template <typename T>
__device__ __forceinline__ void take_flagged(unsigned ballot, const uint4 &q, int idx0, int k,
                                             float &lv, int &li, float &tv, int &ti) {
  constexpr int E = 16 / sizeof(T);
  while (ballot) {
    const int src = __ffs(ballot) - 1;
    ballot &= ballot - 1;
    uint4 w;
    w.x = __shfl_sync(0xffffffffu, q.x, src);
    w.y = __shfl_sync(0xffffffffu, q.y, src);
    w.z = __shfl_sync(0xffffffffu, q.z, src);
    w.w = __shfl_sync(0xffffffffu, q.w, src);
    const int i0 = __shfl_sync(0xffffffffu, idx0, src);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float x = vec_elem<T>(w, e);
      x = (x != x) ? -INFINITY : x;
      if (beats(x, i0 + e, tv, ti)) {
        wl_insert(lv, li, x, i0 + e);
        tv = __shfl_sync(0xffffffffu, lv, k - 1);
        ti = __shfl_sync(0xffffffffu, li, k - 1);
      }
    }
  }
}

// Maximum of a lane's whole load batch (NaN elements ignored): the vectors
// are folded element-wise first, so the batch costs one horizontal maximum.
template <typename T, int U>
__device__ __forceinline__ float batch_max(const uint4 (&q)[U]) {
  uint4 m = q[0];
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int u = 1; u < U; ++u) {
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m.x) : "r"(q[u].x));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m.y) : "r"(q[u].y));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m.z) : "r"(q[u].z));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m.w) : "r"(q[u].w));
    }
  } else {
#pragma unroll
    for (int u = 1; u < U; ++u) {
      m.x = __float_as_uint(fmaxf(__uint_as_float(m.x), __uint_as_float(q[u].x)));
      m.y = __float_as_uint(fmaxf(__uint_as_float(m.y), __uint_as_float(q[u].y)));
      m.z = __float_as_uint(fmaxf(__uint_as_float(m.z), __uint_as_float(q[u].z)));
      m.w = __float_as_uint(fmaxf(__uint_as_float(m.w), __uint_as_float(q[u].w)));
    }
  }
  return vec_max<T>(m);
}

// Lanes with `flag` set hold a vector whose maximum may enter the list.  Each
// such lane marks, by itself, its elements that beat the k-th entry; the warp
// then takes the marked elements one at a time (lowest lane first, then lowest
// element), broadcasting only that pair.  The new k-th entry needs no second
// shuffle: an insert at position p < k-1 moves the old (k-2)-th entry into
// place k-1, read in the same step as the insert.  A marked element that no
// longer beats the k-th entry when its turn comes is dropped, and so is the
// lane's element `excl` (already in the list).
template <typename T>
__device__ __forceinline__ void take_own(bool flag, const uint4 &q, int idx0, int excl, int k,
                                         float &lv, int &li, float &tv, int &ti) {
  constexpr int E = 16 / sizeof(T);
  const int lane = threadIdx.x & 31;
  unsigned cm = 0;
  if (flag) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float x = vec_elem<T>(q, e);
      x = (x != x) ? -INFINITY : x;
      if (idx0 + e != excl && beats(x, idx0 + e, tv, ti)) cm |= 1u << e;
    }
  }
  unsigned who = __ballot_sync(0xffffffffu, cm != 0);
  while (who) {
    const int src = __ffs(who) - 1;
    // this lane's lowest marked element
    const int e = __ffs(cm) - 1;
    float x = -INFINITY;
#pragma unroll
    for (int ee = 0; ee < E; ++ee)
      if (ee == e) x = vec_elem<T>(q, ee);
    x = (x != x) ? -INFINITY : x;
    const float bx = __shfl_sync(0xffffffffu, x, src);
    const int bi = __shfl_sync(0xffffffffu, idx0 + e, src);
    if (lane == src) cm &= cm - 1;
    const float t2v = __shfl_sync(0xffffffffu, lv, k >= 2 ? k - 2 : 0);
    const int t2i = __shfl_sync(0xffffffffu, li, k >= 2 ? k - 2 : 0);
    if (beats(bx, bi, tv, ti)) {
      const unsigned m = __ballot_sync(0xffffffffu, beats(bx, bi, lv, li));
      const int p = __ffs(m) - 1;  // m != 0: lane k-1 at least is beaten
      const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
      const int ui = __shfl_up_sync(0xffffffffu, li, 1);
      if (lane > p) {
        lv = uv;
        li = ui;
      } else if (lane == p) {
        lv = bx;
        li = bi;
      }
      if (p < k - 1) {
        tv = t2v;
        ti = t2i;
      } else {
        tv = bx;
        ti = bi;
      }
    }
    who = __ballot_sync(0xffffffffu, cm != 0);
  }
}

// One compare-exchange step of a 32-lane network over (value, index) pairs:
// this lane ends up with the better pair when keep_better, else the worse.
__device__ __forceinline__ void cx_step(float &v, int &i, int stride, bool keep_better) {
  const float ov = __shfl_xor_sync(0xffffffffu, v, stride);
  const int oi = __shfl_xor_sync(0xffffffffu, i, stride);
  if (keep_better ? beats(ov, oi, v, i) : beats(v, i, ov, oi)) {
    v = ov;
    i = oi;
  }
}

// Fold 32 candidates, one per lane, into the warp's sorted list (lane 0 the
// best): bitonic sort of the candidates into ascending order, the better of
// list[j] and candidate[j] in each lane (the 32 best of both, a bitonic
// sequence), then a bitonic merge back into descending order.
__device__ __forceinline__ void fold32(float &lv, int &li, float cv, int ci) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
      // ascending blocks where lane & size == 0 (all of them at size 32)
      cx_step(cv, ci, stride, ((lane & stride) != 0) == ((lane & size) == 0));
  if (beats(cv, ci, lv, li)) {
    lv = cv;
    li = ci;
  }
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) cx_step(lv, li, stride, (lane & stride) == 0);
}

// The warp's list at the end of a block: warp 0 folds the warps' k best
// (kTopWarps * k candidates, 32 at a time) and returns the block's k best in
// its lanes 0 .. k-1.
__device__ __forceinline__ void block_fold(float &lv, int &li, int k) {
  __shared__ float sv[kTopWarps][32];
  __shared__ int si[kTopWarps][32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  sv[w][lane] = lv;
  si[w][lane] = li;
  __syncthreads();
  if (w == 0) {
    float fv = -INFINITY;
    int fi = INT32_MAX;
    for (int q0 = 0; q0 < kTopWarps * k; q0 += 32) {
      const int j = q0 + lane;
      float x = -INFINITY;
      int xi = INT32_MAX;
      if (j < kTopWarps * k) {
        x = sv[j / k][j % k];
        xi = si[j / k][j % k];
      }
      fold32(fv, fi, x, xi);
    }
    lv = fv;
    li = fi;
  }
}

// grid.x = rows * chunks; warp w of a block scans the w-th eighth of the
// chunk, so each warp sees its indices in increasing order.  Writes the
// chunk's k best to (out_v, out_i) + blockIdx.x * k: the final answer when
// chunks == 1.
template <typename T>
__global__ void __launch_bounds__(kTopThreads)
topk_chunk_kernel(const T *__restrict__ x, int V, long long row_stride, int chunks, int chunk_len,
                  bool vec, int k, float *__restrict__ out_v, int32_t *__restrict__ out_i) {
  pdl_launch_dependents();  // the merge grid may be scheduled now: it waits for this one
  constexpr int E = 16 / sizeof(T);
  const long long row = blockIdx.x / chunks;
  const int c = blockIdx.x - (int)(row * chunks);
  const int begin = c * chunk_len;
  const int end = min(V, begin + chunk_len);
  const T *xr = x + row * row_stride;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT32_MAX, ti = INT32_MAX;  // (tv, ti): the k-th entry, the bar to beat
  // The block's bar: the largest k-th entry of any warp whose list holds k real
  // entries.  No value below it can be among the chunk's k best (that warp
  // already has k values at least as large), so every warp may skip such values.
  __shared__ int s_bar;
  if (threadIdx.x == 0) s_bar = fkey(-INFINITY);
  __syncthreads();
  if (vec) {
    // items are 16-byte vectors; the warp's share is a contiguous run of them
    const int nvec = (end - begin) / E;
    const int w0 = (int)((long long)nvec * w / kTopWarps);
    const int w1 = (int)((long long)nvec * (w + 1) / kTopWarps);
    const uint4 *xv = reinterpret_cast<const uint4 *>(xr + begin);
    bool fresh = true;  // the list does not hold k entries yet
    for (int b0 = w0; b0 < w1; b0 += 32 * kTopUnroll) {
      uint4 q[kTopUnroll];
#pragma unroll
      for (int u = 0; u < kTopUnroll; ++u) {
        const int j = b0 + lane + 32 * u;
        if (j < w1) q[u] = __ldcs(xv + j);
      }
      const float bar = fkey_inv(*(volatile int *)&s_bar);
      if (fresh) {
        // A list short of k entries would take nearly every element as an
        // insert of its own.  Each lane's best element of the batch goes in by
        // one fold instead (32 candidates at once), as in the streaming plan;
        // the lanes' other elements then go through take_own, which skips the
        // one already in (excl).  A vector whose maximum ties the k-th entry
        // may still hold a lower index that beats it, so ties are examined too.
        float lm = -INFINITY;
        int im = INT32_MAX;
#pragma unroll
        for (int u = 0; u < kTopUnroll; ++u) {
          const int j = b0 + lane + 32 * u;
          if (j < w1) {
            const float m = vec_max<T>(q[u]);
            if (m > lm) {  // the earliest vector holding the lane's maximum
              int e = E - 1;
#pragma unroll
              for (int ee = E - 1; ee >= 0; --ee)
                if (vec_elem<T>(q[u], ee) == m) e = ee;
              lm = m;
              im = begin + j * E + e;
            }
          }
        }
        fold32(lv, li, lm, im);
        tv = __shfl_sync(0xffffffffu, lv, k - 1);
        ti = __shfl_sync(0xffffffffu, li, k - 1);
#pragma unroll
        for (int u = 0; u < kTopUnroll; ++u) {
          const int j = b0 + lane + 32 * u;
          const float m = vec_max<T>(q[u]);
          const bool flag = j < w1 && (m >= tv || ti == INT32_MAX) && !(m < bar);
          const unsigned ballot = __ballot_sync(0xffffffffu, flag);
          if (ballot) take_own<T>(flag, q[u], begin + j * E, im, k, lv, li, tv, ti);
        }
        fresh = ti == INT32_MAX;
      } else {
#pragma unroll
        for (int u = 0; u < kTopUnroll; ++u) {
          const int j = b0 + lane + 32 * u;
          const float m = vec_max<T>(q[u]);
          const bool flag = j < w1 && (m > tv || ti == INT32_MAX) && !(m < bar);
          const unsigned ballot = __ballot_sync(0xffffffffu, flag);
          if (ballot) take_flagged<T>(ballot, q[u], begin + j * E, k, lv, li, tv, ti);
        }
      }
      if (lane == 0 && ti != INT32_MAX) atomicMax(&s_bar, fkey(tv));
    }
    // the tail that does not fill a vector: warp 0, one element per lane
    if (w == 0) {
      for (int t0 = begin + nvec * E; t0 < end; t0 += 32) {
        const int i = t0 + lane;
        float xv1 = i < end ? elem(xr + i) : -INFINITY;
        xv1 = (xv1 != xv1) ? -INFINITY : xv1;
        const bool flag = i < end && beats(xv1, i, tv, ti);
        unsigned ballot = __ballot_sync(0xffffffffu, flag);
        while (ballot) {
          const int src = __ffs(ballot) - 1;
          ballot &= ballot - 1;
          const float y = __shfl_sync(0xffffffffu, xv1, src);
          const int yi = __shfl_sync(0xffffffffu, i, src);
          if (beats(y, yi, tv, ti)) {
            wl_insert(lv, li, y, yi);
            tv = __shfl_sync(0xffffffffu, lv, k - 1);
            ti = __shfl_sync(0xffffffffu, li, k - 1);
          }
        }
      }
    }
  } else {
    // unaligned rows: one element per lane per step, contiguous run per warp
    const int n = end - begin;
    const int w0 = begin + (int)((long long)n * w / kTopWarps);
    const int w1 = begin + (int)((long long)n * (w + 1) / kTopWarps);
    for (int t0 = w0; t0 < w1; t0 += 32) {
      const int i = t0 + lane;
      float xv1 = i < w1 ? elem(xr + i) : -INFINITY;
      xv1 = (xv1 != xv1) ? -INFINITY : xv1;
      const bool flag = i < w1 && beats(xv1, i, tv, ti);
      unsigned ballot = __ballot_sync(0xffffffffu, flag);
      while (ballot) {
        const int src = __ffs(ballot) - 1;
        ballot &= ballot - 1;
        const float y = __shfl_sync(0xffffffffu, xv1, src);
        const int yi = __shfl_sync(0xffffffffu, i, src);
        if (beats(y, yi, tv, ti)) {
          wl_insert(lv, li, y, yi);
          tv = __shfl_sync(0xffffffffu, lv, k - 1);
          ti = __shfl_sync(0xffffffffu, li, k - 1);
        }
      }
    }
  }
  block_fold(lv, li, k);
  if (w == 0 && lane < k && TV_CHECK(li == INT32_MAX || (li >= 0 && li < V))) {
    out_v[(size_t)blockIdx.x * k + lane] = lv;
    out_i[(size_t)blockIdx.x * k + lane] = li;
  }
}

// One block per row: its warps fold the row's chunks * k candidates (warp w a
// w-th share, 32 at a time), then warp 0 folds the warps' k best.  Launched as
// a programmatic dependent of the chunk grid: the partials are read after the
// wait.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(32 * kMergeWarps)
topk_merge_kernel(const float *__restrict__ part_v, const int32_t *__restrict__ part_i,
                  long long rows, int chunks, int k, float *__restrict__ out_v,
                  int32_t *__restrict__ out_i) {
  pdl_wait();
  __shared__ float sv[kMergeWarps][32];
  __shared__ int si[kMergeWarps][32];
  const long long row = blockIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int n = chunks * k;
  const int j0 = (int)((long long)n * w / kMergeWarps), j1 = (int)((long long)n * (w + 1) / kMergeWarps);
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT32_MAX, ti = INT32_MAX;
  for (int q0 = j0; q0 < j1; q0 += 32) {
    const int j = q0 + lane;
    float x = -INFINITY;
    int xi = INT32_MAX;
    if (j < j1) {
      x = part_v[row * n + j];
      xi = part_i[row * n + j];
    }
    if (!__any_sync(0xffffffffu, xi != INT32_MAX && beats(x, xi, tv, ti))) continue;
    fold32(lv, li, x, xi);
    tv = __shfl_sync(0xffffffffu, lv, k - 1);
    ti = __shfl_sync(0xffffffffu, li, k - 1);
  }
  sv[w][lane] = lv;
  si[w][lane] = li;
  __syncthreads();
  if (w != 0) return;
  float fv = -INFINITY;
  int fi = INT32_MAX;
  for (int q0 = 0; q0 < kMergeWarps * k; q0 += 32) {  // the warps' k best, 32 at a time
    const int j = q0 + lane;
    float x = -INFINITY;
    int xi = INT32_MAX;
    if (j < kMergeWarps * k) {
      x = sv[j / k][j % k];
      xi = si[j / k][j % k];
    }
    fold32(fv, fi, x, xi);
  }
  if (lane < k) {
    out_v[row * k + lane] = fv;
    out_i[row * k + lane] = fi;
  }
}

// Order-preserving unsigned key of a non-NaN float; 0 is below every float.
// -0 keys as +0: the two compare equal, so a tie between them goes to the
// push counter.
__device__ __forceinline__ unsigned score_key(float f) {
  unsigned b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ------------------------------------------------------------------ stream plan
//
// Dense, aligned rows: the flattened [rows x V] array is cut into equal
// contiguous ranges, one per warp of a one-CTA-per-SM grid (the argmax stream
// plan with a k-list instead of one pair), so every SM moves the same bytes
// and there is no tail wave.  A warp's list covers the piece of the current
// row inside its range; at a row end the list is written (a row lying whole in
// the range goes straight to the output, the range's first and last pieces to
// slots 2w and 2w+1), and a merge kernel folds the pieces of the rows cut by
// range boundaries.
//
// The cost beyond the loads is the inserts, each a chain of warp shuffles
// (hundreds of cycles while the loads of 15 other warps share the SM), and a
// warp that inserts much finishes late: its range is fixed.  So:
//  - a row piece starts with one bitonic fold of the 32 lanes' maxima into the
//    list (instead of a dozen single inserts), whose k-th entry then bounds
//    the piece's k-th largest value from below (bar);
//  - a whole batch inside the row is skipped by one vote on the lanes' batch
//    maxima when none beats the k-th entry;
//  - an insert broadcasts only the winning element: the lane that holds it
//    finds it by itself.

constexpr int kTsWarps = 16;   // warps per CTA
constexpr int kTsUnroll = 8;   // 16-byte loads per lane per batch (two batches in flight)

// The split weighs row starts: each row counts as `pen` empty slots followed
// by its vpr vectors, and the virtual total tot = rows * (vpr + pen) is cut
// evenly, so a warp whose range holds a row start (a second row piece, with
// its own list to build) is given pen fewer vectors.  First vector of warp w:
__device__ __forceinline__ long long ts_split(long long w, long long vpr, long long pen,
                                              long long tot, long long owners) {
  const long long y = w * tot / owners;
  const long long row = y / (vpr + pen), off = y - row * (vpr + pen);
  return row * vpr + (off > pen ? off - pen : 0);
}
// The warp whose range holds vector x: the last w with split(w) <= x.
__device__ __forceinline__ long long ts_owner(long long x, long long vpr, long long pen,
                                              long long tot, long long owners) {
  const long long row = x / vpr;
  const long long y = row * (vpr + pen) + pen + (x - row * vpr);
  return ((y + 1) * owners + tot - 1) / tot - 1;  // ceil((y + 1) * owners / tot) - 1
}

template <typename T>
__global__ void __launch_bounds__(32 * kTsWarps, 1)
topk_stream_kernel(const T *__restrict__ x, long long vpr, long long pen, long long tot,
                   long long owners, int k,
                   float *__restrict__ part_v, int32_t *__restrict__ part_i,
                   float *__restrict__ out_v, int32_t *__restrict__ out_i) {
  constexpr int E = 16 / sizeof(T);
  constexpr int kBatch = 32 * kTsUnroll;
  // the merge grid may be launched now: it waits for this grid's completion
  // before it reads the partial lists
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kTsWarps + (threadIdx.x >> 5);
  if (w >= owners) return;
  const long long v0 = ts_split(w, vpr, pen, tot, owners);
  const long long v1 = ts_split(w + 1, vpr, pen, tot, owners);
  const uint4 *xv = reinterpret_cast<const uint4 *>(x);
  long long r = v0 / vpr, rs = r * vpr;
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT32_MAX, ti = INT32_MAX;
  // bar: a lower bound of the current row piece's k-th largest value; values
  // below it cannot be in the piece's k best and are skipped unexamined
  float bar = -INFINITY;
  bool fresh = true;  // no lower bound yet for the current row piece

  // close the piece of row r that ends at vector pe
  auto emit = [&](long long pe) {
    const long long ps = max(rs, v0);
    if (lane < k) {
      if (ps == rs && pe == rs + vpr) {
        out_v[r * k + lane] = lv;
        out_i[r * k + lane] = li;
      } else {
        const long long slot = 2 * w + (ps == v0 ? 0 : 1);
        part_v[slot * k + lane] = lv;
        part_i[slot * k + lane] = li;
      }
    }
    lv = tv = bar = -INFINITY;
    li = ti = INT32_MAX;
    fresh = true;
  };

  // the next batch's loads are issued before this batch is scanned
  uint4 nq[kTsUnroll];
#pragma unroll
  for (int u = 0; u < kTsUnroll; ++u)
    if (v0 + lane + 32 * u < v1) nq[u] = __ldcs(xv + v0 + lane + 32 * u);
  for (long long b0 = v0; b0 < v1; b0 += kBatch) {
    const int lim = (int)min((long long)kBatch, v1 - b0);
    uint4 q[kTsUnroll];
#pragma unroll
    for (int u = 0; u < kTsUnroll; ++u) q[u] = nq[u];
    const long long b1 = b0 + kBatch;
#pragma unroll
    for (int u = 0; u < kTsUnroll; ++u)
      if (b1 + lane + 32 * u < v1) nq[u] = __ldcs(xv + b1 + lane + 32 * u);
    // The common case: a whole batch inside the current row with k entries in
    // the list.  A batch whose lanes' maxima do not beat the k-th entry (or
    // lie below bar) holds nothing for the list: one vote skips it.
    if (!fresh && ti != INT32_MAX && lim == kBatch && b1 <= rs + vpr) {
      const float bm = batch_max<T>(q);
      if (!__any_sync(0xffffffffu, bm > tv && !(bm < bar))) {
        if (b1 == rs + vpr) {
          emit(b1);
          ++r;
          rs += vpr;
        }
        continue;
      }
    }
    int ps = 0;  // piece [ps, pe) of this batch lies in row r (offsets from b0)
    while (ps < lim) {
      const int pe = (int)min((long long)lim, rs + vpr - b0);
      const int base = (int)((b0 - rs) * E);  // row-local index of vector b0
      int excl = -1;  // a lane's element already in the list, not to be taken twice
      // After a fold the list holds elements from all over this batch, so a
      // vector here whose maximum ties the k-th entry may still hold a lower
      // index that beats it; elsewhere every list entry precedes the batch.
      bool folded = false;
      if (fresh) {
        // No bound yet for this row piece (it starts here, at a range start or
        // in the middle of the batch after a row end).  Each lane's best
        // element in [ps, pe) goes into the list in one fold (32 candidates at
        // once instead of one insert each); with k of them in, the k-th entry
        // bounds the piece's k-th largest from below.
        float lm = -INFINITY;
        int im = INT32_MAX;
#pragma unroll
        for (int u = 0; u < kTsUnroll; ++u) {
          const int j = lane + 32 * u;
          if (j >= ps && j < pe) {
            const float m = vec_max<T>(q[u]);
            if (m > lm) {  // the earliest vector holding the lane's maximum
              int e = E - 1;
#pragma unroll
              for (int ee = E - 1; ee >= 0; --ee)
                if (vec_elem<T>(q[u], ee) == m) e = ee;
              lm = m;
              im = base + j * E + e;
            }
          }
        }
        fold32(lv, li, lm, im);
        tv = __shfl_sync(0xffffffffu, lv, k - 1);
        ti = __shfl_sync(0xffffffffu, li, k - 1);
        excl = im;
        folded = true;
        if (ti != INT32_MAX) {
          bar = tv;
          fresh = false;
        }
      }
#pragma unroll
      for (int u = 0; u < kTsUnroll; ++u) {
        const int j = lane + 32 * u;
        const bool in = j >= ps && j < pe;
        const float m = vec_max<T>(q[u]);
        const bool flag = in && (m > tv || (folded && m == tv) || ti == INT32_MAX) && !(m < bar);
        const unsigned ballot = __ballot_sync(0xffffffffu, flag);
        if (ballot) take_own<T>(flag, q[u], base + j * E, excl, k, lv, li, tv, ti);
      }
      if (b0 + pe == rs + vpr) {
        emit(b0 + pe);
        ++r;
        rs += vpr;
      }
      ps = pe;
    }
  }
  if (v1 > rs && v1 < rs + vpr) emit(v1);  // the range ends inside row r
}

// Rows cut by range boundaries: warp p-1 of the grid owns boundary p when p is
// the first boundary inside its row, and folds that row's pieces.  Launched as
// a programmatic dependent of the streaming grid: the boundary arithmetic and
// the slots of the first kMergeHeld * 32 candidates are worked out while that
// grid still runs; the pieces' lists are read after griddepcontrol.wait, the
// held candidates all at once.
constexpr int kMergeHeld = 4;

__global__ void topk_stream_merge_kernel(const float *__restrict__ part_v,
                                         const int32_t *__restrict__ part_i, long long vpr,
                                         long long pen, long long tot, long long owners, int k,
                                         float *__restrict__ out_v, int32_t *__restrict__ out_i) {
  const long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5) + 1;
  const int lane = threadIdx.x & 31;
  if (p >= owners) return;
  const long long bnd = ts_split(p, vpr, pen, tot, owners);
  const long long r = bnd / vpr, rs = r * vpr;
  if (bnd == rs) return;                          // on a row start: nothing cut
  if (ts_split(p - 1, vpr, pen, tot, owners) > rs) return;  // an earlier boundary owns this row
  const long long c0 = p - 1;
  const long long c1 = ts_owner(rs + vpr - 1, vpr, pen, tot, owners);  // owner of the row's end
  const long long total = (c1 - c0 + 1) * k;
  // candidate qq is entry qq % k of piece c0 + qq / k: its pair's index in the
  // partial arrays, or -1 when that piece's range is empty (nothing written)
  auto cand = [&](long long qq) -> long long {
    if (qq >= total) return -1;
    const long long c = c0 + qq / k;
    const int jj = (int)(qq - (qq / k) * k);
    const long long s0 = ts_split(c, vpr, pen, tot, owners);
    if (s0 == ts_split(c + 1, vpr, pen, tot, owners)) return -1;
    return (2 * c + ((c == c0 && s0 < rs) ? 1 : 0)) * k + jj;
  };
  long long held[kMergeHeld];
#pragma unroll
  for (int h = 0; h < kMergeHeld; ++h) held[h] = cand(32LL * h + lane);
  pdl_wait();
  float hv[kMergeHeld];
  int hi[kMergeHeld];
#pragma unroll
  for (int h = 0; h < kMergeHeld; ++h) {
    hv[h] = held[h] >= 0 ? part_v[held[h]] : -INFINITY;
    hi[h] = held[h] >= 0 ? part_i[held[h]] : INT32_MAX;
  }
  // the pieces' lists, 32 candidates per step, one per lane, folded into the
  // list at once (steps where none beats the k-th entry are skipped)
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT32_MAX, ti = INT32_MAX;
  for (long long q0 = 0; q0 < total; q0 += 32) {
    const int h = (int)(q0 / 32);
    float x = -INFINITY;
    int xi = INT32_MAX;
#pragma unroll
    for (int e = 0; e < kMergeHeld; ++e)
      if (e == h) {
        x = hv[e];
        xi = hi[e];
      }
    if (h >= kMergeHeld) {  // rows cut into more pieces than held
      const long long o = cand(q0 + lane);
      if (o >= 0) {
        x = part_v[o];
        xi = part_i[o];
      }
    }
    if (!__any_sync(0xffffffffu, xi != INT32_MAX && beats(x, xi, tv, ti))) continue;
    fold32(lv, li, x, xi);
    tv = __shfl_sync(0xffffffffu, lv, k - 1);
    ti = __shfl_sync(0xffffffffu, li, k - 1);
  }
  if (lane < k) {
    out_v[r * k + lane] = lv;
    out_i[r * k + lane] = li;
  }
}

// ------------------------------------------------------------------ planning

struct TopkPlan {
  bool stream;
  int chunks;      // chunk plan
  int chunk_len;
  int ctas;        // stream plan
  size_t pairs;    // partial (value, index) pairs the plan writes
};

// Row-start weight of the stream plan's range split, in 16-byte vectors.
// Measured on 512 and 1024 rows of 151936 fp32: 2048 to 6144 vectors (one to
// three row pieces' worth of list building) take 6 to 8 % off the scan; small
// rows get an eighth of a row.
long long topk_row_penalty(long long vpr) { return vpr / 8 < 3072 ? vpr / 8 : 3072; }

bool topk_stream_shape(long long rows, long long V, int esize) {
  return (V * esize) % 16 == 0 && rows * V * esize >= 32768LL * sm_count();
}

TopkPlan topk_chunk_plan(long long rows, long long V, int esize, int k) {
  const int E = 16 / esize;
  // a few thread blocks per SM; never cut a row below 4K elements (a warp's
  // share then fits in one round of loads)
  const long long want = 8LL * sm_count();
  long long chunks = 1;
  if (rows < want) chunks = (want + rows - 1) / rows;
  const long long max_chunks = (V + 4095) / 4096;
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  long long len = (V + chunks - 1) / chunks;
  len = (len + E - 1) / E * E;
  chunks = (V + len - 1) / len;
  return TopkPlan{false, (int)chunks, (int)len, 0,
                  chunks > 1 ? (size_t)rows * chunks * k : (size_t)0};
}

TopkPlan plan_topk(const void *x, long long rows, long long V, long long row_stride, int esize,
                   int k) {
  if (topk_stream_shape(rows, V, esize) && row_stride == V &&
      (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
    const int ctas = sm_count();
    return TopkPlan{true, 1, 0, ctas, (size_t)2 * ctas * kTsWarps * k};
  }
  return topk_chunk_plan(rows, V, esize, k);
}

size_t topk_workspace_pairs(long long rows, long long V, int esize, int k) {
  size_t n = topk_chunk_plan(rows, V, esize, k).pairs;
  if (topk_stream_shape(rows, V, esize))
    n = n > (size_t)2 * sm_count() * kTsWarps * k ? n : (size_t)2 * sm_count() * kTsWarps * k;
  return n;
}

// ------------------------------------------------------------------ build_tree

constexpr int kBtWarps = 4;
constexpr int kBtStreams = TV_MAX_NODES + 1;  // the roots' cursor + one per node
constexpr int kBtSlots = (kBtStreams + 31) / 32;
constexpr int kBtStage = 1024;                // candidate tables up to L*K entries in smem

struct BtWarp {
  float node_score[TV_MAX_NODES];
  int node_tok[TV_MAX_NODES];
  int node_par[TV_MAX_NODES];
  int node_dep[TV_MAX_NODES];
  float lp[kBtStage];     // this sequence's candidate log-probs (when L*K fits)
  int tk[kBtStage];       // and token ids
};


// Candidate of a cursor at its current rank (key 0 once it runs past K).
__device__ __forceinline__ void bt_refresh(const float *lp, int K, int nr, int cb, int dep,
                                           float base, unsigned &key, int &cnt, float &sc) {
  if (nr >= 0 && nr < K) {
    const float v = lp[(size_t)(dep - 1) * K + nr];
    sc = dep == 1 ? v : __fadd_rn(base, v);
    key = score_key(sc);
    cnt = cb + nr;
  } else {
    key = 0;
  }
}

// Cursor u of a lane is stream lane + 32u: stream 0 walks the roots, stream
// t+1 the children of node t.  A lane keeps its cursors' state in registers:
// next rank, push counter of rank 0, the parent's score and the candidate
// depth, and the current candidate's score key and counter (key 0: none).
__global__ void __launch_bounds__(32 * kBtWarps)
build_tree_kernel(const float *cand_lp, const int32_t *cand_idx, int B, int L, int K, int budget,
                  int w, int32_t *__restrict__ tokens, int32_t *__restrict__ parent,
                  int32_t *__restrict__ depth, float *__restrict__ score,
                  int32_t *__restrict__ n_nodes) {
  __shared__ BtWarp sh[kBtWarps];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kBtWarps + wid;
  if (b >= B) return;
  BtWarp &s = sh[wid];
  const float *lp = cand_lp + (size_t)b * L * K;
  const int32_t *tk = cand_idx + (size_t)b * L * K;
  if (L * K <= kBtStage) {  // every pop reads these: keep them next to the warp
    for (int j0 = 0; j0 < L * K; j0 += 128) {  // four loads per lane in flight, then stores
      float v[4];
      int t[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = j0 + lane + 32 * i;
        if (j < L * K) {
          v[i] = __ldg(lp + j);
          t[i] = __ldg(tk + j);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = j0 + lane + 32 * i;
        if (j < L * K) {
          s.lp[j] = v[i];
          s.tk[j] = t[i];
        }
      }
    }
    lp = s.lp;
    tk = s.tk;
    __syncwarp();
  }
  int nr[kBtSlots], cb[kBtSlots], dep[kBtSlots];
  float base[kBtSlots];
  unsigned key[kBtSlots];
  int cnt[kBtSlots];
  float sc[kBtSlots];
#pragma unroll
  for (int u = 0; u < kBtSlots; ++u) {
    nr[u] = -1;
    cb[u] = 0;
    dep[u] = 1;
    base[u] = 0.f;
    key[u] = 0;
    cnt[u] = INT32_MAX;
    sc[u] = -INFINITY;
  }
  if (lane == 0) {  // the roots: depth-1 candidates, counters 0 .. K-1
    nr[0] = 0;
    cb[0] = 0;
    dep[0] = 1;
    base[0] = 0.f;
    bt_refresh(lp, K, nr[0], cb[0], dep[0], base[0], key[0], cnt[0], sc[0]);
  }
  int counter = K;
  int n = 0;
  while (n < budget) {
    const int start = n;
    const int take = min(w, budget - n);
    // children cursors opened by this round's nodes, set up in the registers
    // of the lanes that own them and opened when the round ends
    unsigned pend = 0;  // bit u: this lane's cursor u opens at the round's end
    int pushes = 0;  // this round's popped nodes with children, so far
    for (int q = 0; q < take; ++q) {
      // this lane's best cursor: higher score, then lower counter
      unsigned bk = 0;
      int bc = INT32_MAX, bu = -1;
#pragma unroll
      for (int u = 0; u < kBtSlots; ++u)
        if (key[u] > bk || (key[u] == bk && key[u] != 0 && cnt[u] < bc)) {
          bk = key[u];
          bc = cnt[u];
          bu = u;
        }
      const unsigned wk = __reduce_max_sync(0xffffffffu, bk);
      if (wk == 0) break;  // the heap ran empty: the round ends early
      unsigned win = __ballot_sync(0xffffffffu, bk == wk);
      if (win & (win - 1)) {  // tied scores: the lower push counter wins
        const unsigned wc = __reduce_min_sync(0xffffffffu, bk == wk ? (unsigned)bc : 0xffffffffu);
        win = __ballot_sync(0xffffffffu, bk == wk && (unsigned)bc == wc);
      }
      const int src = __ffs(win) - 1;
      float psc = 0.f;
      int pdep = 0;
      if (lane == src) {
#pragma unroll
        for (int u = 0; u < kBtSlots; ++u) {  // static indices keep the cursors in registers
          if (u == bu && TV_CHECK(n < budget && n < TV_MAX_NODES && dep[u] >= 1 && dep[u] <= L && nr[u] >= 0 && nr[u] < K)) {
            psc = sc[u];
            pdep = dep[u];
            s.node_score[n] = sc[u];
            s.node_tok[n] = tk[(size_t)(dep[u] - 1) * K + nr[u]];
            s.node_par[n] = lane + 32 * u - 1;
            s.node_dep[n] = dep[u];
            ++nr[u];
            bt_refresh(lp, K, nr[u], cb[u], dep[u], base[u], key[u], cnt[u], sc[u]);
          }
        }
      }
      // node n's children are cursor n+1 (lane (n+1) % 32, slot (n+1) / 32),
      // with the next K push counters in pop order
      psc = __shfl_sync(0xffffffffu, psc, src);
      pdep = __shfl_sync(0xffffffffu, pdep, src);
      if (pdep < L) {
        const bool mine = lane == ((n + 1) & 31);
        const int tu = (n + 1) >> 5;
#pragma unroll
        for (int u = 0; u < kBtSlots; ++u) {  // selects, not a store at a computed index
          const bool m = mine && tu == u;
          pend |= m ? 1u << u : 0u;
          cb[u] = m ? counter + K * pushes : cb[u];
          dep[u] = m ? pdep + 1 : dep[u];
          base[u] = m ? psc : base[u];
        }
        ++pushes;
      }
      ++n;
    }
    if (n == start) break;  // nothing left to pop: the K-ary tree of depth L is complete
#pragma unroll
    for (int u = 0; u < kBtSlots; ++u)
      if (pend & (1u << u)) {
        nr[u] = 0;
        bt_refresh(lp, K, nr[u], cb[u], dep[u], base[u], key[u], cnt[u], sc[u]);
      }
    counter += K * pushes;
  }
  __syncwarp();
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
  const size_t n = topk_workspace_pairs(rows, V, esize, k);
  if (n == 0) return 0;
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
  const TopkPlan p = plan_topk(x, rows, V, row_stride, esize, k);
  if (!p.stream && (long long)rows * p.chunks > (long long)INT32_MAX) return TV_ERR_ARG;
  float *pv = out_vals;
  int32_t *pi = out_idx;
  if (p.pairs > 0) {
    if (!workspace || workspace_bytes < tv_topk_workspace_size(rows, V, k, dtype)) return TV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return TV_ERR_ARG;
    const size_t n = topk_workspace_pairs(rows, V, esize, k);
    pv = static_cast<float *>(workspace);
    pi = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                     ((n * sizeof(float) + 255) / 256) * 256);
  }
  cudaStream_t s = as_stream(stream);
  if (p.stream) {
    const long long vpr = V * esize / 16;
    const long long owners = (long long)p.ctas * kTsWarps;
    const long long pen = topk_row_penalty(vpr);
    const long long tot = rows * (vpr + pen);
    if (dtype == TV_BF16)
      topk_stream_kernel<__nv_bfloat16><<<p.ctas, 32 * kTsWarps, 0, s>>>(
          static_cast<const __nv_bfloat16 *>(x), vpr, pen, tot, owners, k, pv, pi, out_vals,
          out_idx);
    else
      topk_stream_kernel<float><<<p.ctas, 32 * kTsWarps, 0, s>>>(
          static_cast<const float *>(x), vpr, pen, tot, owners, k, pv, pi, out_vals, out_idx);
    const int wpb = 8;
    if (launch_pdl(topk_stream_merge_kernel, dim3((unsigned)((owners - 1 + wpb - 1) / wpb)),
                   dim3(32 * wpb), 0, s, pv, pi, vpr, pen, tot, owners, k, out_vals, out_idx) !=
        cudaSuccess)
      return TV_ERR_CUDA;
    return launch_status();
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && ((row_stride * esize) % 16 == 0);
  const unsigned grid = (unsigned)(rows * p.chunks);
  float *cv = p.chunks > 1 ? pv : out_vals;
  int32_t *ci = p.chunks > 1 ? pi : out_idx;
  if (dtype == TV_BF16)
    topk_chunk_kernel<__nv_bfloat16><<<grid, kTopThreads, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(x), (int)V, row_stride, p.chunks, p.chunk_len, vec, k, cv,
        ci);
  else
    topk_chunk_kernel<float><<<grid, kTopThreads, 0, s>>>(static_cast<const float *>(x), (int)V,
                                                          row_stride, p.chunks, p.chunk_len, vec, k,
                                                          cv, ci);
  if (p.chunks > 1 &&
      launch_pdl(topk_merge_kernel, dim3((unsigned)rows), dim3(32 * kMergeWarps), 0, s, pv, pi, rows,
                 p.chunks, k, out_vals, out_idx) != cudaSuccess)
    return TV_ERR_CUDA;
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
