// Vocab-wide argmax of every logits row: an HBM-bound streaming scan.
//
// Source: "Tree spec-decode -> vLLM serve integration spec", "3. Rejection
// sampler: tree walk" -- the walk consumes argmax(target_logits[t]) for every
// node and must stay argmax-exact (no sampling).
//
// Two plans, one result.
//
// Stream plan (dense rows, 16-byte aligned, at least 32 KiB of logits per SM):
// the flattened [rows x V] array is cut into equal contiguous ranges, one per
// warp of a one-CTA-per-SM grid, so every SM moves the same bytes however the
// rows fall.  A warp reads its range in batches of 16 coalesced 16-byte loads
// per lane, all issued before any is used.  A row lying whole in a warp's
// range is written directly; the first and last row pieces of a range go to
// two partial slots, and a small merge kernel (one warp per range boundary)
// finishes the rows cut by a boundary.
//
// Chunk plan (everything else: strided or unaligned rows, small inputs): one
// thread block per row chunk with 16-byte loads, four in flight per thread; a
// row is cut into chunks only when there are too few rows to fill the GPU.
//
// Every thread visits its indices in increasing order and replaces its
// (value, index) only on a strictly larger value, so the lowest index of the
// maximum survives; threads, pieces and chunks merge with "larger value, or
// equal value and lower index".  NaN is mapped to -inf so it never wins (the
// packed bf16 max ignores a NaN operand the same way); +0 and -0 compare equal.
// A piece with no finite maximum keeps its first index with value -inf, so a
// row of only -inf / NaN gives index 0.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"

TV_DEBUG_RECORD(argmax)

namespace tv {

namespace {

constexpr int kArgThreads = 256;
constexpr int kUnroll = 4;

struct Best {
  float v;
  int i;
};

__device__ __forceinline__ void take(Best &a, float v, int i) {
  v = (v != v) ? -INFINITY : v;
  if (v > a.v || (v == a.v && i < a.i)) {
    a.v = v;
    a.i = i;
  }
}

__device__ __forceinline__ void merge(Best &a, const Best &b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) a = b;
}

__device__ __forceinline__ Best block_reduce(Best me) {
  __shared__ float sv[kArgThreads / 32];
  __shared__ int si[kArgThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best other{__shfl_xor_sync(0xffffffffu, me.v, o), __shfl_xor_sync(0xffffffffu, me.i, o)};
    merge(me, other);
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[w] = me.v;
    si[w] = me.i;
  }
  __syncthreads();
  if (w == 0) {
    Best r{-INFINITY, INT32_MAX};
    if (lane < kArgThreads / 32) r = Best{sv[lane], si[lane]};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Best other{__shfl_xor_sync(0xffffffffu, r.v, o), __shfl_xor_sync(0xffffffffu, r.i, o)};
      merge(r, other);
    }
    me = r;
  }
  return me;  // valid in thread 0
}

template <typename T>
__device__ __forceinline__ void take_vec(Best &best, const uint4 &w, int i0);

template <>
__device__ __forceinline__ void take_vec<__nv_bfloat16>(Best &best, const uint4 &w, int i0) {
  take(best, bf16_lo(w.x), i0 + 0);
  take(best, bf16_hi(w.x), i0 + 1);
  take(best, bf16_lo(w.y), i0 + 2);
  take(best, bf16_hi(w.y), i0 + 3);
  take(best, bf16_lo(w.z), i0 + 4);
  take(best, bf16_hi(w.z), i0 + 5);
  take(best, bf16_lo(w.w), i0 + 6);
  take(best, bf16_hi(w.w), i0 + 7);
}

template <>
__device__ __forceinline__ void take_vec<float>(Best &best, const uint4 &w, int i0) {
  take(best, __uint_as_float(w.x), i0 + 0);
  take(best, __uint_as_float(w.y), i0 + 1);
  take(best, __uint_as_float(w.z), i0 + 2);
  take(best, __uint_as_float(w.w), i0 + 3);
}

__device__ __forceinline__ float load_one(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load_one(const float *p) { return *p; }

// grid.x = rows * chunks.  chunk_len is a multiple of the vector width, so
// every chunk starts on a vector boundary when the row does (vec == true).
template <typename T>
__global__ void __launch_bounds__(kArgThreads)
argmax_chunk_kernel(const T *__restrict__ x, int V, long long row_stride, int chunks,
                    int chunk_len, bool vec, float *__restrict__ part_v,
                    int32_t *__restrict__ part_i, int32_t *__restrict__ out_idx) {
  constexpr int E = 16 / sizeof(T);
  const long long row = blockIdx.x / chunks;
  const int c = blockIdx.x - (int)(row * chunks);
  const int begin = c * chunk_len;
  const int end = min(V, begin + chunk_len);
  const T *xr = x + row * row_stride;
  Best best{-INFINITY, INT32_MAX};
  int tail = begin;
  if (vec) {
    const int nvec = (end - begin) / E;
    const uint4 *xv = reinterpret_cast<const uint4 *>(xr + begin);
    const int step = kArgThreads * kUnroll;
    for (int j0 = threadIdx.x; j0 < nvec; j0 += step) {
      uint4 w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int j = j0 + u * kArgThreads;
        if (j < nvec) w[u] = __ldg(xv + j);
      }
      // the u-loop visits this thread's indices in increasing order
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int j = j0 + u * kArgThreads;
        if (j < nvec) take_vec<T>(best, w[u], begin + j * E);
      }
    }
    tail = begin + nvec * E;
  }
  for (int i = tail + threadIdx.x; i < end; i += kArgThreads) take(best, load_one(xr + i), i);
  best = block_reduce(best);
  if (threadIdx.x == 0) {
    if (best.i == INT32_MAX) best.i = begin;  // empty chunk cannot happen; keep in range
    if (!TV_CHECK(best.i >= begin && best.i < end)) {
    } else if (chunks == 1) {
      out_idx[row] = best.i;
    } else {
      part_v[blockIdx.x] = best.v;
      part_i[blockIdx.x] = best.i;
    }
  }
}

// One warp per row merges that row's chunk winners.
__global__ void argmax_final_kernel(const float *__restrict__ part_v,
                                    const int32_t *__restrict__ part_i, long long rows,
                                    int chunks, int32_t *__restrict__ out_idx) {
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  Best me{-INFINITY, INT32_MAX};
  for (int c = lane; c < chunks; c += 32) merge(me, Best{part_v[row * chunks + c], part_i[row * chunks + c]});
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best other{__shfl_xor_sync(0xffffffffu, me.v, o), __shfl_xor_sync(0xffffffffu, me.i, o)};
    merge(me, other);
  }
  if (lane == 0) out_idx[row] = me.i;
}

// ------------------------------------------------------------------ stream plan

constexpr int kStrWarps = 16;                  // warps per CTA, one CTA per SM
constexpr int kStrThreads = 32 * kStrWarps;
constexpr int kStrUnroll = 16;                 // 16-byte loads in flight per lane

// Fold one 16-byte vector into a lane's best, visiting its elements in
// increasing index order: a packed max first, the element search only when the
// vector holds a new strict maximum.  NaN operands are ignored by the max.
template <typename T>
__device__ __forceinline__ void scan_vec(Best &best, const uint4 &w, int i0);

template <>
__device__ __forceinline__ void scan_vec<__nv_bfloat16>(Best &best, const uint4 &w, int i0) {
  uint32_t m2, n2;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(w.x), "r"(w.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(n2) : "r"(w.z), "r"(w.w));
  asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(n2));
  const float m = fmaxf(bf16_lo(m2), bf16_hi(m2));
  if (m > best.v) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    int e = 7;
#pragma unroll
    for (int k = 7; k >= 0; --k) {
      const float v = (k & 1) ? bf16_hi(ws[k >> 1]) : bf16_lo(ws[k >> 1]);
      if (v == m) e = k;
    }
    best.v = m;
    best.i = i0 + e;
  }
}

template <>
__device__ __forceinline__ void scan_vec<float>(Best &best, const uint4 &w, int i0) {
  const float a = __uint_as_float(w.x), b = __uint_as_float(w.y);
  const float c = __uint_as_float(w.z), d = __uint_as_float(w.w);
  const float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
  if (m > best.v) {
    best.v = m;
    best.i = i0 + (a == m ? 0 : b == m ? 1 : c == m ? 2 : 3);
  }
}

__device__ __forceinline__ Best warp_best(Best me) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Best other{__shfl_xor_sync(0xffffffffu, me.v, o), __shfl_xor_sync(0xffffffffu, me.i, o)};
    merge(me, other);
  }
  return me;
}

// First flat vector of owner (warp) w's range: floor(w * nv / owners).
__device__ __forceinline__ long long str_split(long long w, long long nv, long long owners) {
  return w * nv / owners;
}

// The rows are dense: nv = rows * vpr 16-byte vectors, vpr per row.  Global
// warp w owns vectors [w*nv/owners, (w+1)*nv/owners) and reads them in
// batches of 32 * kStrUnroll, every load of a batch issued before any is used.
// A row lying whole in the range is written directly; the range's first and
// last row pieces go to partial slots 2w and 2w+1.
template <typename T>
__global__ void __launch_bounds__(kStrThreads, 1)
argmax_stream_kernel(const T *__restrict__ x, long long nv, long long vpr, long long owners,
                     float *__restrict__ part_v, int32_t *__restrict__ part_i,
                     int32_t *__restrict__ out_idx) {
  constexpr int E = 16 / sizeof(T);
  constexpr int kBatch = 32 * kStrUnroll;
  // the merge grid may be launched now: it waits for this grid's completion
  // before it reads the partials.  (This grid itself is launched normally: as
  // a programmatic dependent of the attention's combine grid the verify step
  // took 22 us longer.)
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kStrWarps + (threadIdx.x >> 5);
  if (w >= owners) return;
  const long long v0 = str_split(w, nv, owners), v1 = str_split(w + 1, nv, owners);
  const uint4 *xv = reinterpret_cast<const uint4 *>(x);
  long long r = v0 / vpr;          // current row
  long long rs = r * vpr;          // its first vector
  Best best{-INFINITY, INT32_MAX};

  // close the piece of row r that ends at vector `pe`
  auto emit = [&](long long pe) {
    const Best b = warp_best(best);
    if (lane == 0) {
      const long long ps = max(rs, v0);
      const int idx = b.i == INT32_MAX ? (int)((ps - rs) * E) : b.i;
      if (!TV_CHECK(idx >= 0 && idx < vpr * E && r < nv / vpr && 2 * w + 1 < 2 * owners)) {
      } else if (ps == rs && pe == rs + vpr) {
        out_idx[r] = idx;
      } else {
        const long long slot = 2 * w + (ps == v0 ? 0 : 1);
        part_v[slot] = b.v;
        part_i[slot] = idx;
      }
    }
    best = Best{-INFINITY, INT32_MAX};
  };

  for (long long b0 = v0; b0 < v1; b0 += kBatch) {
    const uint4 *src = xv + b0;
    const int lim = (int)min((long long)kBatch, v1 - b0);  // vectors in this batch
    uint4 q[kStrUnroll];
#pragma unroll
    for (int u = 0; u < kStrUnroll; ++u)
      if (lane + 32 * u < lim) q[u] = __ldcs(src + lane + 32 * u);
    // offsets below are relative to b0 (32-bit): the batch is at most kBatch long
    int base = (int)((b0 - rs) * E);                  // row-local index of vector b0
    int rend = (int)min((long long)kBatch + 1, rs + vpr - b0);  // row end, capped
    if (lim <= rend) {
      // fast path: the whole batch lies in row r
#pragma unroll
      for (int u = 0; u < kStrUnroll; ++u) {
        const int j = lane + 32 * u;
        if (j < lim) scan_vec<T>(best, q[u], base + j * E);
      }
      if (lim == rend) {
        emit(b0 + lim);
        ++r;
        rs += vpr;
      }
    } else {
      // the batch crosses one or more row ends: one pass per row piece
      int ps = 0;
      while (ps < lim) {
        const int pe = min(lim, rend);
#pragma unroll
        for (int u = 0; u < kStrUnroll; ++u) {
          const int j = lane + 32 * u;
          if (j >= ps && j < pe) scan_vec<T>(best, q[u], base + j * E);
        }
        if (pe == rend) {
          emit(b0 + pe);
          ++r;
          rs += vpr;
          base = (int)((b0 - rs) * E);
          rend = (int)min((long long)kBatch + 1, rs + vpr - b0);
        }
        ps = pe;
      }
    }
  }
  if (v1 > v0 && v1 < rs + vpr && v1 > rs) emit(v1);  // range ends inside row r
}

// Rows cut by owner boundaries: warp p-1 of the grid owns boundary p
// (1 <= p < owners) when p is the first boundary inside its row, and merges
// that row's pieces.
__global__ void argmax_stream_merge_kernel(const float *__restrict__ part_v,
                                           const int32_t *__restrict__ part_i, long long nv,
                                           long long vpr, long long owners,
                                           int32_t *__restrict__ out_idx) {
  // launched as a programmatic dependent of the streaming grid: the partials
  // are read after griddepcontrol.wait; the grid after this one (the tree
  // walk) may be scheduled at once
  pdl_launch_dependents();
  const long long p = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5) + 1;
  const int lane = threadIdx.x & 31;
  if (p >= owners) return;
  const long long bnd = str_split(p, nv, owners);
  const long long r = bnd / vpr, rs = r * vpr;
  if (bnd == rs) return;                            // boundary on a row start: nothing cut
  if (str_split(p - 1, nv, owners) > rs) return;    // an earlier boundary owns this row
  const long long c0 = p - 1;
  // owner of the row's last vector x: ceil((x+1) * owners / nv) - 1
  const long long xl = rs + vpr - 1;
  const long long c1 = ((xl + 1) * owners + nv - 1) / nv - 1;
  // the slot of this lane's piece (or -1: none, or an empty range that wrote
  // nothing), worked out before the streaming grid has finished
  auto slot_of = [&](long long c) -> long long {
    if (c > c1 || !TV_CHECK(c < owners)) return -1;
    const long long s0 = str_split(c, nv, owners);
    if (s0 == str_split(c + 1, nv, owners)) return -1;
    return 2 * c + ((c == c0 && s0 < rs) ? 1 : 0);
  };
  // up to kArgHeld * 32 pieces (a few rows cut into many warp ranges) are
  // worked out before the wait and then read all at once
  constexpr int kArgHeld = 8;
  long long held[kArgHeld];
#pragma unroll
  for (int h = 0; h < kArgHeld; ++h) held[h] = slot_of(c0 + lane + 32LL * h);
  pdl_wait();
  Best got[kArgHeld];
#pragma unroll
  for (int h = 0; h < kArgHeld; ++h)
    got[h] = held[h] >= 0 ? Best{part_v[held[h]], part_i[held[h]]} : Best{-INFINITY, INT32_MAX};
  Best me{-INFINITY, INT32_MAX};
#pragma unroll
  for (int h = 0; h < kArgHeld; ++h)
    if (held[h] >= 0) merge(me, got[h]);
  for (long long c = c0 + lane + 32LL * kArgHeld; c <= c1; c += 32) {  // rows cut into still more pieces
    const long long slot = slot_of(c);
    if (slot >= 0) merge(me, Best{part_v[slot], part_i[slot]});
  }
  me = warp_best(me);
  if (lane == 0 && TV_CHECK(r < nv / vpr && me.i >= 0 && me.i < vpr * (16 / 2))) out_idx[r] = me.i;
}

// ------------------------------------------------------------------ planning

struct ArgmaxPlan {
  bool stream;     // stream plan (else chunk plan)
  int chunks;      // chunk plan: chunks per row
  int chunk_len;   // chunk plan: elements per chunk
  int ctas;        // stream plan: persistent CTAs
  size_t pairs;    // (value, index) partials the plan writes
};

// Shapes the stream plan can take when the rows are dense and aligned: whole
// 16-byte vectors per row and at least two chunks of work per SM.
bool stream_shape(long long rows, long long V, int esize) {
  return (V * esize) % 16 == 0 && rows * V * esize >= 32768LL * sm_count();
}

ArgmaxPlan chunk_plan(long long rows, long long V, int esize) {
  const int E = 16 / esize;
  // Aim for a few thread blocks per SM; never cut a row below 8K elements.
  const long long want = 8LL * sm_count();
  long long chunks = 1;
  if (rows < want) chunks = (want + rows - 1) / rows;
  long long max_chunks = (V + 8191) / 8192;
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1) chunks = 1;
  long long len = (V + chunks - 1) / chunks;
  len = (len + E - 1) / E * E;
  chunks = (V + len - 1) / len;
  return ArgmaxPlan{false, (int)chunks, (int)len, 0,
                    chunks > 1 ? (size_t)rows * (size_t)chunks : (size_t)0};
}

ArgmaxPlan plan_argmax(const void *logits, long long rows, long long V, long long row_stride,
                       int esize, int sm_limit = 0) {
  if (stream_shape(rows, V, esize) && row_stride == V &&
      (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    const int ctas = sm_limit > 0 && sm_limit < sm_count() ? sm_limit : sm_count();
    return ArgmaxPlan{true, 1, 0, ctas, (size_t)2 * ctas * kStrWarps};
  }
  return chunk_plan(rows, V, esize);
}

// Partials the workspace must hold for any call with this shape.
size_t workspace_pairs(long long rows, long long V, int esize) {
  size_t n = chunk_plan(rows, V, esize).pairs;
  if (stream_shape(rows, V, esize)) n = std::max(n, (size_t)2 * sm_count() * kStrWarps);
  return n;
}

tv_status launch_argmax(const void *logits, int dtype, long long rows, long long V,
                        long long row_stride, int32_t *out_idx, const ArgmaxPlan &p, float *pv,
                        int32_t *pi, cudaStream_t s) {
  const int esize = dtype == TV_F32 ? 4 : 2;
  if (p.stream) {
    const long long vpr = V * esize / 16;
    const long long nv = rows * vpr;
    const long long owners = (long long)p.ctas * kStrWarps;
    if (dtype == TV_BF16)
      argmax_stream_kernel<__nv_bfloat16><<<p.ctas, kStrThreads, 0, s>>>(
          static_cast<const __nv_bfloat16 *>(logits), nv, vpr, owners, pv, pi, out_idx);
    else
      argmax_stream_kernel<float><<<p.ctas, kStrThreads, 0, s>>>(
          static_cast<const float *>(logits), nv, vpr, owners, pv, pi, out_idx);
    const int wpb = 8;
    if (launch_pdl(argmax_stream_merge_kernel, dim3((unsigned)((owners - 1 + wpb - 1) / wpb)),
                   dim3(wpb * 32), 0, s, pv, pi, nv, vpr, owners, out_idx) != cudaSuccess)
      return TV_ERR_CUDA;
    return launch_status();
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) &&
                   ((row_stride * esize) % 16 == 0);
  const unsigned grid = (unsigned)(rows * p.chunks);
  if (dtype == TV_BF16)
    argmax_chunk_kernel<__nv_bfloat16><<<grid, kArgThreads, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(logits), (int)V, row_stride, p.chunks, p.chunk_len, vec,
        pv, pi, out_idx);
  else
    argmax_chunk_kernel<float><<<grid, kArgThreads, 0, s>>>(
        static_cast<const float *>(logits), (int)V, row_stride, p.chunks, p.chunk_len, vec, pv, pi,
        out_idx);
  if (p.chunks > 1) {
    const int wpb = 8;
    argmax_final_kernel<<<(unsigned)((rows + wpb - 1) / wpb), wpb * 32, 0, s>>>(pv, pi, rows,
                                                                              p.chunks, out_idx);
  }
  return launch_status();
}

tv_status check_args(const void *logits, int dtype, int64_t rows, int64_t V, int64_t row_stride,
                     const int32_t *out_idx) {
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  if (rows < 0 || V < 1 || row_stride < V || V > INT32_MAX - 1024) return TV_ERR_ARG;
  if (rows == 0) return TV_OK;
  if (rows > (int64_t)INT32_MAX) return TV_ERR_ARG;
  if (!logits || !out_idx) return TV_ERR_ARG;
  return TV_OK;
}

}  // namespace

}  // namespace tv

using namespace tv;

extern "C" size_t tv_argmax_workspace_size(int64_t rows, int64_t V, int dtype) {
  if (rows <= 0 || V <= 0) return 0;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const size_t n = workspace_pairs(rows, V, esize);
  if (n == 0) return 0;
  return ((n * sizeof(float) + 255) / 256) * 256 + n * sizeof(int32_t);
}

extern "C" tv_status tv_argmax_sm(const void *logits, int dtype, int64_t rows, int64_t V,
                                  int64_t row_stride, int32_t *out_idx, void *workspace,
                                  size_t workspace_bytes, int sm_limit, tv_stream stream) {
  if (sm_limit < 0) return TV_ERR_ARG;
  const tv_status st = check_args(logits, dtype, rows, V, row_stride, out_idx);
  if (st != TV_OK || rows == 0) return st;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const ArgmaxPlan p = plan_argmax(logits, rows, V, row_stride, esize, sm_limit);
  if (!p.stream && (long long)rows * p.chunks > (long long)INT32_MAX) return TV_ERR_ARG;
  float *pv = nullptr;
  int32_t *pi = nullptr;
  if (p.pairs > 0) {
    if (!workspace || workspace_bytes < tv_argmax_workspace_size(rows, V, dtype)) return TV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return TV_ERR_ARG;
    const size_t n = workspace_pairs(rows, V, esize);
    pv = static_cast<float *>(workspace);
    pi = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                     ((n * sizeof(float) + 255) / 256) * 256);
  }
  return launch_argmax(logits, dtype, rows, V, row_stride, out_idx, p, pv, pi, as_stream(stream));
}

extern "C" tv_status tv_argmax(const void *logits, int dtype, int64_t rows, int64_t V,
                               int64_t row_stride, int32_t *out_idx, void *workspace,
                               size_t workspace_bytes, tv_stream stream) {
  return tv_argmax_sm(logits, dtype, rows, V, row_stride, out_idx, workspace, workspace_bytes, 0,
                      stream);
}

// ---------------------------------------------------------------------------
// tv_argmax_noalloc: the same argmax for callers that cannot allocate device
// memory.  Its split partials live in a fixed file-scope device array instead
// of a caller-provided workspace.
//
// Device code could name the array directly; host code must not pass its name
// to a kernel (on the host the name is only a stand-in, not a device address),
// so the address is fetched once per device with cudaGetSymbolAddress and
// cached.
namespace tv {
namespace {

constexpr size_t kNoAllocPairs = 8192;  // (value, index) partials: 64 KiB in all
static __device__ __align__(256) unsigned char g_argmax_scratch[kNoAllocPairs * 8];

// Device address of g_argmax_scratch on the current device (set up on the
// first call made with that device current), or nullptr on failure.
void *noalloc_scratch() {
  static std::mutex mu;
  static std::vector<void *> addr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if ((int)addr.size() <= dev) addr.resize(dev + 1, nullptr);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_argmax_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_argmax_noalloc(const void *logits, int dtype, int64_t rows, int64_t V,
                                       int64_t row_stride, int32_t *out_idx, tv_stream stream) {
  const tv_status st = check_args(logits, dtype, rows, V, row_stride, out_idx);
  if (st != TV_OK || rows == 0) return st;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const ArgmaxPlan p = plan_argmax(logits, rows, V, row_stride, esize);
  float *pv = nullptr;
  int32_t *pi = nullptr;
  if (p.pairs > 0) {
    if (p.pairs > kNoAllocPairs) return TV_ERR_SCRATCH_LIMIT;
    char *base = static_cast<char *>(noalloc_scratch());
    if (!base) return TV_ERR_CUDA;
    pv = reinterpret_cast<float *>(base);
    pi = reinterpret_cast<int32_t *>(base + kNoAllocPairs * sizeof(float));
  }
  return launch_argmax(logits, dtype, rows, V, row_stride, out_idx, p, pv, pi, as_stream(stream));
}
