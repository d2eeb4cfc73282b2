// Vocab-wide argmax of every logits row: an HBM-bound streaming scan.
//
// Source: "Tree spec-decode -> vLLM serve integration spec", "3. Rejection
// sampler: tree walk" -- the walk consumes argmax(target_logits[t]) for every
// node and must stay argmax-exact (no sampling).
//
// Each thread block reduces one chunk of one row; a row is split into several
// chunks only when there are too few rows to fill the GPU.  Loads are 16-byte
// vectors, four in flight per thread before any is consumed.  Every thread
// visits its indices in increasing order and keeps (value, index) with a strict
// ">", so within a thread the lowest index of the maximum survives; across
// threads and chunks the pairs merge with "larger value, or equal value and
// lower index".  NaN is mapped to -inf so it never wins; +0 and -0 compare
// equal as floats.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "common.cuh"

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
    if (chunks == 1) {
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

struct ArgmaxPlan {
  int chunks;
  int chunk_len;
};

ArgmaxPlan plan_argmax(long long rows, long long V, int esize) {
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
  return ArgmaxPlan{(int)chunks, (int)len};
}

}  // namespace

}  // namespace tv

using namespace tv;

extern "C" size_t tv_argmax_workspace_size(int64_t rows, int64_t V, int dtype) {
  if (rows <= 0 || V <= 0) return 0;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const ArgmaxPlan p = plan_argmax(rows, V, esize);
  if (p.chunks == 1) return 0;
  const size_t n = (size_t)rows * p.chunks;
  return ((n * sizeof(float) + 255) / 256) * 256 + n * sizeof(int32_t);
}

extern "C" tv_status tv_argmax(const void *logits, int dtype, int64_t rows, int64_t V,
                               int64_t row_stride, int32_t *out_idx, void *workspace,
                               size_t workspace_bytes, tv_stream stream) {
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  if (rows < 0 || V < 1 || row_stride < V || V > INT32_MAX - 1024) return TV_ERR_ARG;
  if (rows == 0) return TV_OK;
  if (rows > (int64_t)INT32_MAX) return TV_ERR_ARG;
  if (!logits || !out_idx) return TV_ERR_ARG;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const ArgmaxPlan p = plan_argmax(rows, V, esize);
  if ((long long)rows * p.chunks > (long long)INT32_MAX) return TV_ERR_ARG;
  float *pv = nullptr;
  int32_t *pi = nullptr;
  if (p.chunks > 1) {
    if (!workspace || workspace_bytes < tv_argmax_workspace_size(rows, V, dtype)) return TV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15) return TV_ERR_ARG;
    const size_t n = (size_t)rows * p.chunks;
    pv = static_cast<float *>(workspace);
    pi = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                     ((n * sizeof(float) + 255) / 256) * 256);
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) &&
                   ((row_stride * esize) % 16 == 0);
  const unsigned grid = (unsigned)(rows * p.chunks);
  cudaStream_t s = as_stream(stream);
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
  if (dtype != TV_F32 && dtype != TV_BF16) return TV_ERR_UNSUPPORTED;
  if (rows < 0 || V < 1 || row_stride < V || V > INT32_MAX - 1024) return TV_ERR_ARG;
  if (rows == 0) return TV_OK;
  if (rows > (int64_t)INT32_MAX) return TV_ERR_ARG;
  if (!logits || !out_idx) return TV_ERR_ARG;
  const int esize = dtype == TV_F32 ? 4 : 2;
  const ArgmaxPlan p = plan_argmax(rows, V, esize);
  float *pv = nullptr;
  int32_t *pi = nullptr;
  if (p.chunks > 1) {
    if ((unsigned long long)rows * p.chunks > kNoAllocPairs) return TV_ERR_SCRATCH_LIMIT;
    char *base = static_cast<char *>(noalloc_scratch());
    if (!base) return TV_ERR_CUDA;
    pv = reinterpret_cast<float *>(base);
    pi = reinterpret_cast<int32_t *>(base + kNoAllocPairs * sizeof(float));
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) &&
                   ((row_stride * esize) % 16 == 0);
  const unsigned grid = (unsigned)(rows * p.chunks);
  cudaStream_t s = as_stream(stream);
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
