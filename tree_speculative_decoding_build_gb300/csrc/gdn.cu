// Rollback-free tree verification of a Gated DeltaNet layer, and the deferred
// commit of its state.
//
// Source: "Technische Samenvatting: Trees from Marginals (DFlash-TfM)",
// "3. Rollback-vrije Boom-verificatie voor GDN".  With u_t = beta_t (v_t -
// alpha_t S_parent^T k_t) and g_t the product of alpha along a node's path,
// the state of node t is S_t = g_t S_0 + sum_{i anc-or-self} (g_t/g_i) k_i u_i^T,
// so the pseudo-values solve (I + X) U = beta * (V - g * K S_0), X masked to
// strict ancestors (lower triangular in parents-first order), and the outputs
// are O = g * (Q S_0) + Y U, Y masked to ancestors-or-self.
//
// tv_gdn_tree_verify: one CTA per (sequence, value head, 64 columns of d_v).
// The columns of U are independent in the triangular system, so splitting d_v
// only repeats the small ancestor-pair dot products.  In shared memory: the
// 64 rows of S_0^T, K and Q rows of the key head (fp32, rows padded), X and Y
// on ancestor pairs (one thread per pair), U's 64 columns.  For K S_0 and
// Q S_0 (fp32 FMA, float4 shared loads, all loads of a step before its FMAs)
// warp w owns rows t = w, w+8, ... and lane l columns l and l + 32.  For the
// solve warp w owns 8 columns and all their rows, so its depth levels (a node
// only needs its ancestors) are separated by warp syncs, not block barriers.
// The path ratios g_t / g_i are products of alpha along the chain from i down
// to t, so no division is made and deep paths cannot produce 0/0.
//
// tv_gdn_commit: one CTA per (sequence, value head, 32 rows of S^T): S_0 read
// once, the accepted path's rank-n_acc update added, S written once.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tv_gdn.h"

TV_DEBUG_RECORD(gdn)

namespace tv {
namespace {

constexpr int kGdnDC = 64;     // d_v columns per CTA (lane l owns l and l + 32)
constexpr int kGcDC = 32;      // rows of S^T per commit CTA
constexpr int kGdnWarps = 8;
constexpr int kGdnThreads = 32 * kGdnWarps;
constexpr int kGdnMaxN = 64;

__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.b32 %0, 1, 0, e;\n\t}"
               : "=r"(p));
  return p != 0;
}

// 16-byte asynchronous global -> shared copy (completes at cp_async_wait_all)
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

struct GdnLayout {
  int N, dk;
  size_t off_s, off_k, off_q, off_x, off_y, off_u, off_g, off_al, off_be, off_anc, off_par,
      off_dep, bytes;
};

constexpr int kGdnUStride = kGdnDC + 1;  // U rows padded: the solve reads U down columns

__host__ __device__ inline GdnLayout gdn_layout(int N, int dk) {
  GdnLayout L;
  L.N = N;
  L.dk = dk;
  size_t o = 0;
  L.off_s = o; o += (size_t)kGdnDC * (dk + 4) * 4;
  L.off_k = o; o += (size_t)N * (dk + 4) * 4;
  L.off_q = o; o += (size_t)N * (dk + 4) * 4;
  L.off_x = o; o += (size_t)N * (N + 1) * 4;
  L.off_y = o; o += (size_t)N * (N + 1) * 4;
  L.off_u = o; o += (size_t)N * kGdnUStride * 4;
  L.off_g = o; o += (size_t)N * 4;
  L.off_al = o; o += (size_t)N * 4;
  L.off_be = o; o += (size_t)N * 4;
  o = (o + 7) / 8 * 8;
  L.off_anc = o; o += (size_t)N * 8;
  L.off_par = o; o += (size_t)N * 4;
  L.off_dep = o; o += (size_t)N * 4;
  L.bytes = o + 16;
  return L;
}

// ROWS: rows of the tree per warp in the K S_0 / Q S_0 product (N <= 8 * ROWS).
template <int ROWS>
__global__ void __launch_bounds__(kGdnThreads)
gdn_tree_verify_kernel(const float *__restrict__ state, const __nv_bfloat16 *__restrict__ q,
                       const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                       const float *__restrict__ alpha, const float *__restrict__ beta,
                       const uint64_t *__restrict__ anc, int N, int Hk, int Hv, int dk, int dv,
                       float *__restrict__ out, float *__restrict__ u_out,
                       float *__restrict__ g_out, const int32_t *__restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (status && status[b] != 0) return;
  const GdnLayout Ly = gdn_layout(N, dk);
  const int ks = dk + 4;                                   // padded row stride of S, K, Q
  float *sS = reinterpret_cast<float *>(smem + Ly.off_s);  // [64][dk + 4]  rows of S_0^T
  float *sK = reinterpret_cast<float *>(smem + Ly.off_k);  // [N][dk + 4]
  float *sQ = reinterpret_cast<float *>(smem + Ly.off_q);
  float *sX = reinterpret_cast<float *>(smem + Ly.off_x);  // [N][N + 1]
  float *sY = reinterpret_cast<float *>(smem + Ly.off_y);
  float *sU = reinterpret_cast<float *>(smem + Ly.off_u);  // [N][65]
  float *sg = reinterpret_cast<float *>(smem + Ly.off_g);
  float *sal = reinterpret_cast<float *>(smem + Ly.off_al);
  float *sbe = reinterpret_cast<float *>(smem + Ly.off_be);
  uint64_t *sanc = reinterpret_cast<uint64_t *>(smem + Ly.off_anc);
  int *spar = reinterpret_cast<int *>(smem + Ly.off_par);
  int *sdep = reinterpret_cast<int *>(smem + Ly.off_dep);
  __shared__ int s_maxdep;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int hk = h / (Hv / Hk);
  const int j0 = c * kGdnDC + lane;  // this lane's columns: j0 and j0 + 32

  // 1. the 64 rows of S_0^T this CTA owns: asynchronous copies, in flight
  //    through everything up to the product
  const float *s0 = state + (((size_t)b * Hv + h) * dv + (size_t)c * kGdnDC) * dk;
  for (int e = tid * 4; e < kGdnDC * dk; e += kGdnThreads * 4) {
    const int r = e / dk, i = e - r * dk;
    cp_async16(sS + r * ks + i, s0 + (size_t)r * dk + i);
  }
  // 2. everything else this CTA reads, loads issued before any is used
  constexpr int kKqIter = kGdnMaxN * 128 / (kGdnThreads * 8);  // at most 4
  uint4 kw[kKqIter], qw[kKqIter];
#pragma unroll
  for (int it = 0; it < kKqIter; ++it) {
    const int e = (tid + it * kGdnThreads) * 8;
    if (e < N * dk) {
      const int t = e / dk, i = e - t * dk;
      const size_t src = (((size_t)b * N + t) * Hk + hk) * dk + i;
      kw[it] = *reinterpret_cast<const uint4 *>(k + src);
      qw[it] = *reinterpret_cast<const uint4 *>(q + src);
    }
  }
  float vpre[ROWS][2];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int t = min(w + kGdnWarps * r, N - 1);
    const __nv_bfloat16 *vt = v + (((size_t)b * N + t) * Hv + h) * dv + j0;
    vpre[r][0] = __bfloat162float(vt[0]);
    vpre[r][1] = __bfloat162float(vt[32]);
  }
  if (tid == 0) s_maxdep = 0;
  for (int t = tid; t < N; t += kGdnThreads) {
    const uint64_t m = anc[(size_t)b * N + t];
    sanc[t] = m;
    sdep[t] = __popcll(m);
    // the deepest strict ancestor (only bits below t count, so every chain
    // walked through spar strictly descends and ends)
    const uint64_t strict = m & ((1ull << t) - 1);
    spar[t] = strict ? 63 - __clzll((long long)strict) : -1;
    sal[t] = alpha[((size_t)b * N + t) * Hv + h];
    sbe[t] = beta[((size_t)b * N + t) * Hv + h];
  }
#pragma unroll
  for (int it = 0; it < kKqIter; ++it) {
    const int e = (tid + it * kGdnThreads) * 8;
    if (e < N * dk) {
      const int t = e / dk, i = e - t * dk;
      const uint32_t kk[4] = {kw[it].x, kw[it].y, kw[it].z, kw[it].w};
      const uint32_t qq[4] = {qw[it].x, qw[it].y, qw[it].z, qw[it].w};
      float4 *dk4 = reinterpret_cast<float4 *>(sK + t * ks + i);
      float4 *dq4 = reinterpret_cast<float4 *>(sQ + t * ks + i);
      dk4[0] = make_float4(bf16_lo(kk[0]), bf16_hi(kk[0]), bf16_lo(kk[1]), bf16_hi(kk[1]));
      dk4[1] = make_float4(bf16_lo(kk[2]), bf16_hi(kk[2]), bf16_lo(kk[3]), bf16_hi(kk[3]));
      dq4[0] = make_float4(bf16_lo(qq[0]), bf16_hi(qq[0]), bf16_lo(qq[1]), bf16_hi(qq[1]));
      dq4[1] = make_float4(bf16_lo(qq[2]), bf16_hi(qq[2]), bf16_lo(qq[3]), bf16_hi(qq[3]));
    }
  }
  __syncthreads();
  // 3. path products g_t (each node walks its own chain) and the deepest level
  for (int t = tid; t < N; t += kGdnThreads) {
    float gt = 1.f;
    for (int i = t; i >= 0; i = spar[i]) gt *= sal[i];
    sg[t] = gt;
    atomicMax(&s_maxdep, sdep[t]);
  }
  // 4. the ancestor pairs, one thread each: X_ti = beta_t (g_t/g_i) k_t.k_i on
  //    strict ancestors, Y_ti = (g_t/g_i) q_t.k_i on ancestors-or-self; g_t/g_i
  //    is the product of alpha over the chain from t up to (not including) i
  __syncthreads();
  const int maxdep = s_maxdep;
  for (int idx = tid; idx < N * maxdep; idx += kGdnThreads) {
    const int t = idx % N, jup = idx / N;
    int i = t;
    float gam = 1.f;
    for (int s = 0; s < jup && i >= 0; ++s) {
      gam *= sal[i];
      i = spar[i];
    }
    if (i < 0) continue;  // the chain of t is shorter than jup
    float kk = 0.f, qk = 0.f;
    for (int e = 0; e < dk; e += 4) {
      const float4 a = *reinterpret_cast<const float4 *>(sK + t * ks + e);
      const float4 qa = *reinterpret_cast<const float4 *>(sQ + t * ks + e);
      const float4 bb = *reinterpret_cast<const float4 *>(sK + i * ks + e);
      kk = fmaf(a.x, bb.x, fmaf(a.y, bb.y, fmaf(a.z, bb.z, fmaf(a.w, bb.w, kk))));
      qk = fmaf(qa.x, bb.x, fmaf(qa.y, bb.y, fmaf(qa.z, bb.z, fmaf(qa.w, bb.w, qk))));
    }
    sY[t * (N + 1) + i] = gam * qk;
    if (jup > 0) sX[t * (N + 1) + i] = sbe[t] * gam * kk;
  }
  // 5. K S_0 and Q S_0: warp w owns rows w, w+8, ... (clamped: spare rows
  //    recompute row N-1 and are dropped), lane l columns l and l+32
  cp_async_wait_all();
  __syncthreads();
  float accp[ROWS][2], accr[ROWS][2];
#pragma unroll
  for (int r = 0; r < ROWS; ++r)
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) accp[r][cc] = accr[r][cc] = 0.f;
  int trow[ROWS];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) trow[r] = min(w + kGdnWarps * r, N - 1);
  for (int i = 0; i < dk; i += 4) {
    const float4 sa = *reinterpret_cast<const float4 *>(sS + lane * ks + i);
    const float4 sb = *reinterpret_cast<const float4 *>(sS + (lane + 32) * ks + i);
    float4 k4[ROWS], q4[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      k4[r] = *reinterpret_cast<const float4 *>(sK + trow[r] * ks + i);
      q4[r] = *reinterpret_cast<const float4 *>(sQ + trow[r] * ks + i);
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      accp[r][0] = fmaf(k4[r].x, sa.x, fmaf(k4[r].y, sa.y, fmaf(k4[r].z, sa.z, fmaf(k4[r].w, sa.w, accp[r][0]))));
      accp[r][1] = fmaf(k4[r].x, sb.x, fmaf(k4[r].y, sb.y, fmaf(k4[r].z, sb.z, fmaf(k4[r].w, sb.w, accp[r][1]))));
      accr[r][0] = fmaf(q4[r].x, sa.x, fmaf(q4[r].y, sa.y, fmaf(q4[r].z, sa.z, fmaf(q4[r].w, sa.w, accr[r][0]))));
      accr[r][1] = fmaf(q4[r].x, sb.x, fmaf(q4[r].y, sb.y, fmaf(q4[r].z, sb.z, fmaf(q4[r].w, sb.w, accr[r][1]))));
    }
  }
  // 6. right-hand sides beta_t (v_t - g_t (K S_0)_t) into U
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int t = w + kGdnWarps * r;
    if (t < N) {
      sU[t * kGdnUStride + lane] = sbe[t] * (vpre[r][0] - sg[t] * accp[r][0]);
      sU[t * kGdnUStride + lane + 32] = sbe[t] * (vpre[r][1] - sg[t] * accp[r][1]);
    }
  }
  __syncthreads();
  // 7. forward substitution: warp w owns columns 8w .. 8w+7 of U and every row
  //    of them (lane l rows l and l+32), so the depth levels only need the warp
  {
    const int col0 = 8 * w;
    for (int d = 2; d <= maxdep; ++d) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int t = lane + 32 * rr;
        if (t < N && sdep[t] == d) {
          float x[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) x[cc] = sU[t * kGdnUStride + col0 + cc];
          for (int i = spar[t]; i >= 0; i = spar[i]) {
            const float xt = sX[t * (N + 1) + i];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) x[cc] = fmaf(-xt, sU[i * kGdnUStride + col0 + cc], x[cc]);
          }
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) sU[t * kGdnUStride + col0 + cc] = x[cc];
        }
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // 8. outputs o_t = g_t (Q S_0)_t + sum over ancestors-or-self of Y_ti u_i
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int t = w + kGdnWarps * r;
    if (t < N) {
      float o0 = sg[t] * accr[r][0], o1 = sg[t] * accr[r][1];
      for (int i = t; i >= 0; i = TV_CHECK(spar[i] < i) ? spar[i] : -1) {
        const float y = sY[t * (N + 1) + i];
        o0 = fmaf(y, sU[i * kGdnUStride + lane], o0);
        o1 = fmaf(y, sU[i * kGdnUStride + lane + 32], o1);
      }
      const size_t dst = (((size_t)b * N + t) * Hv + h) * dv + j0;
      if (!TV_CHECK(dst + 32 < (size_t)gridDim.z * N * Hv * dv)) continue;
      out[dst] = o0;
      out[dst + 32] = o1;
      u_out[dst] = sU[t * kGdnUStride + lane];
      u_out[dst + 32] = sU[t * kGdnUStride + lane + 32];
    }
  }
  if (c == 0)
    for (int t = tid; t < N; t += kGdnThreads) g_out[((size_t)b * N + t) * Hv + h] = sg[t];
}

// ------------------------------------------------------------------ tensor cores
//
// d_k in {64, 128}: [K; Q] S_0 on tcgen05.  A = the 2N rows of K and Q (bf16,
// exactly the inputs), B = the 64 state rows split into three bf16 planes
// (hi + mid + lo reproduces the fp32 value to 24 bits), D = 128 x 64 fp32 in
// TMEM, accumulated over the planes.  Both operands are K-major with the
// 128-byte swizzle, written here by the threads (every 16-byte chunk is one
// swizzle unit).  One elected thread issues the 3 * d_k / 16 MMAs and commits
// them to an mbarrier; the CUDA cores work out g, X and Y meanwhile.  Every
// wait is bounded (2 s); on expiry status[b] = TV_ERR_CUDA.

constexpr int kTcM = 128;
constexpr int kTcCols = 64;  // TMEM columns: one fp32 column per d_v column
constexpr unsigned long long kGdnWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t gdn_sw128_desc(uint32_t addr) {
  // start >> 4, leading offset 16 B, stride 1024 B between 8-row groups,
  // descriptor version 1, 128-byte swizzle
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(16 >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// kind::f16 instruction descriptor: fp32 D, bf16 A and B, both K-major
__host__ __device__ constexpr uint32_t gdn_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// byte offset of 16-byte chunk ch (0..7) of row r in a [rows][64] bf16 half tile
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  return (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint64_t gdn_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __noinline__ bool gdn_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = gdn_timer();
  for (uint32_t i = 0;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && gdn_timer() - t0 > kGdnWaitNs) return false;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}

struct GdnTcLayout {
  size_t off_a, off_b, off_x, off_y, off_u, off_r, off_g, off_al, off_be, off_anc, off_par,
      off_dep, bytes;
};

__host__ __device__ inline GdnTcLayout gdn_tc_layout(int N, int dk) {
  GdnTcLayout L;
  const int halves = dk / 64;
  size_t o = 0;
  L.off_a = o; o += (size_t)halves * kTcM * 128;       // [halves][128][64] bf16
  L.off_b = o; o += (size_t)3 * halves * kTcCols * 128; // [3 planes][halves][64][64] bf16
  L.off_x = o; o += (size_t)N * (N + 1) * 4;
  L.off_y = o; o += (size_t)N * (N + 1) * 4;
  L.off_u = o; o += (size_t)N * kGdnUStride * 4;
  L.off_r = o; o += (size_t)N * kGdnUStride * 4;        // Q S_0 rows, staged from TMEM
  L.off_g = o; o += (size_t)N * 4;
  L.off_al = o; o += (size_t)N * 4;
  L.off_be = o; o += (size_t)N * 4;
  o = (o + 7) / 8 * 8;
  L.off_anc = o; o += (size_t)N * 8;
  L.off_par = o; o += (size_t)N * 4;
  L.off_dep = o; o += (size_t)N * 4;
  L.bytes = o + 1024;  // slack: the tile base is rounded up to 1024 B
  return L;
}

__global__ void __launch_bounds__(kGdnThreads)
gdn_tree_verify_tc_kernel(const float *__restrict__ state, const __nv_bfloat16 *__restrict__ q,
                          const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                          const float *__restrict__ alpha, const float *__restrict__ beta,
                          const uint64_t *__restrict__ anc, int N, int Hk, int Hv, int dk, int dv,
                          float *__restrict__ out, float *__restrict__ u_out,
                          float *__restrict__ g_out, int32_t *__restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ int s_maxdep;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (status && status[b] != 0) return;
  const GdnTcLayout Ly = gdn_tc_layout(N, dk);
  const uint32_t raw = ptx::smem_u32(smem_raw);
  unsigned char *smem = smem_raw + (((raw + 1023) & ~1023u) - raw);
  unsigned char *sA = smem + Ly.off_a;
  unsigned char *sB = smem + Ly.off_b;
  float *sX = reinterpret_cast<float *>(smem + Ly.off_x);  // [N][N + 1]
  float *sY = reinterpret_cast<float *>(smem + Ly.off_y);
  float *sU = reinterpret_cast<float *>(smem + Ly.off_u);  // [N][65]
  float *sR = reinterpret_cast<float *>(smem + Ly.off_r);  // [N][65]
  float *sg = reinterpret_cast<float *>(smem + Ly.off_g);
  float *sal = reinterpret_cast<float *>(smem + Ly.off_al);
  float *sbe = reinterpret_cast<float *>(smem + Ly.off_be);
  uint64_t *sanc = reinterpret_cast<uint64_t *>(smem + Ly.off_anc);
  int *spar = reinterpret_cast<int *>(smem + Ly.off_par);
  int *sdep = reinterpret_cast<int *>(smem + Ly.off_dep);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int hk = h / (Hv / Hk);
  const int halves = dk / 64;
  const uint32_t half_a = kTcM * 128, half_b = kTcCols * 128, plane_b = halves * half_b;

  if (w == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), kTcCols);
    ptx::tmem_relinquish();
  }
  if (tid == 32) {
    ptx::mbar_init(ptx::smem_u32(&s_bar), 1);
    ptx::fence_mbar_init();
    s_maxdep = 0;
  }
  // 1. loads, all issued before use: K / Q chunks, the state rows, v of this
  //    thread's right-hand-side row
  const int nkq = 2 * N * dk / 8;                 // 16-byte chunks of K and Q
  constexpr int kKqIt = 2 * kGdnMaxN * 128 / 8 / kGdnThreads;  // at most 8
  uint4 kq[kKqIt];
#pragma unroll
  for (int it = 0; it < kKqIt; ++it) {
    const int e = tid + it * kGdnThreads;
    if (e < nkq) {
      const int isq = e >= N * dk / 8, rem = isq ? e - N * dk / 8 : e;
      const int t = rem / (dk / 8), i = (rem - t * (dk / 8)) * 8;
      const __nv_bfloat16 *src = (isq ? q : k) + (((size_t)b * N + t) * Hk + hk) * dk + i;
      kq[it] = *reinterpret_cast<const uint4 *>(src);
    }
  }
  const float *s0 = state + (((size_t)b * Hv + h) * dv + (size_t)c * kTcCols) * dk;
  constexpr int kSIt = kTcCols * 128 / 8 / kGdnThreads;  // chunks of 8 per thread: at most 4
  float4 sv[kSIt][2];
#pragma unroll
  for (int it = 0; it < kSIt; ++it) {
    const int e = (tid + it * kGdnThreads) * 8;
    if (e < kTcCols * dk) {
      sv[it][0] = __ldg(reinterpret_cast<const float4 *>(s0 + e));
      sv[it][1] = __ldg(reinterpret_cast<const float4 *>(s0 + e + 4));
    }
  }
  const int quad = w & 3, chalf = w >> 2;  // TMEM lane quadrant, 32-column half
  const int drow = 32 * quad + lane;       // the D row this thread reads
  uint4 vq[4];
  if (drow < N) {
    const uint4 *vs = reinterpret_cast<const uint4 *>(
        v + (((size_t)b * N + drow) * Hv + h) * dv + (size_t)c * kTcCols + 32 * chalf);
#pragma unroll
    for (int p = 0; p < 4; ++p) vq[p] = vs[p];
  }
  for (int t = tid; t < N; t += kGdnThreads) {
    const uint64_t m = anc[(size_t)b * N + t];
    sanc[t] = m;
    sdep[t] = __popcll(m);
    const uint64_t strict = m & ((1ull << t) - 1);
    spar[t] = strict ? 63 - __clzll((long long)strict) : -1;
    sal[t] = alpha[((size_t)b * N + t) * Hv + h];
    sbe[t] = beta[((size_t)b * N + t) * Hv + h];
  }
  // 2. operands into the swizzled tiles
#pragma unroll
  for (int it = 0; it < kKqIt; ++it) {
    const int e = tid + it * kGdnThreads;
    if (e < nkq) {
      const int isq = e >= N * dk / 8, rem = isq ? e - N * dk / 8 : e;
      const int t = rem / (dk / 8), i = (rem - t * (dk / 8)) * 8;
      const int row = isq ? N + t : t;
      *reinterpret_cast<uint4 *>(sA + (i >> 6) * half_a + swz(row, (i & 63) >> 3)) = kq[it];
    }
  }
#pragma unroll
  for (int it = 0; it < kSIt; ++it) {
    const int e = (tid + it * kGdnThreads) * 8;
    if (e < kTcCols * dk) {
      const int r = e / dk, i = e - r * dk;
      const float x[8] = {sv[it][0].x, sv[it][0].y, sv[it][0].z, sv[it][0].w,
                          sv[it][1].x, sv[it][1].y, sv[it][1].z, sv[it][1].w};
      float hi[8], mid[8], lo[8];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        hi[p] = __bfloat162float(__float2bfloat16_rn(x[p]));
        const float r1 = x[p] - hi[p];
        mid[p] = __bfloat162float(__float2bfloat16_rn(r1));
        lo[p] = r1 - mid[p];
      }
      const uint32_t off = (i >> 6) * half_b + swz(r, (i & 63) >> 3);
      *reinterpret_cast<uint4 *>(sB + off) =
          make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                     pack_bf16x2(hi[4], hi[5]), pack_bf16x2(hi[6], hi[7]));
      *reinterpret_cast<uint4 *>(sB + plane_b + off) =
          make_uint4(pack_bf16x2(mid[0], mid[1]), pack_bf16x2(mid[2], mid[3]),
                     pack_bf16x2(mid[4], mid[5]), pack_bf16x2(mid[6], mid[7]));
      *reinterpret_cast<uint4 *>(sB + 2 * plane_b + off) =
          make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                     pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
    }
  }
  ptx::fence_proxy_async_smem();  // the tiles are read by the tensor cores next
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t bar = ptx::smem_u32(&s_bar);
  // 3. the MMAs: one elected thread
  if (w == 0) {
    if (elect_one()) {
      const uint32_t a0 = ptx::smem_u32(sA), b0 = ptx::smem_u32(sB);
      const uint32_t idesc = gdn_idesc(kTcM, kTcCols);
      for (int p = 0; p < 3; ++p)
        for (int kk = 0; kk < dk / 16; ++kk) {
          const uint32_t in = (kk >> 2), ks = (kk & 3) * 32;
          const uint64_t ad = gdn_sw128_desc(a0 + in * half_a + ks);
          const uint64_t bd = gdn_sw128_desc(b0 + p * plane_b + in * half_b + ks);
          ptx::umma_f16(tmem, ad, bd, idesc, (p | kk) != 0);
        }
      ptx::umma_commit(bar);
    }
    __syncwarp();
  }
  // 4. meanwhile: path products, then the ancestor pairs from the bf16 tile
  for (int t = tid; t < N; t += kGdnThreads) {
    float gt = 1.f;
    for (int i = t; i >= 0; i = spar[i]) gt *= sal[i];
    sg[t] = gt;
    atomicMax(&s_maxdep, sdep[t]);
  }
  __syncthreads();
  const int maxdep = s_maxdep;
  for (int idx = tid; idx < N * maxdep; idx += kGdnThreads) {
    const int t = idx % N, jup = idx / N;
    int i = t;
    float gam = 1.f;
    for (int s2 = 0; s2 < jup && i >= 0; ++s2) {
      gam *= sal[i];
      i = spar[i];
    }
    if (i < 0) continue;
    float kk = 0.f, qk = 0.f;
    for (int hf = 0; hf < halves; ++hf)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 a = *reinterpret_cast<const uint4 *>(sA + hf * half_a + swz(t, ch));
        const uint4 qa = *reinterpret_cast<const uint4 *>(sA + hf * half_a + swz(N + t, ch));
        const uint4 bb = *reinterpret_cast<const uint4 *>(sA + hf * half_a + swz(i, ch));
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, qw[4] = {qa.x, qa.y, qa.z, qa.w},
                       bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          kk = fmaf(bf16_lo(aw[p]), bf16_lo(bw[p]), fmaf(bf16_hi(aw[p]), bf16_hi(bw[p]), kk));
          qk = fmaf(bf16_lo(qw[p]), bf16_lo(bw[p]), fmaf(bf16_hi(qw[p]), bf16_hi(bw[p]), qk));
        }
      }
    sY[t * (N + 1) + i] = gam * qk;
    if (jup > 0) sX[t * (N + 1) + i] = sbe[t] * gam * kk;
  }
  // 5. the product: D row d (K row d, or Q row d - N), 32 columns per warp
  bool ok = gdn_wait(bar, 0);
  if (!ok) ok = gdn_wait(bar, 0);  // a second bounded chance before TMEM is freed
  ptx::tc_fence_after();
  uint32_t dv32[32];
  ptx::tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + 32 * chalf, dv32);
  ptx::tmem_wait_ld();
  if (!ok && tid == 0) set_status(status, b, TV_ERR_CUDA);
  // 6. right-hand sides beta_t (v_t - g_t (K S_0)_t) into U
  if (drow < N) {
    const int t = drow;
    const float bt = sbe[t], gt = sg[t];
    const uint32_t vw[16] = {vq[0].x, vq[0].y, vq[0].z, vq[0].w, vq[1].x, vq[1].y, vq[1].z, vq[1].w,
                             vq[2].x, vq[2].y, vq[2].z, vq[2].w, vq[3].x, vq[3].y, vq[3].z, vq[3].w};
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const float vv = (jj & 1) ? bf16_hi(vw[jj >> 1]) : bf16_lo(vw[jj >> 1]);
      sU[t * kGdnUStride + 32 * chalf + jj] = bt * (vv - gt * __uint_as_float(dv32[jj]));
    }
  } else if (drow < 2 * N) {  // a Q row: stage (Q S_0)_t for the output phase
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) sR[(drow - N) * kGdnUStride + 32 * chalf + jj] = __uint_as_float(dv32[jj]);
  }
  __syncthreads();
  // 7. forward substitution (warp w: columns 8w .. 8w+7, every row)
  {
    const int col0 = 8 * w;
    for (int d = 2; d <= maxdep; ++d) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int t = lane + 32 * rr;
        if (t < N && sdep[t] == d) {
          float x[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) x[cc] = sU[t * kGdnUStride + col0 + cc];
          for (int i = spar[t]; i >= 0; i = spar[i]) {
            const float xt = sX[t * (N + 1) + i];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) x[cc] = fmaf(-xt, sU[i * kGdnUStride + col0 + cc], x[cc]);
          }
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) sU[t * kGdnUStride + col0 + cc] = x[cc];
        }
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // 8. outputs o_t = g_t (Q S_0)_t + sum over ancestors-or-self of Y_ti u_i:
  //    warp w rows w, w+8, ...; lane l columns l and l+32 (coalesced writes)
  for (int t = w; t < N; t += kGdnWarps) {
    const float gt = sg[t];
    float o0 = gt * sR[t * kGdnUStride + lane], o1 = gt * sR[t * kGdnUStride + lane + 32];
    for (int i = t; i >= 0; i = TV_CHECK(spar[i] < i) ? spar[i] : -1) {
      const float y = sY[t * (N + 1) + i];
      o0 = fmaf(y, sU[i * kGdnUStride + lane], o0);
      o1 = fmaf(y, sU[i * kGdnUStride + lane + 32], o1);
    }
    const size_t dst = (((size_t)b * N + t) * Hv + h) * dv + (size_t)c * kTcCols + lane;
    if (!TV_CHECK(dst + 32 < (size_t)gridDim.z * N * Hv * dv)) continue;
    out[dst] = o0;
    out[dst + 32] = o1;
    u_out[dst] = sU[t * kGdnUStride + lane];
    u_out[dst + 32] = sU[t * kGdnUStride + lane + 32];
  }
  if (c == 0)
    for (int t = tid; t < N; t += kGdnThreads) g_out[((size_t)b * N + t) * Hv + h] = sg[t];
  ptx::tc_fence_before();
  __syncthreads();
  if (w == 0) ptx::tmem_dealloc(tmem, kTcCols);
}

// ----------------------------------------------------------------------------
// gdn_tree_verify_pipe_kernel: the same verification as a persistent,
// warp-specialised pipeline.  One CTA per SM walks the (sequence, value head)
// items blockIdx.x, blockIdx.x + gridDim.x, ...; while one item is solved the
// state of the next is in flight.  Trees of at most 32 nodes; d_k 64 or 128,
// d_v 64 or 128.
//
// Roles (12 warps, three warpgroups):
//   warps 0-3   convert the staged fp32 rows of S_0^T to three bf16 planes in
//               TMEM (hi + mid + lo = the fp32 value; thread j owns TMEM lane
//               j = row j); the last warp done with item k sends the TMA of
//               S_0^T (fp32, [d_v rows][d_k], 128-byte swizzled boxes of 32
//               columns) for item k + 2 into the staging buffer k leaves, and
//               warp 2, the only MMA issuer, issues D1 = S_0^T [K; Q]^T (A =
//               the planes in TMEM, B = the [K; Q] tile) and the node pairs
//               D2 = [K; Q] K^T;
//   warps 4-7, 8-11  two post-processing warpgroups, alternate items; each
//               loads its own items' [K; Q] (32 rows each, bf16, swizzled), V
//               (32 rows) and, by asynchronous copies, the per-node alpha,
//               beta, ancestor masks and status word, the next as soon as it
//               has read the current stage; from
//               D2 the masked matrices X and Y (one thread per tree row), then
//               per column j of d_v (thread j, its TMEM lane of D1) the
//               right-hand sides, the triangular solve for U and the outputs,
//               dense over the 32 rows (zero off the ancestor pairs) with U in
//               registers and packed fp32 FMAs.
// TMEM: two plane buffers (item k in buffer k % 2) at columns 0 and 192, each
// [0, 3 d_k / 2); one D at 384 (D1, K S_0 then Q S_0, in 64 columns; D2 at
// 448): the post-processing warps copy it to registers as soon as it is ready,
// and the MMAs of the next item wait for that (d_empty); d_full[k % 2] tells
// the warpgroup of item k.  Each wait is bounded
// (2 s); a wait that runs out raises a CTA-wide abort, every role leaves its
// loop, copies in flight get a bounded chance to land, and status[b] of the
// item is set to TV_ERR_CUDA.

constexpr int kPipeN = 32;  // tree rows per tile
constexpr int kPipeWarps = 12;
constexpr int kPipeThreads = 32 * kPipeWarps;
constexpr uint32_t kPipeStage = 25 * 1024;  // [K; Q] halves (2 x 8 KB), V (8 KB), scalars
constexpr uint32_t kPipeOffV = 16384;
constexpr uint32_t kPipeOffMeta = 24576;    // alpha [32], beta [32], anc [32], status word
constexpr uint32_t kPipeOffStg = 2 * kPipeStage;
constexpr uint32_t kPipeStgBytes = 128 * 128 * 4;  // S_0^T of one head, fp32
constexpr uint32_t kPipeOffScr = kPipeOffStg + 2 * kPipeStgBytes;
constexpr int kPipeXS = 36;  // row stride of X and Y (floats; rows 16-byte aligned)
constexpr uint32_t kPipeScrBytes = (2 * kPipeN * kPipeXS + 2 * kPipeN) * 4;  // X, Y, g, beta
constexpr uint32_t kPipeSmem = kPipeOffScr + 4 * kPipeScrBytes + 1024;
constexpr uint32_t kPipeTmemCols = 512;
constexpr uint32_t kPipeColPlanes = 192;  // planes buffer s at 192 s
constexpr uint32_t kPipeColD = 384;       // D1 at 384, D2 at 448
static_assert(kPipeSmem <= 227 * 1024, "shared memory budget");

struct PipeBars {
  unsigned long long s0_full[2], kqv_full[2];
  unsigned long long planes_full[2], planes_empty[2];
  unsigned long long d_full[2], d_empty, wg[2];
};

__device__ __noinline__ bool pipe_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  const uint64_t t0 = gdn_timer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (gdn_timer() - t0 > kGdnWaitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// every lane of the warp waits; true when the phase completed for all of them
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  const bool ok = ptx::mbar_try_wait(bar, parity) || pipe_wait_slow(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// 4- or 8-byte asynchronous global -> shared copy; `valid` false writes zeros
// (source size 0) without reading the source
__device__ __forceinline__ void cp_async_zfill(uint32_t dst, const void *src, int bytes, bool valid) {
  const int n = valid ? bytes : 0;
  if (bytes == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// x0, x1 -> hi + mid + lo, each a bf16 pair (x0 in the low half); every
// residual is exact in fp32, so the planes sum to x to 24 bits
__device__ __forceinline__ void split3(float x0, float x1, uint32_t &h, uint32_t &m, uint32_t &l) {
  h = ptx::pack_bf16(x0, x1);
  const float2 r = __fadd2_rn(make_float2(x0, x1),
                              make_float2(-__uint_as_float(h << 16), -__uint_as_float(h & 0xffff0000u)));
  m = ptx::pack_bf16(r.x, r.y);
  const float2 q = __fadd2_rn(r, make_float2(-__uint_as_float(m << 16), -__uint_as_float(m & 0xffff0000u)));
  l = ptx::pack_bf16(q.x, q.y);
}

__global__ void __launch_bounds__(kPipeThreads)
gdn_tree_verify_pipe_kernel(const __grid_constant__ CUtensorMap tm_s,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_v,
                            const float *__restrict__ alpha, const float *__restrict__ beta,
                            const uint64_t *__restrict__ anc, int B, int N, int Hk, int Hv,
                            int dk, int dv, float *__restrict__ out, float *__restrict__ u_out,
                            float *__restrict__ g_out, int32_t *__restrict__ status,
                            int withheld_cta) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ PipeBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_s0cnt[2];  // warps done with staging buffer s this round
  __shared__ int s_fills[4];  // copies sent into staging 0, 1 and stage 0, 1
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023) & ~1023u;
  unsigned char *smem = smem_raw + (sb - raw);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int items = B * Hv;
  const int nk = (int)blockIdx.x < items ? (items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int G = Hv / Hk;
  const int halves = dk / 64;

  if (w == 2) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), kPipeTmemCols);
    ptx::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      // test hook: one arrival more than the state copy makes, in one CTA
      ptx::mbar_init(ptx::smem_u32(&bars.s0_full[i]), (i == 0 && (int)blockIdx.x == withheld_cta) ? 2 : 1);
      ptx::mbar_init(ptx::smem_u32(&bars.kqv_full[i]), 33);
      s_s0cnt[i] = 0;
      ptx::mbar_init(ptx::smem_u32(&bars.d_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.planes_full[i]), 128);
      ptx::mbar_init(ptx::smem_u32(&bars.planes_empty[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.wg[i]), 128);
    }
    ptx::mbar_init(ptx::smem_u32(&bars.d_empty), 128);
    for (int i = 0; i < 4; ++i) s_fills[i] = 0;
    s_abort = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int *abort_flag = &s_abort;
  int fail_b = -1;  // the sequence of the item a role gave up on

  // The copies.  S_0^T of item kk into staging buffer kk % 2 (one thread);
  // [K; Q], V, the per-node scalars (zero past N) and the status word (zero
  // without a status array) of item kk into stage kk % 2 (a whole warp; the
  // scalars by asynchronous copies whose arrival on the stage's barrier fires
  // once they have landed, so the warp does not wait for them).
  auto issue_s0 = [&](int kk) {
    const int item = (int)blockIdx.x + kk * (int)gridDim.x;
    const uint32_t fb = ptx::smem_u32(&bars.s0_full[kk & 1]);
    ptx::mbar_arrive_expect_tx(fb, (uint32_t)(dv * dk * 4));
    const uint32_t dst = sb + kPipeOffStg + (uint32_t)(kk & 1) * kPipeStgBytes;
    for (int m = 0; m < dk / 32; ++m)
      ptx::tma_load_2d(dst + (uint32_t)(m * dv * 128), &tm_s, fb, 32 * m, item * dv);
    s_fills[kk & 1] = kk / 2 + 1;
  };
  auto issue_kqv = [&](int kk) {
    const int item = (int)blockIdx.x + kk * (int)gridDim.x;
    const int b = item / Hv, h = item - b * Hv, hk = h / G;
    const int q = kk & 1;
    const uint32_t st = sb + (uint32_t)q * kPipeStage;
    const uint32_t fb = ptx::smem_u32(&bars.kqv_full[q]);
    if (lane == 0) {
      // rows past N are the next sequence's nodes or zero fill past the end
      ptx::mbar_arrive_expect_tx(fb, (uint32_t)(halves * 8192 + 64 * dv));
      for (int hf = 0; hf < halves; ++hf) {
        ptx::tma_load_2d(st + hf * 8192, &tm_k, fb, hk * dk + 64 * hf, b * N);
        ptx::tma_load_2d(st + hf * 8192 + 4096, &tm_q, fb, hk * dk + 64 * hf, b * N);
      }
      ptx::tma_load_2d(st + kPipeOffV, &tm_v, fb, h * dv, b * N);
      s_fills[2 + q] = kk / 2 + 1;
    }
    const uint32_t meta = st + kPipeOffMeta;
    const int t = lane;
    const size_t bt = (size_t)b * N + (t < N ? t : 0);
    cp_async_zfill(meta + 4 * t, alpha + bt * Hv + h, 4, t < N);
    cp_async_zfill(meta + 128 + 4 * t, beta + bt * Hv + h, 4, t < N);
    cp_async_zfill(meta + 256 + 8 * t, anc + bt, 8, t < N);
    if (t == 0)
      cp_async_zfill(meta + 512, status ? static_cast<const void *>(status + b) : static_cast<const void *>(alpha), 4,
                     status != nullptr);
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(fb) : "memory");
  };

  if (w < 4) {
    // ---------------------------------------------------------- warpgroup 0
    // Every warp converts a quarter of the rows (thread j owns TMEM lane j =
    // row j of S_0^T) into plane buffer k % 2; the last warp done with item k
    // sends the copy of S_0^T for item k + 2 into the staging buffer item k
    // leaves; warp 2, the only MMA issuer, then issues the MMAs of item k.
    const int qd = w, j = 32 * qd + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    if (w == 0 && lane == 0) {
      ptx::prefetch_tensormap(&tm_s);
      for (int kk = 0; kk < 2 && kk < nk; ++kk) issue_s0(kk);
    }
    const uint32_t idesc1 = gdn_idesc(kTcM, 2 * kPipeN);  // D1: N = 64 ([K; Q] rows)
    const uint32_t idesc2 = gdn_idesc(kTcM, kPipeN);      // D2: N = 32 (K rows)
    int issued_mma = 0;
    int k = 0;
    for (; k < nk; ++k) {
      const int s = k & 1;
      // ---- convert item k
      if (!warp_wait(ptx::smem_u32(&bars.s0_full[s]), (uint32_t)((k >> 1) & 1), abort_flag) ||
          (k >= 2 && !warp_wait(ptx::smem_u32(&bars.planes_empty[s]), (uint32_t)(((k >> 1) - 1) & 1), abort_flag)))
        break;
      ptx::tc_fence_after();
      const unsigned char *stg = smem + kPipeOffStg + (size_t)s * kPipeStgBytes;
      for (int m = 0; m < dk / 32; ++m) {
        float x[32];
        if (j < dv) {
          const unsigned char *row = stg + (size_t)m * dv * 128 + (size_t)j * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 v4 = *reinterpret_cast<const float4 *>(row + ((c ^ (j & 7)) << 4));
            x[4 * c] = v4.x;
            x[4 * c + 1] = v4.y;
            x[4 * c + 2] = v4.z;
            x[4 * c + 3] = v4.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = 0.f;
        }
        uint32_t hi[16], mid[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) split3(x[2 * e], x[2 * e + 1], hi[e], mid[e], lo[e]);
        const uint32_t tp = tl + kPipeColPlanes * (uint32_t)s;
        tmem_st16(tp + (uint32_t)(16 * m), hi);
        tmem_st16(tp + (uint32_t)(dk / 2 + 16 * m), mid);
        tmem_st16(tp + (uint32_t)(dk + 16 * m), lo);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.planes_full[s]));
      // ---- the last of the four warps to leave staging buffer s refills it
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&s_s0cnt[s], 1) == 3) {
          s_s0cnt[s] = 0;
          if (k + 2 < nk) {
            ptx::fence_proxy_async_smem();
            issue_s0(k + 2);
          }
        }
      }
      __syncwarp();
      // ---- the MMAs of item k (the issuing thread stalls while the tensor
      //      core's queue is full: about the time the MMAs take)
      if (w == 2) {
        const int q = k & 1, n = k >> 1;
        if (!warp_wait(ptx::smem_u32(&bars.planes_full[q]), (uint32_t)(n & 1), abort_flag) ||
            !warp_wait(ptx::smem_u32(&bars.kqv_full[q]), (uint32_t)(n & 1), abort_flag) ||
            (k >= 1 && !warp_wait(ptx::smem_u32(&bars.d_empty), (uint32_t)((k - 1) & 1), abort_flag)))
          break;
        ptx::tc_fence_after();
        const uint32_t kq = sb + (uint32_t)q * kPipeStage;
        const uint32_t d = tmem + kPipeColD;
        const uint32_t ap = tmem + kPipeColPlanes * (uint32_t)q;
        // the [K; Q] tile's descriptor; K step kk starts (kk >> 2) * 8192 +
        // (kk & 3) * 32 bytes in (the same for the three planes and for D2),
        // added to the descriptor's start field (shared addresses stay far
        // below its 256 KB range).  One elected lane issues every MMA.
        const int nkk = dk / 16;
        const uint64_t kd0 = gdn_sw128_desc(kq);
#define KD(kk) (kd0 + (uint64_t)((((kk) >> 2) * 8192 + ((kk) & 3) * 32) >> 4))
        if (ptx::elect_one()) {
#pragma unroll
          for (int pl = 0; pl < 3; ++pl)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              if (kk < nkk)
                ptx::umma_f16_ta(d, ap + (uint32_t)(pl * (dk / 2) + kk * 8), KD(kk), idesc1,
                                 (pl | kk) != 0 ? 1u : 0u);
          // A = the [K; Q] tile read as 128 rows (rows past 64 are other data
          // of the stage: rows of D2 nobody reads), B = its 32 K rows
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            if (kk < nkk) ptx::umma_f16(d + 64, KD(kk), KD(kk), idesc2, kk != 0 ? 1u : 0u);
          ptx::umma_commit(ptx::smem_u32(&bars.planes_empty[q]));
          ptx::umma_commit(ptx::smem_u32(&bars.d_full[q]));
        }
        __syncwarp();
#undef KD
        issued_mma = k + 1;
      }
    }
    if (k < nk) {
      fail_b = ((int)blockIdx.x + k * (int)gridDim.x) / Hv;
      if (w == 2 && lane == 0 && issued_mma > 0) {
        int dummy = 0;  // MMAs in flight finish before TMEM is freed
        pipe_wait_slow(ptx::smem_u32(&bars.planes_empty[(issued_mma - 1) & 1]),
                       (uint32_t)(((issued_mma - 1) >> 1) & 1), &dummy);
      }
    }
  } else {
    // --------------------------------------- X, Y, solve and outputs
    // warpgroup p takes the items k = p, p + 2, ...: stage and D buffer p
    const int pb = (w - 4) >> 2, qd = w & 3, j = 32 * qd + lane;
    // each warpgroup loads its own items' [K; Q], V and scalars: the first
    // now, the next one as soon as all its warps have read the current stage
    if (qd == 0 && pb < nk) {
      if (lane == 0) {
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_v);
      }
      issue_kqv(pb);
    }
    for (int k = pb, n = 0; k < nk; k += 2, ++n) {
      const uint32_t ph = (uint32_t)(n & 1);
      const int item = (int)blockIdx.x + k * (int)gridDim.x;
      const int b = item / Hv, h = item - b * Hv;
      const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16) + kPipeColD;
      const unsigned char *stage = smem + (size_t)pb * kPipeStage;
      const float *ma = reinterpret_cast<const float *>(stage + kPipeOffMeta);
      const float *mb = ma + 32;
      const uint64_t *mc = reinterpret_cast<const uint64_t *>(stage + kPipeOffMeta + 256);
      const uint16_t *sv = reinterpret_cast<const uint16_t *>(stage + kPipeOffV);
      if (!warp_wait(ptx::smem_u32(&bars.kqv_full[pb]), ph, abort_flag) ||
          !warp_wait(ptx::smem_u32(&bars.d_full[pb]), ph, abort_flag)) {
        fail_b = b;
        break;
      }
      ptx::tc_fence_after();
      const bool store = reinterpret_cast<const int *>(stage + kPipeOffMeta + 512)[0] == 0;
      float *X = reinterpret_cast<float *>(smem + kPipeOffScr + (size_t)(2 * pb + (n & 1)) * kPipeScrBytes);
      float *Y = X + kPipeN * kPipeXS;
      float *sg = Y + kPipeN * kPipeXS;
      float *sbeta = sg + kPipeN;
      // D2 and both halves of D1 leave TMEM at once, before the next item's
      // MMAs load the tensor memory, and the D buffer is handed back
      uint32_t dot[32], ks[32], qs[32];
      ptx::tmem_ld32(tl + 64, dot);
      ptx::tmem_ld32(tl, ks);
      ptx::tmem_ld32(tl + 32, qs);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.d_empty));
      // 1. node pairs: lanes 0-31 of D2 are K rows, 32-63 Q rows
      {
        if (qd < 2) {
          const int t = lane;
          const uint64_t msk = mc[t] & ((2ull << t) - 1);  // ancestors-or-self
          const float bt = mb[t];
          float *row = (qd == 0 ? X : Y) + t * kPipeXS;
          // the raw row first, then a short loop (not unrolled: its code is
          // fetched once, not per problem) turns it into the row of X or Y in place
#pragma unroll
          for (int i0 = 0; i0 < kPipeN; i0 += 4)
            *reinterpret_cast<uint4 *>(row + i0) = make_uint4(dot[i0], dot[i0 + 1], dot[i0 + 2], dot[i0 + 3]);
          __syncwarp();
          float gam = 1.f;  // g_t / g_i, built from alpha going up the path
#pragma unroll 1
          for (int i0 = kPipeN - 4; i0 >= 0; i0 -= 4) {  // four columns at a time
            const float4 a4 = *reinterpret_cast<const float4 *>(ma + i0);
            const float4 d4 = *reinterpret_cast<const float4 *>(row + i0);
            const float al[4] = {a4.x, a4.y, a4.z, a4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
            float rv[4];
#pragma unroll
            for (int e = 3; e >= 0; --e) {
              const int i = i0 + e;
              const bool a = (msk >> i) & 1;
              const float dv_i = gam * dd[e];
              rv[e] = qd == 0 ? ((a && i != t) ? bt * dv_i : 0.f) : (a ? dv_i : 0.f);
              gam = a ? gam * al[e] : gam;
            }
            *reinterpret_cast<float4 *>(row + i0) = make_float4(rv[0], rv[1], rv[2], rv[3]);
          }
          if (qd == 0) {
            sg[t] = gam;
            sbeta[t] = bt;
            if (store && t < N) g_out[((size_t)b * N + t) * Hv + h] = gam;
          }
        }
      }
      // this thread's column of V, then the stage may be refilled
      uint32_t vcol[kPipeN / 2];
#pragma unroll
      for (int e = 0; e < kPipeN / 2; ++e)
        vcol[e] = j < dv ? (uint32_t)sv[2 * e * dv + j] | ((uint32_t)sv[(2 * e + 1) * dv + j] << 16) : 0u;
      ptx::mbar_arrive(ptx::smem_u32(&bars.wg[pb]));
      if (!warp_wait(ptx::smem_u32(&bars.wg[pb]), ph, abort_flag)) {
        fail_b = b;
        break;
      }
      // the stage is read (V and the scalars by every warp, [K; Q] by the
      // MMAs behind d_full): the item after next takes it
      if (qd == 0 && k + 2 < nk) issue_kqv(k + 2);
      // 2. column j: right-hand sides and forward substitution (K S_0), then
      //    the outputs (Q S_0)
      const size_t o0 = ((size_t)b * N * Hv + h) * dv + j, rs = (size_t)Hv * dv;
      float *uo = u_out + o0, *oo = out + o0;
      const bool mine = j < dv && TV_CHECK(b < B && h < Hv);
      // U and the products run on pairs (packed fp32 FMA, one rounding per
      // element as fmaf): U2[p] = (u_2p, u_2p+1), rows of X and Y in pairs of
      // columns.  X and Y are zero past each row's own column, and U starts at
      // zero, so a pair that runs one column past the row adds exact zeros.
      float2 U2[kPipeN / 2];
#pragma unroll
      for (int e = 0; e < kPipeN / 2; ++e) U2[e] = make_float2(0.f, 0.f);
      if (mine) {
        // rows in order, each from the rows before it
#pragma unroll
        for (int t = 0; t < kPipeN; ++t) {
          const float vv = __uint_as_float((t & 1) ? (vcol[t >> 1] & 0xffff0000u) : (vcol[t >> 1] << 16));
          const float r = sbeta[t] * (vv - sg[t] * __uint_as_float(ks[t]));
          const float *xr = X + t * kPipeXS;
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < t; i += 4) {
            const float4 c = *reinterpret_cast<const float4 *>(xr + i);
            acc = __ffma2_rn(make_float2(c.x, c.y), U2[i >> 1], acc);
            if (i + 2 < t) acc = __ffma2_rn(make_float2(c.z, c.w), U2[(i >> 1) + 1], acc);
          }
          const float ut = r - (acc.x + acc.y);
          if (t & 1) U2[t >> 1].y = ut;
          else U2[t >> 1].x = ut;
        }
        if (store) {
#pragma unroll
          for (int t = 0; t < kPipeN; ++t)
            {
              if (t < N) *uo = (t & 1) ? U2[t >> 1].y : U2[t >> 1].x;
              uo += rs;
            }
        }
        // outputs: independent dot products over ancestors-or-self
#pragma unroll
        for (int t = 0; t < kPipeN; ++t) {
          const float *yr = Y + t * kPipeXS;
          float2 acc = make_float2(sg[t] * __uint_as_float(qs[t]), 0.f);
#pragma unroll
          for (int i = 0; i <= t; i += 4) {
            const float4 c = *reinterpret_cast<const float4 *>(yr + i);
            acc = __ffma2_rn(make_float2(c.x, c.y), U2[i >> 1], acc);
            if (i + 2 <= t) acc = __ffma2_rn(make_float2(c.z, c.w), U2[(i >> 1) + 1], acc);
          }
          if (store && t < N) *oo = acc.x + acc.y;
          oo += rs;
        }
      }
    }
  }
  if (fail_b >= 0 && lane == 0) set_status(status, fail_b, TV_ERR_CUDA);

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // copies still in flight get a bounded chance to land before exit
    int dummy = 0;
    for (int i = 0; i < 4; ++i)
      if (s_fills[i] > 0)
        pipe_wait_slow(ptx::smem_u32(i < 2 ? &bars.s0_full[i] : &bars.kqv_full[i - 2]),
                       (uint32_t)((s_fills[i] - 1) & 1), &dummy);
  }
  if (w == 2) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kPipeTmemCols);
  }
}

// ------------------------------------------------------------------ state commit
//
// S_out^T[j][i] = g_l S_0^T[j][i] + sum_p gam_p u_p[j] k_p[i] over the accepted
// path (gam_p: product of alpha over the path nodes after p; g_l: over the
// whole path).  An item is (sequence, value head, 32 rows of S^T): a 16 KB
// tile at d_k = 128, contiguous in the [B, Hv, d_v, d_k] state.
//
// Persistent: the (sequence, value head) groups of d_v / 32 tiles each are
// dealt to the CTAs in turn (group g to CTA g mod P), so that at any moment
// the CTAs read one contiguous stretch of the state (CTAs reading far-apart
// ranges of their own ran at a third of the rate), and a group's tiles share
// its path data.
//   warp 0    state tiles by bulk copy into a ring of 16 KB stages (as many as
//             the shared memory left by the path buffers holds, <= 12), as far
//             ahead as the ring allows;
//   warps 1-3 each group's path data (warp w every third group, into buffer
//             w - 1, up to three groups ahead): path length, the alphas of the
//             path nodes, k rows (bf16, as stored) and u rows (fp32, all d_v
//             columns), by one round of asynchronous copies (the path itself
//             is read when the sequence changes); under full memory load such a
//             round takes microseconds, so one warp alone held the pipeline back;
//   warps 4-11 two halves of four warps, taking alternate tiles: read the
//             tile, free its stage, then the new rows (thread: up to eight
//             16-byte pieces of the tile), stored straight to global memory.
// Every wait is bounded (2 s); a wait that runs out makes every role stop,
// copies in flight get a bounded chance to land, and the rows of the tiles not
// reached are left unwritten.
constexpr int kCpStagesMax = 12;  // the ring takes what shared memory the path buffers leave
constexpr int kCpConsumers = 256;
constexpr int kCpSetupBufs = 3;  // path-data buffers, one per path-data warp
constexpr int kCpThreads = 32 * (1 + kCpSetupBufs) + kCpConsumers;
constexpr uint32_t kCpTileMax = kGcDC * 128 * 4;  // d_k <= 128

struct CpBars {
  unsigned long long full[kCpStagesMax], empty[kCpStagesMax], setup_full[kCpSetupBufs],
      setup_empty[kCpSetupBufs];
};

// bytes of one path-data buffer for N nodes: header (L), alphas [N],
// k rows [N][d_k] bf16, u rows [N][d_v] fp32, each part 16-byte aligned
__host__ __device__ inline uint32_t cp_setup_bytes(int N, int dk, int dv) {
  const uint32_t gam = ((uint32_t)N * 4 + 15) / 16 * 16;
  return 16 + gam + (uint32_t)N * dk * 2 + (uint32_t)N * dv * 4;
}

// bounded wait by every lane of a warp; false when it ran out or another role
// gave up
__device__ __forceinline__ bool cp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  return warp_wait(bar, parity, abort_flag);
}

__global__ void __launch_bounds__(kCpThreads, 1)
gdn_commit_pipe_kernel(const __grid_constant__ CUtensorMap tm_st, const __nv_bfloat16 *__restrict__ k,
                       const float *__restrict__ u, const float *__restrict__ alpha,
                       const int32_t *__restrict__ acc_nodes, const int32_t *__restrict__ n_acc,
                       const int32_t *__restrict__ status, int B, int N, int Hk, int Hv, int dk,
                       int dv, float *__restrict__ state_out, int stages) {
  // the tiles are tensor-copy destinations (and sources): 128-byte aligned,
  // whatever the static shared memory before the dynamic buffer
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = smem_raw + (((ptx::smem_u32(smem_raw) + 127u) & ~127u) - ptx::smem_u32(smem_raw));
  __shared__ CpBars bars;
  __shared__ int s_abort;
  __shared__ long long s_issued;  // state tiles the copy warp sent
  __shared__ int s_path[kCpSetupBufs][kGdnMaxN];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nC = dv / kGcDC;                      // items (tiles) per group
  const long long groups = (long long)B * Hv;     // (sequence, value head)
  const uint32_t tile = (uint32_t)kGcDC * dk * 4;
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t setup_off = stages * kCpTileMax;
  const uint32_t setup_bytes = cp_setup_bytes(N, dk, dv);
  const uint32_t gam_bytes = ((uint32_t)N * 4 + 15) / 16 * 16;
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.empty[i]), kCpConsumers / 2);  // one consumer half per tile
    }
    for (int i = 0; i < kCpSetupBufs; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.setup_full[i]), 32);
      ptx::mbar_init(ptx::smem_u32(&bars.setup_empty[i]), kCpConsumers);
    }
    s_abort = 0;
    s_issued = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  volatile int *abort_flag = &s_abort;

  if (warp == 0) {
    // ---------------------------------------------------------- state tiles
    long long n = 0;
    bool ok = true;
    for (long long gr = blockIdx.x; ok && gr < groups; gr += gridDim.x) {
      for (int c = 0; c < nC; ++c, ++n) {
        const int st = (int)(n % stages);
        if (n >= stages &&
            !(ok = cp_wait(ptx::smem_u32(&bars.empty[st]), (uint32_t)(((n / stages) - 1) & 1), abort_flag)))
          break;
        if (lane == 0) {
          // one tensor copy of the tile's 32 rows (256-byte L2 promotion: a
          // plain bulk copy of the same bytes ran at a third of the rate)
          const uint32_t fb = ptx::smem_u32(&bars.full[st]);
          ptx::mbar_arrive_expect_tx(fb, tile);
          if (n == 0) ptx::prefetch_tensormap(&tm_st);
          ptx::tma_load_2d(sbase + (uint32_t)st * kCpTileMax, &tm_st, fb, 0, (int)((gr * nC + c) * kGcDC));
        }
        __syncwarp();
      }
    }
    if (lane == 0) s_issued = n;
  } else if (warp <= kCpSetupBufs) {
    // ---------------------------------------------------------- path data
    // warp w takes the CTA's groups g = w - 1, w - 1 + kCpSetupBufs, ... into
    // buffer w - 1 (the gathers are latency-bound: several warps keep several
    // groups' copies in flight).  The path (length, nodes) is read when the
    // sequence changes; per group one round of asynchronous copies brings the
    // alphas, k rows and u rows.
    const int sb = warp - 1;
    int cur_b = -1, L = 0;
    int *path = s_path[sb];
    for (int g = sb; blockIdx.x + (long long)g * gridDim.x < groups; g += kCpSetupBufs) {
      const long long gr = blockIdx.x + (long long)g * gridDim.x;
      if (g >= kCpSetupBufs &&
          !cp_wait(ptx::smem_u32(&bars.setup_empty[sb]), (uint32_t)((g / kCpSetupBufs - 1) & 1), abort_flag))
        break;
      const int b = (int)(gr / Hv), h = (int)(gr - (long long)b * Hv), hk = h / (Hv / Hk);
      if (b != cur_b) {
        cur_b = b;
        L = 0;
        if (lane == 0) {
          L = (status && status[b] != 0) ? 0 : n_acc[b];
          if (L < 0 || L > N) L = 0;
        }
        const int t0 = lane < N ? acc_nodes[(size_t)b * N + lane] : 0;
        const int t1 = lane + 32 < N ? acc_nodes[(size_t)b * N + lane + 32] : 0;
        L = __shfl_sync(0xffffffffu, L, 0);
        const bool bad = (lane < L && (t0 < 0 || t0 >= N)) || (lane + 32 < L && (t1 < 0 || t1 >= N));
        if (__any_sync(0xffffffffu, bad)) L = 0;
        if (lane < L) path[lane] = t0;
        if (lane + 32 < L) path[lane + 32] = t1;
        __syncwarp();
      }
      unsigned char *buf = smem + setup_off + (uint32_t)sb * setup_bytes;
      // alphas of the path nodes (raw: the consumers form the products), k rows, u rows
      for (int pp = lane; pp < L; pp += 32) {
        const int t = path[pp];
        if (TV_CHECK(t >= 0 && t < N))
          cp_async_zfill(ptx::smem_u32(buf + 16 + pp * 4), alpha + ((size_t)b * N + t) * Hv + h, 4, true);
      }
      const int kc = dk / 8, uc = dv / 4;  // 16-byte pieces per k row, per u row
      for (int e = lane; e < L * kc; e += 32) {
        const int pp = e / kc, q = e - pp * kc;
        const int t = path[pp];
        if (TV_CHECK(t >= 0 && t < N))
          cp_async16(buf + 16 + gam_bytes + (size_t)pp * dk * 2 + q * 16,
                     k + (((size_t)b * N + t) * Hk + hk) * dk + q * 8);
      }
      for (int e = lane; e < L * uc; e += 32) {
        const int pp = e / uc, q = e - pp * uc;
        const int t = path[pp];
        if (TV_CHECK(t >= 0 && t < N))
          cp_async16(buf + 16 + gam_bytes + (size_t)N * dk * 2 + (size_t)pp * dv * 4 + q * 16,
                     u + (((size_t)b * N + t) * Hv + h) * dv + q * 4);
      }
      if (lane == 0) reinterpret_cast<int *>(buf)[0] = L;
      cp_async_wait_all();
      __syncwarp();
      ptx::mbar_arrive(ptx::smem_u32(&bars.setup_full[sb]));
    }
  } else {
    // ---------------------------------------------------------- new rows
    // S_out = g_l S_0 + sum_p gam_p u_p[j] k_p, with gam_p (the product of
    // alpha over the path nodes after p) formed from the end of the path, and
    // g_l the product over all of it
    // two halves of the consumers take alternate tiles, so two tiles are in
    // work at once
    const int cid = tid - 32 * (1 + kCpSetupBufs);
    const int half = cid / (kCpConsumers / 2), ct = cid - half * (kCpConsumers / 2);
    constexpr int kHalf = kCpConsumers / 2;
    long long n = 0;
    int g = 0;
    bool ok = true;
    constexpr int kIter = kGcDC * 128 / (kHalf * 4);  // 16-byte pieces per thread (<= 8)
    // the pieces of a thread lie kHalf * 4 elements apart: in the same columns
    // when d_k divides that
    const bool same_col = (kHalf * 4) % dk == 0;
    for (long long gr = blockIdx.x; ok && gr < groups; gr += gridDim.x, ++g) {
      if (g > 0) ptx::mbar_arrive(ptx::smem_u32(&bars.setup_empty[(g - 1) % kCpSetupBufs]));
      const int sb = g % kCpSetupBufs;
      if (!(ok = cp_wait(ptx::smem_u32(&bars.setup_full[sb]), (uint32_t)((g / kCpSetupBufs) & 1), abort_flag)))
        break;
      const unsigned char *buf = smem + setup_off + (uint32_t)sb * setup_bytes;
      const int L = reinterpret_cast<const int *>(buf)[0];
      const float *al = reinterpret_cast<const float *>(buf + 16);
      const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(buf + 16 + gam_bytes);
      const float *us = reinterpret_cast<const float *>(buf + 16 + gam_bytes + (size_t)N * dk * 2);
      for (int c = 0; c < nC; ++c, ++n) {
        if ((int)(n & 1) != half) continue;
        const int st = (int)(n % stages);
        if (!(ok = cp_wait(ptx::smem_u32(&bars.full[st]), (uint32_t)((n / stages) & 1), abort_flag))) break;
        const float *tl = reinterpret_cast<const float *>(smem + (uint32_t)st * kCpTileMax);
        float4 sv[kIter];
#pragma unroll
        for (int i2 = 0; i2 < kIter; ++i2) {
          const int e = (ct + i2 * kHalf) * 4;
          if (e < kGcDC * dk) sv[i2] = *reinterpret_cast<const float4 *>(tl + e);
        }
        ptx::mbar_arrive(ptx::smem_u32(&bars.empty[st]));  // the stage may be refilled
        float *dst = state_out + (size_t)(gr * nC + c) * kGcDC * dk;
        // the path loop outside, the thread's pieces inside: their chains
        // interleave, and a piece's column of k is one load per node (the
        // pieces of a thread lie in rows kHalf * 4 / d_k apart, in the same
        // columns when d_k divides kHalf * 4)
        float4 acc[kIter];
        int jj[kIter], ii[kIter];
#pragma unroll
        for (int i2 = 0; i2 < kIter; ++i2) {
          const int e = (ct + i2 * kHalf) * 4;
          jj[i2] = e / dk;
          ii[i2] = e - jj[i2] * dk;
          acc[i2] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float cur = 1.f;
        if (same_col) {
          // every piece of the thread reads the same four k values per node
          for (int pp = L - 1; pp >= 0; --pp) {
            const float *ur = us + (size_t)pp * dv + c * kGcDC;
            const uint2 kw = *reinterpret_cast<const uint2 *>(ks + (size_t)pp * dk + ii[0]);
            const float k0 = bf16_lo(kw.x), k1 = bf16_hi(kw.x), k2 = bf16_lo(kw.y), k3 = bf16_hi(kw.y);
#pragma unroll
            for (int i2 = 0; i2 < kIter; ++i2) {
              const float up = cur * ur[jj[i2] < kGcDC ? jj[i2] : 0];
              acc[i2].x = fmaf(up, k0, acc[i2].x);
              acc[i2].y = fmaf(up, k1, acc[i2].y);
              acc[i2].z = fmaf(up, k2, acc[i2].z);
              acc[i2].w = fmaf(up, k3, acc[i2].w);
            }
            cur *= al[pp];
          }
        } else {
          for (int pp = L - 1; pp >= 0; --pp) {
            const float *ur = us + (size_t)pp * dv + c * kGcDC;
            const __nv_bfloat16 *kr = ks + (size_t)pp * dk;
#pragma unroll
            for (int i2 = 0; i2 < kIter; ++i2) {
              const float up = cur * ur[jj[i2] < kGcDC ? jj[i2] : 0];
              const uint2 kw = *reinterpret_cast<const uint2 *>(kr + ii[i2]);
              acc[i2].x = fmaf(up, bf16_lo(kw.x), acc[i2].x);
              acc[i2].y = fmaf(up, bf16_hi(kw.x), acc[i2].y);
              acc[i2].z = fmaf(up, bf16_lo(kw.y), acc[i2].z);
              acc[i2].w = fmaf(up, bf16_hi(kw.y), acc[i2].w);
            }
            cur *= al[pp];
          }
        }
#pragma unroll
        for (int i2 = 0; i2 < kIter; ++i2) {
          const int e = (ct + i2 * kHalf) * 4;
          if (e >= kGcDC * dk) continue;
          __stcs(reinterpret_cast<float4 *>(dst + e),  // streamed: written once, not read back here
                 make_float4(fmaf(sv[i2].x, cur, acc[i2].x), fmaf(sv[i2].y, cur, acc[i2].y),
                             fmaf(sv[i2].z, cur, acc[i2].z), fmaf(sv[i2].w, cur, acc[i2].w)));
        }
      }
    }
  }
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // a role gave up: state copies still in flight get a bounded chance to
    // land before the CTA leaves
    int dummy = 0;
    const long long n = s_issued;
    for (long long m = n > stages ? n - stages : 0; m < n; ++m)
      pipe_wait_slow(ptx::smem_u32(&bars.full[m % stages]), (uint32_t)((m / stages) & 1), &dummy);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 gdn_encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// a 2-D map over rows of `inner` elements, `row_bytes` apart; box0 x box1
bool gdn_map(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t inner,
             uint64_t rows, uint64_t row_bytes, uint32_t box0, uint32_t box1,
             CUtensorMapSwizzle swizzle) {
  auto fn = gdn_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, type, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the pipelined kernel's shapes: trees of at most 32 nodes, d_k 64 or 128,
// coordinates within the 32-bit range of the tensor copies
bool gdn_pipe_ok(int B, int N, int Hv, int dk, int dv) {
  return N <= kPipeN && (dk == 64 || dk == 128) && (dv == 64 || dv == 128) &&
         (uint64_t)B * Hv * dv < (1ull << 31) && (uint64_t)B * N + kPipeN < (1ull << 31);
}

tv_status launch_gdn_pipe(const float *state, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                          const __nv_bfloat16 *v, const float *alpha, const float *beta,
                          const uint64_t *anc, int B, int N, int Hk, int Hv, int dk, int dv,
                          float *out, float *u, float *g, int32_t *status, cudaStream_t stream) {
  CUtensorMap ms, mk, mq, mv;
  const uint64_t rows_s = (uint64_t)B * Hv * dv, rows_n = (uint64_t)B * N;
  if (!gdn_map(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, state, dk, rows_s, (uint64_t)dk * 4, 32,
               (uint32_t)dv, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !gdn_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k, (uint64_t)Hk * dk, rows_n,
               (uint64_t)Hk * dk * 2, 64, kPipeN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !gdn_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, (uint64_t)Hk * dk, rows_n,
               (uint64_t)Hk * dk * 2, 64, kPipeN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !gdn_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v, (uint64_t)Hv * dv, rows_n,
               (uint64_t)Hv * dv * 2, (uint32_t)dv, kPipeN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return TV_ERR_CUDA;
  if (cudaFuncSetAttribute(gdn_tree_verify_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPipeSmem) != cudaSuccess)
    return TV_ERR_CUDA;
  const int items = B * Hv;
  const int grid = items < sm_count() ? items : sm_count();
  gdn_tree_verify_pipe_kernel<<<grid, kPipeThreads, kPipeSmem, stream>>>(
      ms, mk, mq, mv, alpha, beta, anc, B, N, Hk, Hv, dk, dv, out, u, g, status,
      debug_withheld_cta());
  return launch_status();
}

bool gdn_shape_ok(int B, int N, int Hk, int Hv, int dk, int dv) {
  return B >= 0 && N >= 1 && N <= kGdnMaxN && Hk >= 1 && Hv >= 1 && Hv % Hk == 0 && dk >= 32 &&
         dk <= 128 && dk % 32 == 0 && dv >= 64 && dv <= 128 && dv % 64 == 0;
}

}  // namespace
}  // namespace tv

using namespace tv;

extern "C" tv_status tv_gdn_tree_verify(const float *state, const void *q, const void *k,
                                        const void *v, const float *alpha, const float *beta,
                                        const uint64_t *anc, int B, int N, int Hk, int Hv, int dk,
                                        int dv, float *out, float *u, float *g, int kernel,
                                        int32_t *status, tv_stream stream) {
  if (!gdn_shape_ok(B, N, Hk, Hv, dk, dv)) return TV_ERR_ARG;
  if (kernel < 0 || kernel > 3) return TV_ERR_ARG;
  const bool tc_ok = dk == 64 || dk == 128;
  const bool pipe_ok = gdn_pipe_ok(B, N, Hv, dk, dv);
  if ((kernel == 2 && !tc_ok) || (kernel == 3 && !pipe_ok)) return TV_ERR_UNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!state || !q || !k || !v || !alpha || !beta || !anc || !out || !u || !g) return TV_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(q) |
       reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(u)) & 15)
    return TV_ERR_ARG;
  const dim3 grid(dv / kGdnDC, Hv, B);
  const auto *qb = static_cast<const __nv_bfloat16 *>(q);
  const auto *kb = static_cast<const __nv_bfloat16 *>(k);
  const auto *vb = static_cast<const __nv_bfloat16 *>(v);
  if (pipe_ok && (kernel == 3 || kernel == 0)) {
    const tv_status st = launch_gdn_pipe(state, qb, kb, vb, alpha, beta, anc, B, N, Hk, Hv, dk, dv,
                                         out, u, g, status, as_stream(stream));
    if (st == TV_OK || kernel == 3) return st;
  }
  if (tc_ok && kernel != 1) {
    const GdnTcLayout Ly = gdn_tc_layout(N, dk);
    if (cudaFuncSetAttribute(gdn_tree_verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Ly.bytes) != cudaSuccess)
      return TV_ERR_CUDA;
    gdn_tree_verify_tc_kernel<<<grid, kGdnThreads, Ly.bytes, as_stream(stream)>>>(
        state, qb, kb, vb, alpha, beta, anc, N, Hk, Hv, dk, dv, out, u, g, status);
    return launch_status();
  }
  const GdnLayout Ly = gdn_layout(N, dk);
  auto kern = N <= 32 ? gdn_tree_verify_kernel<4> : gdn_tree_verify_kernel<8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly.bytes) !=
      cudaSuccess)
    return TV_ERR_CUDA;
  kern<<<grid, kGdnThreads, Ly.bytes, as_stream(stream)>>>(state, qb, kb, vb, alpha, beta, anc, N,
                                                          Hk, Hv, dk, dv, out, u, g, status);
  return launch_status();
}

extern "C" tv_status tv_gdn_commit(const float *state_in, const void *k, const float *u,
                                   const float *alpha, const int32_t *acc_nodes,
                                   const int32_t *n_acc, int B, int N, int Hk, int Hv, int dk,
                                   int dv, float *state_out, const int32_t *status,
                                   tv_stream stream) {
  if (!gdn_shape_ok(B, N, Hk, Hv, dk, dv)) return TV_ERR_ARG;
  if (B == 0) return TV_OK;
  if (!state_in || !k || !u || !alpha || !acc_nodes || !n_acc || !state_out) return TV_ERR_ARG;
  if (state_in == state_out) return TV_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(state_in) | reinterpret_cast<uintptr_t>(state_out) |
       reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(u)) & 15)
    return TV_ERR_ARG;
  const size_t setup = kCpSetupBufs * (size_t)cp_setup_bytes(N, dk, dv);
  const int stages = (int)std::min<size_t>(kCpStagesMax, (220u * 1024u - setup) / kCpTileMax);
  const size_t smem = (size_t)stages * kCpTileMax + setup + 128;  // + alignment slack
  if (cudaFuncSetAttribute(gdn_commit_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return TV_ERR_CUDA;
  const long long groups = (long long)B * Hv;
  const int grid = groups < sm_count() ? (int)groups : sm_count();
  CUtensorMap mst;
  if (!gdn_map(&mst, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, state_in, (uint64_t)dk,
               (uint64_t)B * Hv * dv, (uint64_t)dk * 4, (uint32_t)dk, (uint32_t)kGcDC,
               CU_TENSOR_MAP_SWIZZLE_NONE))
    return TV_ERR_CUDA;
  gdn_commit_pipe_kernel<<<grid, kCpThreads, smem, as_stream(stream)>>>(
      mst, static_cast<const __nv_bfloat16 *>(k), u, alpha, acc_nodes, n_acc, status, B, N, Hk,
      Hv, dk, dv, state_out, stages);
  return launch_status();
}
