// Tree attention: the entry point, the split combine and the CUDA-core kernel.
//
// Source: "Tree spec-decode -> vLLM serve integration spec", "2. Verify: tree
// attention mask".  Node t of sequence b attends
//   (a) every context key j < ctx_len[b] of the paged cache, and
//   (b) the tree nodes a that are ancestors of t or t itself,
// both restricted to keys at positions >= pos[t] - window_left when a sliding
// window is set.  Scores are sm_scale * q.k, softmax in fp32, output bf16.
//
// Work decomposition (flash-decoding): one thread block per (sequence, KV head,
// context split).  The G query heads of the KV head and the N nodes are packed
// into R = G*N rows that all reuse each K/V tile staged in shared memory.  The
// node -> node block (N keys from k_tree / v_tree, ancestor-masked) is one more
// tile handled by split 0.  Splits write (m, l, O) partials that a combine
// kernel merges; with a single split the kernel writes the output directly.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attention.cuh"

TV_DEBUG_RECORD(attention)

namespace tv {

namespace {

constexpr int kCcThreads = 256;
// rows per thread block: 64, or 32 at D = 256 (the output accumulators of 8
// rows x 8 dims per lane would take every register and leave one CTA per SM)
template <int D>
constexpr int cc_rows() { return D >= 256 ? 32 : 64; }
constexpr int kCcRowsMax = 64;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int n = valid ? 16 : 0;  // n = 0: zero-fill the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }

// CUDA-core tree attention.
// Lane roles in the score phase: key kk = lane/2 of the 16-key tile and half
// hh = lane%2 of the head dimension (8-element groups interleaved by half), so
// a warp computes 16 dot products per row with one shuffle to join halves.
// In the P.V phase lane l owns output dims [l*D/32, (l+1)*D/32).
// Launched as a programmatic dependent of the kernel before it: context
// lengths and Q are read before griddepcontrol.wait; positions, ancestor
// masks, block tables and every write come after it.
template <int D>
__global__ void __launch_bounds__(kCcThreads, D >= 256 ? 2 : 1)
attn_generic_kernel(const AttnParams p) {
  constexpr int kCcRows = cc_rows<D>();
  constexpr int kCcRowsPerWarp = kCcRows / (kCcThreads / 32);
  constexpr int KP = D + 16;         // padded K row: consecutive keys 32 bytes apart mod 128
  constexpr int DL = D / 32;         // output dims per lane
  constexpr int NG = D / 16;         // 8-dim groups per lane in the score phase
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float *q_s = reinterpret_cast<float *>(smem_raw);                          // [kCcRows][D]
  __nv_bfloat16 *k_s = reinterpret_cast<__nv_bfloat16 *>(q_s + kCcRows * D);  // [2][16][KP]
  __nv_bfloat16 *v_s = k_s + 2 * 16 * KP;                                     // [2][16][D]
  __shared__ int s_rpos[kCcRows];
  __shared__ unsigned long long s_ranc[kCcRows];
  __shared__ int s_npos[kMaxNodes];
  __shared__ int s_tile_ok[2];

  const int bk = blockIdx.x;
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int split = blockIdx.y;
  const int r0 = blockIdx.z * kCcRows;
  const int nrows = min(kCcRows, p.R - r0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the combine grid launched after this one may be scheduled now: it waits
  // for this grid's completion before reading the partials
  pdl_launch_dependents();

  int ctx = p.ctx_len[b];
  const int ctx_cap = p.max_blocks * kBlock;
  if (ctx < 0 || ctx > ctx_cap) {
    if (tid == 0) {
      pdl_wait();
      set_status(p.status, b, TV_ERR_BLOCK);
    }
    ctx = ctx < 0 ? 0 : ctx_cap;
  }
  const int blk_lo = first_visible_block(ctx, p.window_left);
  const int blk_end = (ctx + kBlock - 1) / kBlock;
  const int t_begin = blk_lo + split * p.bps;
  const int t_stop = min(blk_end, t_begin + p.bps);
  const int n_ctx_tiles = max(0, t_stop - t_begin);
  const int n_node_tiles = split == 0 ? (p.N + 15) / 16 : 0;
  const int n_tiles = n_ctx_tiles + n_node_tiles;

  // rows: queries pre-scaled into the base-2 domain, positions and ancestor masks
  for (int i = tid; i < nrows * (D / 4); i += kCcThreads) {
    const int rr = i / (D / 4), c4 = i - rr * (D / 4);
    const int r = r0 + rr, t = r / p.G, g = r - t * p.G;
    if (!TV_CHECK(b < p.B && t < p.N && kvh * p.G + g < p.Hq)) continue;
    const __nv_bfloat16 *src = p.q + (((size_t)b * p.N + t) * p.Hq + kvh * p.G + g) * D + c4 * 4;
    const uint2 w = *reinterpret_cast<const uint2 *>(src);
    float4 f = make_float4(bf16_lo(w.x) * p.qscale, bf16_hi(w.x) * p.qscale,
                           bf16_lo(w.y) * p.qscale, bf16_hi(w.y) * p.qscale);
    *reinterpret_cast<float4 *>(q_s + rr * D + c4 * 4) = f;
  }
  // positions and ancestor masks come from the ancestor kernel before this
  // grid, and every write below (status, partials, output) may race with the
  // grid before: wait for its completion here
  pdl_wait();
  for (int rr = tid; rr < nrows; rr += kCcThreads) {
    const int t = (r0 + rr) / p.G;
    if (!TV_CHECK(t < p.N && rr < kCcRows)) continue;
    s_rpos[rr] = p.pos[(size_t)b * p.N + t];
    s_ranc[rr] = p.anc[(size_t)b * p.N + t];
  }
  for (int a = tid; a < p.N; a += kCcThreads) s_npos[a] = p.pos[(size_t)b * p.N + a];

  // stage tile i into buffer st; rows past the valid range are zero-filled so
  // that 0 * V never meets a non-finite value
  auto load_tile = [&](int i, int st) {
    __nv_bfloat16 *kd = k_s + st * 16 * KP;
    __nv_bfloat16 *vd = v_s + st * 16 * D;
    constexpr int W = D / 8;  // 16-byte words per row
    if (i < n_ctx_tiles) {
      const int slot = t_begin + i;
      const int blk = TV_CHECK(slot >= 0 && slot < p.max_blocks)
                          ? p.block_table[(size_t)b * p.max_blocks + slot] : -1;
      const bool blk_ok = blk >= 0 && blk < p.num_blocks;
      if (tid == 0) {
        s_tile_ok[st] = blk_ok;
        if (!blk_ok) set_status(p.status, b, TV_ERR_BLOCK);
      }
      const int valid_rows = blk_ok ? min(kBlock, ctx - slot * kBlock) : 0;
      const size_t base = ((size_t)(blk_ok ? blk : 0) * p.Hkv + kvh) * kBlock * D;
      for (int c = tid; c < 16 * W; c += kCcThreads) {
        const int row = c / W, wd = c - row * W;
        const bool v = row < valid_rows;
        cp_async16(kd + row * KP + wd * 8, p.k_cache + base + (size_t)row * D + wd * 8, v);
        cp_async16(vd + row * D + wd * 8, p.v_cache + base + (size_t)row * D + wd * 8, v);
      }
    } else {
      const int nt = i - n_ctx_tiles;
      if (tid == 0) s_tile_ok[st] = 1;
      for (int c = tid; c < 16 * W; c += kCcThreads) {
        const int row = c / W, wd = c - row * W;
        const int a = nt * 16 + row;
        const bool v = a < p.N;
        const size_t off = (((size_t)b * p.N + (v ? a : 0)) * p.Hkv + kvh) * D + wd * 8;
        cp_async16(kd + row * KP + wd * 8, p.k_tree + off, v);
        cp_async16(vd + row * D + wd * 8, p.v_tree + off, v);
      }
    }
    cp_async_commit();
  };

  float o[kCcRowsPerWarp][DL];
  float m[kCcRowsPerWarp], l[kCcRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kCcRowsPerWarp; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) o[j][e] = 0.f;
  }

  const int kk = lane >> 1, hh = lane & 1;
  if (n_tiles > 0) load_tile(0, 0);
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i & 1;
    cp_async_wait_all();
    __syncthreads();                       // tile i visible; tile i-1 fully consumed
    if (i + 1 < n_tiles) load_tile(i + 1, st ^ 1);
    const bool is_node = i >= n_ctx_tiles;
    const int key = is_node ? (i - n_ctx_tiles) * 16 + kk : (t_begin + i) * kBlock + kk;
    const bool key_ok = s_tile_ok[st] && (is_node ? key < p.N : key < ctx);
    const int key_pos = is_node ? (key_ok ? s_npos[key] : 0) : key;
    const __nv_bfloat16 *krow = k_s + st * 16 * KP + kk * KP;
    const __nv_bfloat16 *vt = v_s + st * 16 * D + lane * DL;
    // scores of this warp's rows against key kk, in chunks of at most 8
    // 16-byte K fragments so that no more than 8 are live at once
    constexpr int NGC = NG < 8 ? NG : 8;
    float sc[kCcRowsPerWarp][2];
#pragma unroll
    for (int j = 0; j < kCcRowsPerWarp; ++j) sc[j][0] = sc[j][1] = 0.f;
#pragma unroll
    for (int g0 = 0; g0 < NG; g0 += NGC) {
      uint4 kf[NGC];
#pragma unroll
      for (int gi = 0; gi < NGC; ++gi)
        kf[gi] = *reinterpret_cast<const uint4 *>(krow + (2 * (g0 + gi) + hh) * 8);
#pragma unroll
      for (int j = 0; j < kCcRowsPerWarp; ++j) {
        const int rr = warp + j * (kCcThreads / 32);
        if (rr >= nrows) break;                         // warp-uniform
        const float *qr = q_s + rr * D;
        float s0 = sc[j][0], s1 = sc[j][1];
#pragma unroll
        for (int gi = 0; gi < NGC; ++gi) {
          const float4 qa = *reinterpret_cast<const float4 *>(qr + (2 * (g0 + gi) + hh) * 8);
          const float4 qb = *reinterpret_cast<const float4 *>(qr + (2 * (g0 + gi) + hh) * 8 + 4);
          const uint4 kw = kf[gi];
          s0 = fmaf(qa.x, bf16_lo(kw.x), s0);
          s1 = fmaf(qa.y, bf16_hi(kw.x), s1);
          s0 = fmaf(qa.z, bf16_lo(kw.y), s0);
          s1 = fmaf(qa.w, bf16_hi(kw.y), s1);
          s0 = fmaf(qb.x, bf16_lo(kw.z), s0);
          s1 = fmaf(qb.y, bf16_hi(kw.z), s1);
          s0 = fmaf(qb.z, bf16_lo(kw.w), s0);
          s1 = fmaf(qb.w, bf16_hi(kw.w), s1);
        }
        sc[j][0] = s0;
        sc[j][1] = s1;
      }
    }
#pragma unroll
    for (int j = 0; j < kCcRowsPerWarp; ++j) {
      const int rr = warp + j * (kCcThreads / 32);
      if (rr >= nrows) break;                         // warp-uniform
      float s = sc[j][0] + sc[j][1];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      const int rpos = s_rpos[rr];
      bool ok = key_ok;
      if (is_node) ok = ok && ((s_ranc[rr] >> key) & 1ull);
      if (p.window_left >= 0) ok = ok && (key_pos >= rpos - p.window_left);
      s = ok ? s : -INFINITY;
      float tmax = s;
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float m_new = fmaxf(m[j], tmax);
      if (m_new == -INFINITY) continue;               // no visible key yet (warp-uniform)
      const float alpha = exp2f(m[j] - m_new);
      const float pk = ok ? exp2f(s - m_new) : 0.f;
      float psum = pk;
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l[j] = l[j] * alpha + psum;
      m[j] = m_new;
#pragma unroll
      for (int e = 0; e < DL; ++e) o[j][e] *= alpha;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float pkk = __shfl_sync(0xffffffffu, pk, 2 * k);
        const __nv_bfloat16 *vr = vt + k * D;
        if constexpr (DL == 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t *>(vr);
          o[j][0] = fmaf(pkk, bf16_lo(w), o[j][0]);
          o[j][1] = fmaf(pkk, bf16_hi(w), o[j][1]);
        } else if constexpr (DL == 4) {
          const uint2 w = *reinterpret_cast<const uint2 *>(vr);
          o[j][0] = fmaf(pkk, bf16_lo(w.x), o[j][0]);
          o[j][1] = fmaf(pkk, bf16_hi(w.x), o[j][1]);
          o[j][2] = fmaf(pkk, bf16_lo(w.y), o[j][2]);
          o[j][3] = fmaf(pkk, bf16_hi(w.y), o[j][3]);
        } else {
          const uint4 w = *reinterpret_cast<const uint4 *>(vr);
          o[j][0] = fmaf(pkk, bf16_lo(w.x), o[j][0]);
          o[j][1] = fmaf(pkk, bf16_hi(w.x), o[j][1]);
          o[j][2] = fmaf(pkk, bf16_lo(w.y), o[j][2]);
          o[j][3] = fmaf(pkk, bf16_hi(w.y), o[j][3]);
          o[j][4] = fmaf(pkk, bf16_lo(w.z), o[j][4]);
          o[j][5] = fmaf(pkk, bf16_hi(w.z), o[j][5]);
          o[j][6] = fmaf(pkk, bf16_lo(w.w), o[j][6]);
          o[j][7] = fmaf(pkk, bf16_hi(w.w), o[j][7]);
        }
      }
    }
  }

  // epilogue: direct bf16 output with one split, else fp32 partials
#pragma unroll
  for (int j = 0; j < kCcRowsPerWarp; ++j) {
    const int rr = warp + j * (kCcThreads / 32);
    if (rr >= nrows) break;
    const int r = r0 + rr;
    if (p.splits == 1) {
      const int t = r / p.G, g = r - t * p.G;
      if (!TV_CHECK(t < p.N && kvh * p.G + g < p.Hq)) continue;
      const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
      __nv_bfloat16 *dst = p.out + (((size_t)b * p.N + t) * p.Hq + kvh * p.G + g) * D + lane * DL;
#pragma unroll
      for (int e = 0; e < DL; e += 2)
        *reinterpret_cast<__nv_bfloat162 *>(dst + e) =
            __floats2bfloat162_rn(o[j][e] * inv, o[j][e + 1] * inv);
    } else {
      const size_t row = ((size_t)bk * p.splits + split) * p.R + r;
      if (!TV_CHECK(row < (size_t)p.B * p.Hkv * p.splits * p.R)) continue;
      float *dst = p.part_o + row * D + lane * DL;
#pragma unroll
      for (int e = 0; e < DL; ++e) dst[e] = o[j][e];
      if (lane == 0) p.part_ml[row] = make_float2(m[j], l[j]);
    }
  }
}

// One warp per output row: O = sum_s O_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
constexpr int kCombAtOnce = 16;  // splits whose partials are loaded in one round
__global__ void attn_combine_kernel(const AttnParams p) {
  // A grid launched after this one as a programmatic dependent reads, before
  // its own wait, nothing this grid writes.
  pdl_launch_dependents();
  // One warp per output row; lane l owns dims 8l .. 8l+7 (D <= 256).  With at
  // most kCombAtOnce splits every partial is loaded in one round.  Otherwise
  // the split maxima and weights are formed by the lanes in parallel (lane j
  // holds split c*32 + j of each chunk of 32) and the weighted sum walks the
  // splits four at a time so their loads overlap.  Both merge the splits in
  // increasing order, so they give the same bits.
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.Hkv * p.R;
  if (row >= rows) return;
  const int bk = (int)(row / p.R), r = (int)(row - (long long)bk * p.R);
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int D = p.D;
  const size_t pr0 = (size_t)bk * p.splits * p.R + r;  // partial row of split s: pr0 + s * R
  pdl_wait();  // the partials are the attention grid's output
  float L = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const bool mine = lane * 8 < D;
  if (p.splits <= kCombAtOnce) {
    // Up to kCombAtOnce splits: every split's (max, sum) and O slice are
    // loaded in one round, then merged in split order as below.  The O of a
    // split with weight 0 (no keys) is loaded but not used.
    const int n = p.splits;
    const float2 ml = lane < n ? p.part_ml[pr0 + (size_t)lane * p.R] : make_float2(-INFINITY, 0.f);
    float4 va[kCombAtOnce], vb[kCombAtOnce];
#pragma unroll
    for (int u = 0; u < kCombAtOnce; ++u) {
      if (u < n && mine) {
        const float *src = p.part_o + (pr0 + (size_t)u * p.R) * D + lane * 8;
        va[u] = *reinterpret_cast<const float4 *>(src);
        vb[u] = *reinterpret_cast<const float4 *>(src + 4);
      }
    }
    float M = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float wl = 0.f;
    if (ml.x != -INFINITY) {
      wl = exp2f(ml.x - M);
      L += ml.y * wl;
    }
#pragma unroll
    for (int u = 0; u < kCombAtOnce; ++u) {
      const float w = __shfl_sync(0xffffffffu, wl, u);
      if (u < n && w != 0.f && mine) {
        acc[0] += va[u].x * w; acc[1] += va[u].y * w;
        acc[2] += va[u].z * w; acc[3] += va[u].w * w;
        acc[4] += vb[u].x * w; acc[5] += vb[u].y * w;
        acc[6] += vb[u].z * w; acc[7] += vb[u].w * w;
      }
    }
  } else {
    float M = -INFINITY;
    for (int s = lane; s < p.splits; s += 32) M = fmaxf(M, p.part_ml[pr0 + (size_t)s * p.R].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    for (int c0 = 0; c0 < p.splits; c0 += 32) {
      // this chunk's weights, one split per lane
      const int sl = c0 + lane;
      float wl = 0.f;
      if (sl < p.splits) {
        const float2 ml = p.part_ml[pr0 + (size_t)sl * p.R];
        if (ml.x != -INFINITY) {
          wl = exp2f(ml.x - M);
          L += ml.y * wl;
        }
      }
      const int n = min(32, p.splits - c0);
      for (int j = 0; j < n; j += 4) {
        float4 va[4], vb[4];
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wl, (j + u) & 31);
          if (j + u < n && w[u] != 0.f && mine) {
            const float *src = p.part_o + (pr0 + (size_t)(c0 + j + u) * p.R) * D + lane * 8;
            va[u] = *reinterpret_cast<const float4 *>(src);
            vb[u] = *reinterpret_cast<const float4 *>(src + 4);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (j + u < n && w[u] != 0.f && mine) {
            acc[0] += va[u].x * w[u]; acc[1] += va[u].y * w[u];
            acc[2] += va[u].z * w[u]; acc[3] += va[u].w * w[u];
            acc[4] += vb[u].x * w[u]; acc[5] += vb[u].y * w[u];
            acc[6] += vb[u].z * w[u]; acc[7] += vb[u].w * w[u];
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  if (mine) {
    const int t = r / p.G, g = r - t * p.G;
    __nv_bfloat16 *o = p.out + (((size_t)b * p.N + t) * p.Hq + kvh * p.G + g) * D + lane * 8;
#pragma unroll
    for (int e = 0; e < 8; e += 2)
      *reinterpret_cast<__nv_bfloat162 *>(o + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

template <int D>
void launch_generic_d(const AttnParams &p, cudaStream_t stream) {
  constexpr int kCcRows = cc_rows<D>();
  const size_t smem = (size_t)kCcRows * D * sizeof(float) +
                      (size_t)2 * 16 * (D + 16) * sizeof(__nv_bfloat16) +
                      (size_t)2 * 16 * D * sizeof(__nv_bfloat16);
  cudaFuncSetAttribute(attn_generic_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  dim3 grid(p.B * p.Hkv, p.splits, (p.R + kCcRows - 1) / kCcRows);
  launch_pdl(attn_generic_kernel<D>, grid, dim3(kCcThreads), smem, stream, p);
}

struct SplitPlan {
  int splits, bps;
};

SplitPlan plan_splits(const tv_attn_args *a, int R, bool tc) {
  const int vis = visible_blocks_bound(a->max_blocks, a->window_left);
  int splits;
  if (a->num_splits > 0) {
    splits = a->num_splits;
  } else {
    const int rows_cta = a->D >= 256 ? cc_rows<256>() : cc_rows<128>();
    const long long base = (long long)a->B * a->Hkv * (tc ? 1 : (R + rows_cta - 1) / rows_cta);
    const long long target = 2LL * sm_count();
    splits = base > 0 ? (int)((target + base - 1) / base) : 1;
  }
  if (splits > vis) splits = vis;
  if (splits < 1) splits = 1;
  int bps = vis > 0 ? (vis + splits - 1) / splits : 1;
  splits = vis > 0 ? (vis + bps - 1) / bps : 1;
  return SplitPlan{splits, bps};
}

bool shape_ok(const tv_attn_args *a) {
  return a->B >= 0 && a->N >= 0 && a->N <= kMaxNodes && a->Hq > 0 && a->Hkv > 0 &&
         a->max_blocks >= 0 && a->num_blocks >= 0 && a->window_left >= -1 &&
         a->window_right >= -1;
}

}  // namespace

void launch_combine(const AttnParams &p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.Hkv * p.R;
  // 4 warps (128 threads) per block: a block holds the partials of up to 16
  // splits in registers (about 21K), which leaves room on its SM for a CTA of
  // the attention launched after it, as a programmatic dependent, to start
  const int wpb = 4;
  launch_pdl(attn_combine_kernel, dim3((unsigned)((rows + wpb - 1) / wpb)), dim3(wpb * 32), 0, stream, p);
}

void launch_attention_generic(const AttnParams &p, cudaStream_t stream) {
  switch (p.D) {
    case 64: launch_generic_d<64>(p, stream); break;
    case 128: launch_generic_d<128>(p, stream); break;
    default: launch_generic_d<256>(p, stream); break;
  }
}

}  // namespace tv

using namespace tv;

namespace {

// Which kernel serves these arguments: true = tcgen05, false = CUDA cores.
// kernel 2 (tensor cores) on a shape the tcgen05 kernel does not cover is
// reported by the caller as TV_ERR_UNSUPPORTED.
bool tc_shape(const tv_attn_args *a) {
  AttnParams probe{};
  probe.B = a->B;
  probe.D = a->D;
  probe.G = a->Hkv > 0 ? a->Hq / a->Hkv : 0;
  probe.N = a->N;
  probe.R = probe.G * a->N;
  return attention_tc_supported(probe);
}

bool use_tc(const tv_attn_args *a) {
  if (a->kernel == 1) return false;
  return tc_shape(a);
}

// The D = 256 tensor-core kernel (split-K, generic partials and combine).
bool tc256_shape(const tv_attn_args *a) {
  AttnParams probe{};
  probe.D = a->D;
  probe.G = a->Hkv > 0 ? a->Hq / a->Hkv : 0;
  probe.N = a->N;
  probe.R = probe.G * a->N;
  return attention_tc256_supported(probe);
}

bool use_tc256(const tv_attn_args *a) { return a->kernel != 1 && tc256_shape(a); }

// Splits for the D = 256 tensor-core kernel: about one CTA per SM, each split
// a whole number of 64-key tiles (four blocks).
SplitPlan plan_splits_tc256(const tv_attn_args *a) {
  const int vis = visible_blocks_bound(a->max_blocks, a->window_left);
  const long long base = (long long)a->B * a->Hkv;
  int splits = a->num_splits > 0 ? a->num_splits
                                 : (base > 0 ? (int)((sm_count() + base - 1) / base) : 1);
  if (splits < 1) splits = 1;
  int bps = vis > 0 ? (vis + splits - 1) / splits : 4;
  bps = (bps + 3) / 4 * 4;
  splits = vis > 0 ? (vis + bps - 1) / bps : 1;
  return SplitPlan{splits, bps};
}

size_t workspace_bytes_for(const tv_attn_args *a, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = (size_t)a->B * a->Hkv * splits * (size_t)(a->Hq / a->Hkv) * a->N;
  const size_t o_bytes = ((rows * a->D * sizeof(float) + 255) / 256) * 256;
  return o_bytes + rows * sizeof(float2);
}

}  // namespace

extern "C" size_t tv_tree_attention_workspace_size(const tv_attn_args *a) {
  if (!a || !shape_ok(a) || a->Hq % a->Hkv != 0) return 0;
  if (use_tc(a)) return attention_tc_workspace(a->B, sm_count());
  if (use_tc256(a)) return workspace_bytes_for(a, plan_splits_tc256(a).splits);
  const int R = (a->Hq / a->Hkv) * a->N;
  const SplitPlan sp = plan_splits(a, R, false);
  return workspace_bytes_for(a, sp.splits);
}

extern "C" tv_status tv_tree_attention(const tv_attn_args *a, void *workspace,
                                       size_t workspace_bytes, tv_stream stream) {
  if (!a || !shape_ok(a)) return TV_ERR_ARG;
  if (a->block_size != kBlock) return TV_ERR_UNSUPPORTED;
  if (a->D != 64 && a->D != 128 && a->D != 256) return TV_ERR_UNSUPPORTED;
  if (a->Hq % a->Hkv != 0) return TV_ERR_ARG;
  if (a->kernel < 0 || a->kernel > 2) return TV_ERR_ARG;
  if (a->kernel == 2 && !tc_shape(a) && !tc256_shape(a)) return TV_ERR_UNSUPPORTED;
  const int G = a->Hq / a->Hkv;
  const int R = G * a->N;
  if (R > 256) return TV_ERR_UNSUPPORTED;
  if (a->B == 0 || a->N == 0) return TV_OK;
  if (!a->q || !a->k_tree || !a->v_tree || !a->k_cache || !a->v_cache || !a->ctx_len ||
      !a->pos || !a->anc || !a->out || !a->status)
    return TV_ERR_ARG;
  if (a->max_blocks > 0 && !a->block_table) return TV_ERR_ARG;
  const uintptr_t align = reinterpret_cast<uintptr_t>(a->q) | reinterpret_cast<uintptr_t>(a->k_tree) |
                          reinterpret_cast<uintptr_t>(a->v_tree) |
                          reinterpret_cast<uintptr_t>(a->k_cache) |
                          reinterpret_cast<uintptr_t>(a->v_cache) | reinterpret_cast<uintptr_t>(a->out);
  if (align & 15) return TV_ERR_ARG;
  const bool tc = use_tc(a);
  const bool tc256 = !tc && use_tc256(a);
  const SplitPlan sp = tc256 ? plan_splits_tc256(a) : plan_splits(a, R, tc);
  const size_t need = tc ? attention_tc_workspace(a->B, sm_count()) : workspace_bytes_for(a, sp.splits);
  if (need > workspace_bytes || (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255))))
    return TV_ERR_ARG;

  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16 *>(a->q);
  p.k_tree = static_cast<const __nv_bfloat16 *>(a->k_tree);
  p.v_tree = static_cast<const __nv_bfloat16 *>(a->v_tree);
  p.k_cache = static_cast<const __nv_bfloat16 *>(a->k_cache);
  p.v_cache = static_cast<const __nv_bfloat16 *>(a->v_cache);
  p.block_table = a->block_table;
  p.ctx_len = a->ctx_len;
  p.pos = a->pos;
  p.anc = a->anc;
  p.B = a->B;
  p.N = a->N;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.G = G;
  p.R = R;
  p.D = a->D;
  p.max_blocks = a->max_blocks;
  p.num_blocks = a->num_blocks;
  p.window_left = a->window_left;
  const float scale = a->sm_scale > 0.f ? a->sm_scale : 1.0f / sqrtf((float)a->D);
  p.qscale = scale * 1.4426950408889634f;
  p.splits = sp.splits;
  p.bps = sp.bps;
  if (!tc && sp.splits > 1) {
    const size_t rows = (size_t)a->B * a->Hkv * sp.splits * R;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                           ((rows * a->D * sizeof(float) + 255) / 256) * 256);
  }
  p.out = static_cast<__nv_bfloat16 *>(a->out);
  p.status = a->status;
  if (a->max_ctas < 0) return TV_ERR_ARG;
  p.ctas = a->max_ctas;
  p.withheld_cta = debug_withheld_cta();
  cudaStream_t s = as_stream(stream);
  if (tc) {
    if (launch_attention_tc(p, workspace, s) != cudaSuccess) return TV_ERR_CUDA;
    return TV_OK;
  }
  if (tc256) {
    if (launch_attention_tc256(p, s) != cudaSuccess) return TV_ERR_CUDA;
    if (sp.splits > 1) launch_combine(p, s);
    return launch_status();
  }
  launch_attention_generic(p, s);
  if (sp.splits > 1) launch_combine(p, s);
  return launch_status();
}
