// Tree attention on the tensor cores for head dimension 256 (tcgen05 / TMEM /
// TMA, sm_100a and later), split-K flash decoding.
//
// Source: "Technische Samenvatting: Trees from Marginals (DFlash-TfM)",
// "2. Tree Attention": every row (node t, query head h) attends to the
// visible context of its sequence and to its ancestors-or-self among the tree
// nodes, with the sliding window applied to both.  The G query heads of one KV
// head and the N nodes are packed into R = G*N <= 128 rows (row r = t*G + g),
// so one pass over a tile of keys serves every row.
//
// One CTA per (sequence, KV head, context split); split 0 also takes the node
// tile.  A CTA walks its 64-key tiles (four paged blocks) through a 3-stage
// TMA ring:
//   warp 0      TMA of K ([4 d-quarters][64 keys][64], 128-byte swizzled,
//               K-major) and V ([4 blocks][4 d-quarters][16 keys][64], the
//               MN-major B operand of P V); rows outside the context, the split
//               or a bad block are zero-filled and masked;
//   warp 1      the only MMA issuer: S = Q K^T (M128, N = keys, 16 K=16 steps,
//               A = Q in TMEM) and O += P V (M128 N256, A = P in TMEM, one
//               K=16 step per 16-key block);
//   warps 2-5   softmax warpgroup: thread = row = TMEM lane; S from TMEM,
//               masks, online max with lazy rescaling of O (only when a row's
//               max grows by more than 2^8), P (bf16) into TMEM, and at the end
//               O into the bf16 output (one split) or the fp32 partials that
//               the split combine merges.
// TMEM: S [0, 64), P [64, 96), Q [128, 256) (256 dims as bf16 pairs), O
// [256, 512).  Scores live in the base-2 domain (q scaled by
// log2(e)/sqrt(D)), as in the other attention kernels.  Every wait is bounded
// (2 s); on expiry status[b] = TV_ERR_CUDA and the CTA winds down.
// Programmatic dependent launch: the grid may start while the kernel before
// it on the stream finishes.  Before griddepcontrol.wait it reads only inputs
// that no earlier kernel of a verify step writes (context lengths, block
// tables, Q, K/V); positions and ancestor masks are read, and status words,
// partials and the output written, only after it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "attention.cuh"
#include "tc_ptx.cuh"

TV_DEBUG_RECORD(attention_tc256)

namespace tv {
namespace {

using namespace ptx;

constexpr int kD = 256;
constexpr int kM = 128;                // UMMA M: rows per tile
constexpr int kBN = 64;                // keys per context tile (4 paged blocks)
constexpr int kStages = 3;
constexpr int kThreads = 192;          // producer, MMA, softmax warpgroup (warps 2-5)
constexpr uint32_t kQuarter = kBN * 128;               // [64 keys][64 d] bf16 = 8 KB
constexpr uint32_t kKBytes = 4 * kQuarter;             // K tile: 32 KB
constexpr uint32_t kBlkQuarter = kBlock * 128;         // [16 keys][64 d] = 2 KB
constexpr uint32_t kBlkBytes = 4 * kBlkQuarter;        // V block: [4][16][64] = 8 KB
constexpr uint32_t kStageBytes = kKBytes + 4 * kBlkBytes;  // 64 KB
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 64, kColQ = 128, kColO = 256;
constexpr float kTau = 8.0f;
constexpr unsigned long long kWaitNs = 2000000000ull;

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Bars {
  unsigned long long kv_full[kStages], kv_empty[kStages];
  unsigned long long q_full, s_full, s_free, p_full, pv_done, fin;
};

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kWaitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// every lane waits; true when the phase completed for all of them
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  const bool ok = mbar_try_wait(bar, parity) || wait_slow(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The tiles of one CTA: context tiles of four blocks from block t_begin (the
// split's range [t_begin, t_stop), within [blk_lo, blk_end)), then the node
// tile when this is split 0.
struct Range {
  int t_begin, t_stop, n_ctx, n_tiles, np;
};
__device__ __forceinline__ Range range_of(const AttnParams &p, int ctx, int split) {
  Range r;
  const int blk_lo = first_visible_block(ctx, p.window_left);
  const int blk_end = (ctx + kBlock - 1) / kBlock;
  r.t_begin = blk_lo + split * p.bps;
  r.t_stop = min(blk_end, r.t_begin + p.bps);
  r.n_ctx = r.t_stop > r.t_begin ? (r.t_stop - r.t_begin + 3) / 4 : 0;
  r.np = (p.N + 15) / 16 * 16;
  r.n_tiles = r.n_ctx + (split == 0 ? 1 : 0);
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc256_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_krow,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vrow,
                  const __grid_constant__ CUtensorMap tm_tk, const __grid_constant__ CUtensorMap tm_tv,
                  const AttnParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bk = blockIdx.x, split = blockIdx.y;
  const int b = bk / p.Hkv, kvh = bk - b * p.Hkv;
  const int N = p.N, G = p.G, R = p.R;

  int ctx = p.ctx_len[b];
  const int cap = p.max_blocks * kBlock;
  if (ctx < 0 || ctx > cap) {
    if (tid == 0 && split == 0) {
      pdl_wait();
      set_status(p.status, b, TV_ERR_BLOCK);
    }
    ctx = ctx < 0 ? 0 : cap;
  }
  const Range rg = range_of(p, ctx, split);

  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // test hook: one arrival more than the producer makes, in one CTA
      const bool held = s == 0 && (int)(blockIdx.y * gridDim.x + blockIdx.x) == p.withheld_cta;
      mbar_init(smem_u32(&bars.kv_full[s]), held ? 2 : 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.q_full), 128);
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.s_free), 128);
    mbar_init(smem_u32(&bars.p_full), 128);
    mbar_init(smem_u32(&bars.pv_done), 1);
    mbar_init(smem_u32(&bars.fin), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int *abort_flag = &s_abort;
  bool ok = true;
  // the combine grid launched after this one may be scheduled now: it waits
  // for this grid's completion before reading the partials
  if (tid == 0) pdl_launch_dependents();

  if (warp == 0) {
    // ============================================================ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_tk);
      prefetch_tensormap(&tm_tv);
    }
    int j = 0;
    for (; j < rg.n_tiles; ++j) {
      const int stage = j % kStages;
      if (j >= kStages &&
          !(ok = warp_wait(smem_u32(&bars.kv_empty[stage]), (uint32_t)((j / kStages - 1) & 1), abort_flag)))
        break;
      unsigned char *st = smem + stage * kStageBytes;
      const uint32_t sa = sbase + stage * kStageBytes;
      const uint32_t fb = smem_u32(&bars.kv_full[stage]);
      if (j < rg.n_ctx) {
        // context tile: blocks slot0 .. slot0+3 of the split's range
        const int slot0 = rg.t_begin + 4 * j;
        int ids[4], rows[4];
        uint32_t bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int slot = slot0 + i;
          int r = slot < rg.t_stop ? ctx - slot * kBlock : 0;
          r = r < 0 ? 0 : (r > kBlock ? kBlock : r);
          int id = (r > 0 && TV_CHECK(b < p.B && slot >= 0 && slot < p.max_blocks))
                       ? __ldg(p.block_table + (size_t)b * p.max_blocks + slot) : -1;
          if (r > 0 && (id < 0 || id >= p.num_blocks)) {
            if (lane == 0) {
              pdl_wait();
              set_status(p.status, b, TV_ERR_BLOCK);
            }
            r = 0;
          }
          ids[i] = id;
          rows[i] = r;
          bytes += (uint32_t)r * (uint32_t)(kD * 2 * 2);
        }
        // zero the rows no copy fills: K rows (4 quarters) and V rows (4 quarters)
        bool zeroed = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (rows[i] == kBlock) continue;
          zeroed = true;
          const int nz = (kBlock - rows[i]) * 8;  // 16-byte words per quarter
          for (int w = lane; w < 8 * nz; w += 32) {
            const int kc = w / nz, k = w - kc * nz;  // kc 0-3: K quarters, 4-7: V quarters
            const uint32_t r = rows[i] * 128 + k * 16;
            const uint32_t off = kc < 4 ? kc * kQuarter + i * kBlkQuarter + r
                                        : kKBytes + i * kBlkBytes + (kc - 4) * kBlkQuarter + r;
            *reinterpret_cast<uint4 *>(st + off) = make_uint4(0, 0, 0, 0);
          }
        }
        if (zeroed) fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
        __syncwarp();
        // whole blocks: lanes 0-15 copy K (block lane/4, quarter lane%4),
        // lanes 16-19 copy V of block lane-16 ([4 quarters][16][64])
        if (lane < 20) {
          const int i = lane < 16 ? lane >> 2 : lane - 16;
          if (rows[i] == kBlock) {
            const int row0 = (ids[i] * p.Hkv + kvh) * kBlock;
            if (lane < 16) {
              const int q = lane & 3;
              tma_load_2d(sa + q * kQuarter + i * kBlkQuarter, &tm_k, fb, 64 * q, row0);
            } else {
              tma_load_3d(sa + kKBytes + i * kBlkBytes, &tm_v, fb, 0, row0, 0);
            }
          }
        }
        // a partial last block: row by row; lane q < 4 copies quarter q of K,
        // lane 4 + q quarter q of V
        if (lane < 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (rows[i] == 0 || rows[i] == kBlock) continue;
            const int row0 = (ids[i] * p.Hkv + kvh) * kBlock;
            const int q = lane & 3;
            if (lane < 4) {
              const uint32_t dst = sa + q * kQuarter + i * kBlkQuarter;
              for (int r = 0; r < rows[i]; ++r) tma_load_2d(dst + r * 128, &tm_krow, fb, 64 * q, row0 + r);
            } else {
              const uint32_t dst = sa + kKBytes + i * kBlkBytes + q * kBlkQuarter;
              for (int r = 0; r < rows[i]; ++r) tma_load_2d(dst + r * 128, &tm_vrow, fb, 64 * q, row0 + r);
            }
          }
        }
      } else {
        // node tile: K rows = the nodes of this head (4 quarters per 16-node
        // group), V per group as [4 quarters][16][64]; rows past N hold the
        // next sequence's nodes (finite, masked) or zero fill past the end
        if (lane == 0) {
          const int groups = rg.np / 16;
          mbar_arrive_expect_tx(fb, (uint32_t)groups * 2u * kBlkBytes);
          for (int gi = 0; gi < groups; ++gi) {
            for (int q = 0; q < 4; ++q)
              tma_load_3d(sa + q * kQuarter + gi * kBlkQuarter, &tm_tk, fb, 64 * q, kvh, b * N + 16 * gi);
            tma_load_4d(sa + kKBytes + gi * kBlkBytes, &tm_tv, fb, 0, kvh, b * N + 16 * gi, 0);
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      int dummy = 0;  // copies still in flight get a bounded chance to land
      for (int k = j > kStages ? j - kStages : 0; k < j; ++k)
        wait_slow(smem_u32(&bars.kv_full[k % kStages]), (uint32_t)((k / kStages) & 1), &dummy);
      pdl_wait();
      set_status(p.status, b, TV_ERR_CUDA);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    const uint32_t idesc_pv = idesc_f16(kM, kD, true);
    // One elected lane issues a tile's MMAs and their commits (the same lane
    // every time: elect.sync takes the lowest lane of the converged warp).
    // The descriptors of the K steps and V blocks are the tile's base
    // descriptor plus the step's offset in its start field (shared addresses
    // stay below that field's 256 KB range).
    auto issue_s = [&](int j) {
      const int stage = j % kStages;
      const int keys = j < rg.n_ctx ? kBN : rg.np;
      const uint64_t bd0 = desc_sw128(sbase + stage * kStageBytes, 16);
      const uint32_t id = idesc_f16(kM, keys, false);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          umma_f16_ta(tmem + kColS, tmem + kColQ + kk * 8,
                      bd0 + (uint64_t)(((kk >> 2) * kQuarter + (kk & 3) * 32) >> 4), id, kk > 0 ? 1u : 0u);
        umma_commit(smem_u32(&bars.s_full));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int j) {
      const int stage = j % kStages;
      const int nblk = j < rg.n_ctx ? 4 : rg.np / 16;
      const uint64_t bd0 = desc_sw128(sbase + stage * kStageBytes + kKBytes, kBlkQuarter);
      if (elect_one()) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < nblk)
            umma_f16_ta(tmem + kColO, tmem + kColP + i * 8, bd0 + (uint64_t)((i * kBlkBytes) >> 4), idesc_pv,
                        (j > 0 || i > 0) ? 1u : 0u);
        umma_commit(smem_u32(&bars.pv_done));
        umma_commit(smem_u32(&bars.kv_empty[stage]));
      }
      __syncwarp();
    };
    if (rg.n_tiles > 0) {
      ok = warp_wait(smem_u32(&bars.q_full), 0, abort_flag);
      for (int j = 0; ok && j < rg.n_tiles; ++j) {
        // S_j needs its K tile and the softmax to have read S_{j-1}
        ok = warp_wait(smem_u32(&bars.kv_full[j % kStages]), (uint32_t)((j / kStages) & 1), abort_flag) &&
             (j == 0 || warp_wait(smem_u32(&bars.s_free), (uint32_t)((j - 1) & 1), abort_flag));
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
        // P_{j-1} V_{j-1} once the softmax has written P_{j-1}
        if (j > 0) {
          if (!(ok = warp_wait(smem_u32(&bars.p_full), (uint32_t)((j - 1) & 1), abort_flag))) break;
          tc_fence_after();
          issue_pv(j - 1);
        }
      }
      if (ok) {
        const int jl = rg.n_tiles - 1;
        ok = warp_wait(smem_u32(&bars.p_full), (uint32_t)(jl & 1), abort_flag);
        if (ok) {
          tc_fence_after();
          issue_pv(jl);
        }
      }
    }
    // every MMA issued so far has completed once this arrives
    umma_commit_warp(smem_u32(&bars.fin));
    int dummy = 0;
    if (lane == 0) wait_slow(smem_u32(&bars.fin), 0, &dummy);
    __syncwarp();
    if (!ok && lane == 0) {
      pdl_wait();
      set_status(p.status, b, TV_ERR_CUDA);
    }
  } else {
    // ============================================================ softmax
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(quad * 32) << 16);
    const bool row_ok = m < R;
    const int t = row_ok ? m / G : 0;
    const int g = row_ok ? m - t * G : 0;
    const float qscale = p.qscale;
    const int wl = p.window_left;
    float m_used = -INFINITY, l = 0.f;
    if (rg.n_tiles > 0) {
      // Q row into TMEM (rows past R are zero)
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + (((size_t)b * N + t) * p.Hq + kvh * G + g) * kD);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t qr[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 w = (row_ok && TV_CHECK(kvh * G + g < p.Hq)) ? __ldg(src + 8 * c + v) : make_uint4(0, 0, 0, 0);
          qr[4 * v] = w.x;
          qr[4 * v + 1] = w.y;
          qr[4 * v + 2] = w.z;
          qr[4 * v + 3] = w.w;
        }
        tmem_st32(tlane + kColQ + 32 * c, qr);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.q_full));
    }
    // positions and ancestor masks come from the ancestor kernel before this
    // grid, and every write below (status, partials, output) may race with
    // the grid before: wait for its completion here
    pdl_wait();
    int pos_t = 0;
    unsigned long long allowed = 0;
    if (row_ok && TV_CHECK(b < p.B && t < N)) {
      pos_t = p.pos[(size_t)b * N + t];
      allowed = p.anc[(size_t)b * N + t];
      if (wl >= 0) {
        unsigned long long win = 0;
        for (int a = 0; a < N; ++a)
          if (p.pos[(size_t)b * N + a] >= pos_t - wl) win |= 1ull << a;
        allowed &= win;
      }
    }
    for (int j = 0; j < rg.n_tiles; ++j) {
      if (!(ok = warp_wait(smem_u32(&bars.s_full), (uint32_t)(j & 1), abort_flag))) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(tlane + kColS, sr[0]);
      tmem_ld32(tlane + kColS + 32, sr[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.s_free));  // the S columns may be refilled
      const bool node = j >= rg.n_ctx;
      float s[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      if (!row_ok) {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = -INFINITY;
      } else if (node) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= N || !((allowed >> c) & 1ull)) s[c] = -INFINITY;
      } else {
        const int kb = (rg.t_begin + 4 * j) * kBlock;
        const int c0 = wl >= 0 ? pos_t - wl - kb : 0;
        const int c1 = min(ctx, rg.t_stop * kBlock) - kb;
        if (c0 > 0 || c1 < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < c0 || c >= c1) s[c] = -INFINITY;
        }
      }
      float mt[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) mt[i] = fmaxf(fmaxf(s[i], s[i + 16]), fmaxf(s[i + 32], s[i + 48]));
#pragma unroll
      for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) mt[i] = fmaxf(mt[i], mt[i + w]);
      const float mxs = mt[0] * qscale;
      // rescale O only when some row's max grew by more than 2^kTau (a warp
      // decides together: tcgen05.ld/st are warp-collective)
      const bool need = m_used != -INFINITY && mxs > m_used + kTau;
      if (j > 0) {
        // P V of the previous tile done: P is free and O quiescent
        if (!(ok = warp_wait(smem_u32(&bars.pv_done), (uint32_t)((j - 1) & 1), abort_flag))) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m_used - mxs) : 1.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(tlane + kColO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tlane + kColO + c * 32, o);
        }
        tmem_wait_st();
        if (need) {
          l *= alpha;
          m_used = mxs;
        }
      }
      if (m_used == -INFINITY) m_used = mxs;
      // a running max of -inf means every score so far is -inf: 2^(-inf) = 0
      const float neg_m = m_used != -INFINITY ? -m_used : 0.f;
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float p0 = ex2(fmaf(s[c], qscale, neg_m));
        const float p1 = ex2(fmaf(s[c + 1], qscale, neg_m));
        ps[(c >> 1) & 7] += p0 + p1;
        pk[c >> 1] = pack_bf16(p0, p1);
      }
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      tmem_st32(tlane + kColP, pk);  // key 2c in the low half of column c
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full));
    }
    if (ok && rg.n_tiles > 0) {
      ok = warp_wait(smem_u32(&bars.pv_done), (uint32_t)((rg.n_tiles - 1) & 1), abort_flag);
      tc_fence_after();
    }
    // epilogue: bf16 output with one split, else fp32 partials (a split
    // without tiles writes max -inf, sum 0: the combine gives it weight 0).
    // Every lane of a warp reads TMEM (tcgen05.ld is warp-collective; ok and
    // the tile count are warp-uniform); only rows < R write.
    if (ok) {
      if (p.splits == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16 *dst = p.out + (((size_t)b * N + t) * p.Hq + kvh * G + g) * kD;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          if (rg.n_tiles > 0) {
            tmem_ld32(tlane + kColO + c * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
              w.y = pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
              w.z = pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
              w.w = pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
              *reinterpret_cast<uint4 *>(dst + c * 32 + e) = w;
            }
          }
        }
      } else {
        const size_t row = ((size_t)bk * p.splits + split) * R + m;
        const bool row_in = row_ok && TV_CHECK(row < (size_t)p.B * p.Hkv * p.splits * R);
        if (rg.n_tiles > 0) {
          float *dst = p.part_o + row * kD;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[32];
            tmem_ld32(tlane + kColO + c * 32, o);
            tmem_wait_ld();
            if (row_in) {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(dst + c * 32 + e) =
                    make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
            }
          }
        }
        if (row_in) p.part_ml[row] = make_float2(rg.n_tiles > 0 ? m_used : -INFINITY, l);
      }
    }
    if (!ok && lane == 0) set_status(p.status, b, TV_ERR_CUDA);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode256() {
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

bool map256(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
            const uint32_t *box) {
  auto fn = encode256();
  if (!fn) return false;
  const uint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
            reinterpret_cast<const cuuint64_t *>(dims), reinterpret_cast<const cuuint64_t *>(strides),
            reinterpret_cast<const cuuint32_t *>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attention_tc256_supported(const AttnParams &p) {
  return p.D == kD && p.G >= 1 && p.N >= 1 && p.R >= 1 && p.R <= kM && p.N <= kMaxNodes;
}

cudaError_t launch_attention_tc256(const AttnParams &p, cudaStream_t stream) {
  const uint64_t row_bytes = kD * 2;
  CUtensorMap mk, mkr, mv, mvr, mtk, mtv;
  {
    // cache rows (block, head, token) of 256 d: K per (block, quarter) and per
    // row, V blocks whole as [4 quarters][16][64] and per (row, quarter)
    const uint64_t rows = (uint64_t)(p.num_blocks > 0 ? p.num_blocks : 1) * p.Hkv * kBlock;
    const uint64_t dims2[2] = {(uint64_t)kD, rows};
    const uint64_t str2[1] = {row_bytes};
    const uint32_t box16[2] = {64, (uint32_t)kBlock};
    const uint32_t box1[2] = {64, 1};
    const uint64_t dims3[3] = {64, rows, 4};
    const uint64_t str3[2] = {row_bytes, 128};
    const uint32_t box3[3] = {64, (uint32_t)kBlock, 4};
    if (!map256(&mk, p.k_cache, 2, dims2, str2, box16) || !map256(&mkr, p.k_cache, 2, dims2, str2, box1) ||
        !map256(&mv, p.v_cache, 3, dims3, str3, box3) || !map256(&mvr, p.v_cache, 2, dims2, str2, box1))
      return cudaErrorInvalidValue;
  }
  {
    // tree K [B*N][Hkv][256]: 16 consecutive nodes of one head per quarter;
    // tree V viewed as [quarter][node][head][64]: 16 nodes as [4][16][64]
    const uint64_t dimsk[3] = {(uint64_t)kD, (uint64_t)p.Hkv, (uint64_t)p.B * p.N};
    const uint64_t strk[2] = {row_bytes, row_bytes * p.Hkv};
    const uint32_t boxk[3] = {64, 1, 16};
    const uint64_t dims[4] = {64, (uint64_t)p.Hkv, (uint64_t)p.B * p.N, 4};
    const uint64_t str[3] = {row_bytes, row_bytes * p.Hkv, 128};
    const uint32_t box[4] = {64, 1, 16, 4};
    if (!map256(&mtk, p.k_tree, 3, dimsk, strk, boxk) || !map256(&mtv, p.v_tree, 4, dims, str, box))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(attn_tc256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.B * p.Hkv, p.splits);
  e = launch_pdl(attn_tc256_kernel, grid, dim3(kThreads), kSmemBytes, stream, mk, mkr, mv, mvr, mtk, mtv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tv
