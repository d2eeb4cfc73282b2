// Tree attention on the 5th-generation tensor cores (tcgen05), head dim 128.
//
// Source: "Tree spec-decode -> vLLM serve integration spec", "2. Verify: tree
// attention mask": every node attends the whole paged context of its sequence
// plus its ancestors and itself, composed with the layer's sliding window.
//
// Why tensor cores: the G = Hq/Hkv query heads of a KV head and the N tree
// nodes share every K/V row, so one KV head serves R = G*N rows (128 for
// 32 nodes x 4 heads): 128 flop per byte of KV, far beyond what CUDA cores
// sustain at HBM speed.  R rows are exactly one M = 128 UMMA tile.
//
// Design (one persistent CTA per SM, 192 threads):
//   warp 0     TMA producer: Q tile once per (sequence, KV head) segment, then
//              64-key K/V tiles (four 16-token paged blocks, 128-byte swizzle)
//              into a 4-stage shared-memory ring; the tree node K/V rows form
//              one more tile per segment.
//   warp 1     TMEM allocation and the single MMA-issuing thread:
//              S_j = Q K_j^T into a double-buffered TMEM S tile, then
//              O += P_j V_j (V read as an MN-major operand) into TMEM O.
//   warps 2-5  softmax: thread r owns row r; reads S_j from TMEM, applies the
//              context / window / ancestor mask, keeps the running max and sum,
//              writes P_j (bf16) to swizzled shared memory.  O is rescaled in
//              TMEM only when the row max grows by more than 2^8 (the final
//              division by the running sum makes any reference max exact).
// Work balance: the (sequence, KV head, tile) list, ragged in sequence length,
// is cut into equal contiguous ranges, one per CTA.  A (sequence, KV head)
// pair that falls inside one range is written directly; a pair cut across
// ranges leaves (max, sum, O) partials that a small combine kernel merges.
// Every mbarrier wait is bounded in time; on expiry the kernel records
// TV_ERR_CUDA in status[] and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "attention.cuh"
#include "tc_ptx.cuh"

namespace tv {
namespace {

using namespace ptx;

constexpr int kD = 128;
constexpr int kM = 128;                 // UMMA M: rows per tile
constexpr int kBN = 64;                 // keys per context tile (4 paged blocks)
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kMaxB = 1024;             // sequences the in-CTA schedule can hold
constexpr uint32_t kQChunk = kM * 64 * 2;              // [128 rows][64 d] bf16 = 16 KB
constexpr uint32_t kKVChunk = kBN * 64 * 2;            // [64 keys][64 d] bf16 = 8 KB
constexpr uint32_t kStageBytes = 4 * kKVChunk;         // K (2 chunks) + V (2 chunks)
constexpr uint32_t kPBytes = kM * kBN * 2;             // [128 rows][64 keys] bf16 = 16 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = 2 * kQChunk;
constexpr uint32_t kOffP = kOffKV + kStages * kStageBytes;
constexpr uint32_t kOffPre = kOffP + 2 * kPBytes;
constexpr uint32_t kOffCtx = kOffPre + 4 * (kMaxB + 1);
constexpr uint32_t kSmemBytes = kOffCtx + 4 * kMaxB + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;     // S0 [0,64), S1 [64,128), O [128,256)
constexpr uint32_t kColO = 128;
constexpr float kTau = 8.0f;            // rescale O only when the max grows by > 2^8
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait at most

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct TcParams {
  AttnParams a;
  int *pre_out;       // [B+1] flat tile offsets, written by CTA 0 for the combine
  float *part_o;      // [2*P][128][128]
  float2 *part_ml;    // [2*P][128]
  int node_pad;       // N rounded up to 16
};

struct Bars {
  unsigned long long kv_full[kStages];
  unsigned long long kv_empty[kStages];
  unsigned long long q_full, q_empty;
  unsigned long long s_full[2];
  unsigned long long p_full[2];
  unsigned long long pv_done[2];
  unsigned long long o_free;
  unsigned long long fin;
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: false when the barrier did not complete within kWaitNs or
// another role has already given up (abort flag).
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// UMMA shared-memory descriptor, 128-byte swizzle (sm_100 layout):
// start address >> 4 [0,14), leading byte offset >> 4 [16,30), stride byte
// offset >> 4 [32,46), descriptor version 1 at bit 46, swizzle mode 2 at [61,64).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// A K-major, B K-major or MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The per-CTA schedule: pre[b] is the flat index of sequence b's first tile
// (its Hkv pairs are consecutive, each with tiles(b) = context tiles + 1 node
// tile); pre[B] is the total.
struct Cursor {
  const int *pre;
  int B, Hkv;
  long long f, hi;
  int b, kvh, u, tiles;

  __device__ void locate(long long flat) {
    f = flat;
    int lo = 0, up = B - 1;
    while (lo < up) {  // largest b with pre[b] <= f
      const int mid = (lo + up + 1) >> 1;
      if (pre[mid] <= f) lo = mid;
      else up = mid - 1;
    }
    b = lo;
    tiles = (pre[b + 1] - pre[b]) / Hkv;
    const int r = (int)(f - pre[b]);
    kvh = r / tiles;
    u = r - kvh * tiles;
  }
  __device__ bool valid() const { return f < hi; }
  __device__ bool seg_start(long long lo_f) const { return f == lo_f || u == 0; }
  __device__ bool seg_end() const { return f == hi - 1 || u == tiles - 1; }
  __device__ void next() {
    ++f;
    if (++u == tiles) {
      u = 0;
      if (++kvh == Hkv) {
        kvh = 0;
        ++b;
        if (b < B) tiles = (pre[b + 1] - pre[b]) / Hkv;
      }
    }
  }
};

__device__ __forceinline__ int ctx_tiles(int ctx, int window_left) {
  const int blk_lo = first_visible_block(ctx, window_left);
  const int nblk = (ctx + kBlock - 1) / kBlock - blk_lo;
  return nblk > 0 ? (nblk + 3) / 4 : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
               const __grid_constant__ CUtensorMap tm_vc,
               const __grid_constant__ CUtensorMap tm_kc_row,
               const __grid_constant__ CUtensorMap tm_vc_row,
               const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
               const TcParams tp) {
  const AttnParams &p = tp.a;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  int *s_pre = reinterpret_cast<int *>(smem + kOffPre);
  int *s_ctx = reinterpret_cast<int *>(smem + kOffCtx);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, N = p.N, G = p.G, R = p.R;
  const int NP = tp.node_pad;

  // ---- schedule: context tiles per sequence, prefix over (sequence, KV head)
  for (int b = tid; b < B; b += kThreads) {
    int ctx = p.ctx_len[b];
    const int cap = p.max_blocks * kBlock;
    if (ctx < 0 || ctx > cap) {
      if (blockIdx.x == 0) set_status(p.status, b, TV_ERR_BLOCK);
      ctx = ctx < 0 ? 0 : cap;
    }
    s_ctx[b] = ctx;
    s_pre[b + 1] = (ctx_tiles(ctx, p.window_left) + 1) * Hkv;
  }
  if (tid == 0) {
    s_pre[0] = 0;
    s_abort = 0;
  }
  // zero the Q rows no TMA ever writes (R < 128)
  if (R < kM) {
    const int words = (kM - R) * 8;  // 16-byte words per chunk
    for (int i = tid; i < 2 * words; i += kThreads) {
      const int c = i / words, w = i - c * words;
      *reinterpret_cast<uint4 *>(smem + kOffQ + c * kQChunk + R * 128 + w * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan of s_pre[1..B]
    const int per = (B + 31) / 32;
    const int b0 = lane * per, b1 = min(B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += s_pre[b + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      run += s_pre[b + 1];
      s_pre[b + 1] = run;
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32 * 2) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.kv_full[s]), 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars.o_free), 128);
    mbar_init(smem_u32(&bars.fin), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const long long T = s_pre[B];
  const long long P = gridDim.x;
  const long long lo = (long long)blockIdx.x * T / P;
  const long long hi = (long long)(blockIdx.x + 1) * T / P;
  if (blockIdx.x == 0)
    for (int b = tid; b <= B; b += kThreads) tp.pre_out[b] = s_pre[b];
  volatile int *abort_flag = &s_abort;

  Cursor cur{s_pre, B, Hkv, hi, hi, 0, 0, 0, 1};
  if (lo < hi) cur.locate(lo);  // an empty range leaves f == hi: nothing to do

  if (warp == 0) {
    // ======================================================== TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_kc);
      prefetch_tensormap(&tm_vc);
      prefetch_tensormap(&tm_kt);
      prefetch_tensormap(&tm_vt);
    }
    long long j = 0;
    int seg = 0;
    int ctx = 0, blk_lo = 0;
    bool ok = true;
    while (ok && cur.valid()) {
      const int b = cur.b, kvh = cur.kvh;
      if (cur.seg_start(lo)) {
        if (lane == 0 && seg > 0) ok = wait_bar(smem_u32(&bars.q_empty), (seg - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t qb = smem_u32(&bars.q_full);
          mbar_arrive_expect_tx(qb, 2u * R * 128u);
          tma_load_3d(sbase + kOffQ, &tm_q, qb, 0, kvh * G, b * N);
          tma_load_3d(sbase + kOffQ + kQChunk, &tm_q, qb, 64, kvh * G, b * N);
        }
        ctx = s_ctx[b];
        blk_lo = first_visible_block(ctx, p.window_left);
        ++seg;
      }
      const int stage = (int)(j % kStages);
      if (lane == 0 && j >= kStages)
        ok = wait_bar(smem_u32(&bars.kv_empty[stage]), (uint32_t)((j / kStages - 1) & 1), abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      unsigned char *st = smem + kOffKV + stage * kStageBytes;
      const uint32_t st_addr = sbase + kOffKV + stage * kStageBytes;
      const uint32_t fb = smem_u32(&bars.kv_full[stage]);
      const int nct = cur.tiles - 1;
      if (cur.u < nct) {
        // context tile: paged blocks blk_lo + 4u .. +3
        int ids[4], rows[4];
        uint32_t bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int slot = blk_lo + 4 * cur.u + i;
          int r = ctx - slot * kBlock;
          r = r < 0 ? 0 : (r > kBlock ? kBlock : r);
          int id = -1;
          if (r > 0) {
            id = p.block_table[(size_t)b * p.max_blocks + slot];
            if (id < 0 || id >= p.num_blocks) {
              if (lane == 0) set_status(p.status, b, TV_ERR_BLOCK);
              r = 0;
            }
          }
          ids[i] = id;
          rows[i] = r;
          bytes += (uint32_t)r * 128u * 4u;
        }
        // zero the rows no copy fills (past the context end, bad blocks)
        bool zeroed = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (rows[i] == kBlock) continue;
          zeroed = true;
          const int nz = (kBlock - rows[i]) * 8;  // 16-byte words per chunk
          for (int w = lane; w < 4 * nz; w += 32) {
            const int c = w / nz, k = w - c * nz;
            *reinterpret_cast<uint4 *>(st + c * kKVChunk + (i * kBlock + rows[i]) * 128 + k * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        if (zeroed) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (rows[i] == 0) continue;
            const int row0 = (ids[i] * Hkv + kvh) * kBlock;
            const uint32_t dk = st_addr + i * kBlock * 128;
            const uint32_t dv = dk + 2 * kKVChunk;
            if (rows[i] == kBlock) {
              tma_load_2d(dk, &tm_kc, fb, 0, row0);
              tma_load_2d(dk + kKVChunk, &tm_kc, fb, 64, row0);
              tma_load_2d(dv, &tm_vc, fb, 0, row0);
              tma_load_2d(dv + kKVChunk, &tm_vc, fb, 64, row0);
            } else {
              for (int r = 0; r < rows[i]; ++r) {
                tma_load_2d(dk + r * 128, &tm_kc_row, fb, 0, row0 + r);
                tma_load_2d(dk + kKVChunk + r * 128, &tm_kc_row, fb, 64, row0 + r);
                tma_load_2d(dv + r * 128, &tm_vc_row, fb, 0, row0 + r);
                tma_load_2d(dv + kKVChunk + r * 128, &tm_vc_row, fb, 64, row0 + r);
              }
            }
          }
        }
      } else {
        // node tile: rows 0..N-1 from k_tree / v_tree, rows N..NP-1 zero
        if (NP > N) {
          const int nz = (NP - N) * 8;
          for (int w = lane; w < 4 * nz; w += 32) {
            const int c = w / nz, k = w - c * nz;
            *reinterpret_cast<uint4 *>(st + c * kKVChunk + N * 128 + k * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, 4u * N * 128u);
          tma_load_3d(st_addr, &tm_kt, fb, 0, kvh, b * N);
          tma_load_3d(st_addr + kKVChunk, &tm_kt, fb, 64, kvh, b * N);
          tma_load_3d(st_addr + 2 * kKVChunk, &tm_vt, fb, 0, kvh, b * N);
          tma_load_3d(st_addr + 3 * kKVChunk, &tm_vt, fb, 64, kvh, b * N);
        }
      }
      ++j;
      cur.next();
    }
    if (!ok && lane == 0) {
      // give copies still in flight a bounded chance to land before exit
      int dummy = 0;
      for (long long k = j > kStages ? j - kStages : 0; k < j; ++k)
        wait_bar(smem_u32(&bars.kv_full[k % kStages]), (uint32_t)((k / kStages) & 1), &dummy);
      if (seg > 0) wait_bar(smem_u32(&bars.q_full), (seg - 1) & 1, &dummy);
      set_status(p.status, cur.valid() ? cur.b : 0, TV_ERR_CUDA);
    }
  } else if (warp == 1) {
    // ======================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc_pv = make_idesc(kM, kD, true);
      bool ok = true;
      long long j = 0;
      int seg = 0;
      // pending PV (tile j-1): stage, node-tile flag, first-in-segment, segment ordinal
      int pv_stage = 0, pv_keys = 0, pv_first = 0, pv_seg = 0;
      bool pv_pending = false;
      auto issue_pv = [&](long long jj) -> bool {
        if (!wait_bar(smem_u32(&bars.p_full[jj & 1]), (uint32_t)((jj >> 1) & 1), abort_flag))
          return false;
        if (pv_first && pv_seg > 0)
          if (!wait_bar(smem_u32(&bars.o_free), (uint32_t)((pv_seg - 1) & 1), abort_flag))
            return false;
        tc_fence_after();
        const uint32_t pa = sbase + kOffP + (uint32_t)(jj & 1) * kPBytes;
        const uint32_t va = sbase + kOffKV + pv_stage * kStageBytes + 2 * kKVChunk;
        for (int ks = 0; ks < pv_keys / 16; ++ks) {
          const uint64_t ad = sw128_desc(pa + ks * 32, 16, 1024);
          const uint64_t bd = sw128_desc(va + ks * 2048, kKVChunk, 1024);
          umma_f16(tmem + kColO, ad, bd, idesc_pv, (ks > 0 || !pv_first) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.pv_done[jj & 1]));
        umma_commit(smem_u32(&bars.kv_empty[pv_stage]));
        return true;
      };
      while (ok && cur.valid()) {
        const bool first = cur.seg_start(lo);
        const bool last = cur.seg_end();
        if (first) {
          ok = wait_bar(smem_u32(&bars.q_full), seg & 1, abort_flag);
          if (!ok) break;
          ++seg;
        }
        const int stage = (int)(j % kStages);
        ok = wait_bar(smem_u32(&bars.kv_full[stage]), (uint32_t)((j / kStages) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
        const bool node = cur.u == cur.tiles - 1;
        const int keys = node ? NP : kBN;
        const uint32_t idesc_s = make_idesc(kM, keys, false);
        const uint32_t ka = sbase + kOffKV + stage * kStageBytes;
        const uint32_t sc = tmem + (uint32_t)(j & 1) * kBN;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint32_t c = ks >> 2, kk = ks & 3;
          const uint64_t ad = sw128_desc(sbase + kOffQ + c * kQChunk + kk * 32, 16, 1024);
          const uint64_t bd = sw128_desc(ka + c * kKVChunk + kk * 32, 16, 1024);
          umma_f16(sc, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.s_full[j & 1]));
        if (last) umma_commit(smem_u32(&bars.q_empty));
        if (pv_pending) {
          ok = issue_pv(j - 1);
          if (!ok) break;
        }
        pv_pending = true;
        pv_stage = stage;
        pv_keys = keys;
        pv_first = first;
        pv_seg = seg - 1;
        ++j;
        cur.next();
      }
      if (ok && pv_pending) ok = issue_pv(j - 1);
      // every MMA issued so far has completed once this arrives
      umma_commit(smem_u32(&bars.fin));
      int dummy = 0;
      wait_bar(smem_u32(&bars.fin), 0, &dummy);
      if (!ok) set_status(p.status, cur.valid() ? cur.b : 0, TV_ERR_CUDA);
    }
  } else {
    // ======================================================== softmax / epilogue
    const int quad = warp & 3;
    const int m = quad * 32 + lane;                   // row == TMEM lane
    const uint32_t tlane = tmem + ((uint32_t)(quad * 32) << 16);
    const bool row_ok = m < R;
    const int t = row_ok ? m / G : 0;
    const int g = row_ok ? m - t * G : 0;
    const float qscale = p.qscale;
    const int wl = p.window_left;
    long long j = 0;
    int seg = 0;
    bool ok = true;
    float m_used = -INFINITY, l = 0.f;
    int ctx = 0, blk_lo = 0, pos_t = 0;
    unsigned long long allowed = 0;
    long long seg_f0 = lo;
    bool seg_complete = false;
    const uint32_t p_row = (uint32_t)m * 128u;
    const uint32_t sw = (uint32_t)(m & 7);
    while (cur.valid()) {
      const int b = cur.b, kvh = cur.kvh;
      if (cur.seg_start(lo)) {
        m_used = -INFINITY;
        l = 0.f;
        ctx = s_ctx[b];
        blk_lo = first_visible_block(ctx, wl);
        seg_f0 = cur.f;
        seg_complete = cur.u == 0 && cur.f + (cur.tiles - 1) <= hi - 1;
        allowed = 0;
        if (row_ok) {
          pos_t = p.pos[(size_t)b * N + t];
          allowed = p.anc[(size_t)b * N + t];
          if (wl >= 0) {
            unsigned long long win = 0;
            for (int a = 0; a < N; ++a)
              if (p.pos[(size_t)b * N + a] >= pos_t - wl) win |= 1ull << a;
            allowed &= win;
          }
        }
      }
      // every wait is made warp-uniform: the tcgen05.ld/st that follow are
      // warp-collective
      ok = __all_sync(0xffffffffu,
                      wait_bar(smem_u32(&bars.s_full[j & 1]), (uint32_t)((j >> 1) & 1), abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(tlane + (uint32_t)(j & 1) * kBN, sr[0]);
      tmem_ld32(tlane + (uint32_t)(j & 1) * kBN + 32, sr[1]);
      tmem_wait_ld();
      const bool node = cur.u == cur.tiles - 1;
      float s[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      // mask
      if (!row_ok) {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = -INFINITY;
      } else if (node) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= N || !((allowed >> c) & 1ull)) s[c] = -INFINITY;
      } else {
        const int kb = (blk_lo + 4 * cur.u) * kBlock;
        int c0 = wl >= 0 ? pos_t - wl - kb : 0;
        int c1 = ctx - kb;
        if (c0 > 0 || c1 < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < c0 || c >= c1) s[c] = -INFINITY;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 64; ++c) mx = fmaxf(mx, s[c]);
      const float mxs = mx * qscale;
      // Rescale O only when some row's max grew by more than 2^kTau.  The
      // decision is made per warp (tcgen05.ld/st are warp-collective); rows that
      // do not need it scale by 1.  A finite running max means an earlier tile
      // of this segment exists, so PV_{j-1} is the last write to O.
      const bool need = m_used != -INFINITY && mxs > m_used + kTau;
      if (__any_sync(0xffffffffu, need)) {
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars.pv_done[(j - 1) & 1]),
                                              (uint32_t)(((j - 1) >> 1) & 1), abort_flag));
        if (!ok) break;
        tc_fence_after();
        const float alpha = need ? ex2(m_used - mxs) : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
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
      // P = 2^(s*scale - m), written as bf16 into the 128B-swizzled P buffer
      float rowsum = 0.f;
      uint32_t pk[32];
      const bool live = m_used != -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float p0 = live ? ex2(fmaf(s[c], qscale, -m_used)) : 0.f;
        const float p1 = live ? ex2(fmaf(s[c + 1], qscale, -m_used)) : 0.f;
        rowsum += p0 + p1;
        pk[c >> 1] = pack_bf16(p0, p1);
      }
      l += rowsum;
      if (j >= 2) {
        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars.pv_done[j & 1]),
                                              (uint32_t)(((j - 2) >> 1) & 1), abort_flag));
        if (!ok) break;
      }
      const uint32_t pbuf = sbase + kOffP + (uint32_t)(j & 1) * kPBytes + p_row;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(pbuf + (((uint32_t)u ^ sw) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                     pk[4 * u + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full[j & 1]));
      if (cur.seg_end()) {
        // epilogue: wait for PV_j, read O, write output or partial
        ok = __all_sync(0xffffffffu,
                        wait_bar(smem_u32(&bars.pv_done[j & 1]), (uint32_t)((j >> 1) & 1), abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (seg_complete) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16 *dst =
              p.out + (((size_t)b * N + t) * p.Hq + kvh * G + g) * kD;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tlane + kColO + c * 32, o);
            tmem_wait_ld();
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
          const int slot = 2 * (int)blockIdx.x + (seg_f0 == lo ? 0 : 1);
          float *dst = tp.part_o + ((size_t)slot * kM + m) * kD;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tlane + kColO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<uint4 *>(dst + c * 32 + e) = make_uint4(o[e], o[e + 1], o[e + 2], o[e + 3]);
          }
          tp.part_ml[(size_t)slot * kM + m] = make_float2(m_used, l);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.o_free));
        ++seg;
      }
      ++j;
      cur.next();
    }
    if (!ok && lane == 0) set_status(p.status, cur.valid() ? cur.b : 0, TV_ERR_CUDA);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the partials of every (sequence, KV head) pair whose tiles were split
// across CTAs.  One warp per output row; lane l owns dims 4l .. 4l+3.
__global__ void attn_tc_combine_kernel(const TcParams tp, int P) {
  const AttnParams &p = tp.a;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.Hkv * p.R;
  if (row >= rows) return;
  const int pair = (int)(row / p.R), m = (int)(row - (long long)pair * p.R);
  const int b = pair / p.Hkv, kvh = pair - b * p.Hkv;
  const long long T = tp.pre_out[p.B];
  const int tiles = (tp.pre_out[b + 1] - tp.pre_out[b]) / p.Hkv;
  const long long S = tp.pre_out[b] + (long long)kvh * tiles, E = S + tiles;
  auto cta_of = [&](long long f) { return (int)(((f + 1) * P + T - 1) / T - 1); };
  const int c0 = cta_of(S), c1 = cta_of(E - 1);
  if (c0 == c1) return;  // written directly by its CTA
  // CTA c covers flat tiles [c*T/P, (c+1)*T/P); ranges can be empty when T < P
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c) {
    const long long loc = (long long)c * T / P;
    if (loc == (long long)(c + 1) * T / P) continue;
    const int slot = 2 * c + ((c == c0 && loc < S) ? 1 : 0);
    M = fmaxf(M, tp.part_ml[(size_t)slot * kM + m].x);
  }
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = c0; c <= c1; ++c) {
    const long long loc = (long long)c * T / P;
    if (loc == (long long)(c + 1) * T / P) continue;
    const int slot = 2 * c + ((c == c0 && loc < S) ? 1 : 0);
    const float2 ml = tp.part_ml[(size_t)slot * kM + m];
    if (ml.x == -INFINITY) continue;
    const float w = exp2f(ml.x - M);
    L += ml.y * w;
    const float4 o = *reinterpret_cast<const float4 *>(tp.part_o + ((size_t)slot * kM + m) * kD + lane * 4);
    acc.x += o.x * w;
    acc.y += o.y * w;
    acc.z += o.z * w;
    acc.w += o.w * w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int t = m / p.G, g = m - t * p.G;
  __nv_bfloat16 *dst = p.out + (((size_t)b * p.N + t) * p.Hq + kvh * p.G + g) * kD + lane * 4;
  uint2 w;
  w.x = pack_bf16(acc.x * inv, acc.y * inv);
  w.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(dst) = w;
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool make_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
              const uint64_t *strides, const uint32_t *box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
            reinterpret_cast<const cuuint64_t *>(dims), reinterpret_cast<const cuuint64_t *>(strides),
            reinterpret_cast<const cuuint32_t *>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attention_tc_supported(const AttnParams &p) {
  return p.D == kD && p.G >= 1 && p.N >= 1 && p.R >= 1 && p.R <= kM && p.N <= kMaxNodes &&
         p.B <= kMaxB && p.G <= 256;
}

size_t attention_tc_workspace(int B, int P) {
  const size_t pre = ((size_t)(B + 1) * sizeof(int) + 255) / 256 * 256;
  const size_t ml = ((size_t)2 * P * kM * sizeof(float2) + 255) / 256 * 256;
  const size_t o = (size_t)2 * P * kM * kD * sizeof(float);
  return pre + ml + o;
}

cudaError_t launch_attention_tc(const AttnParams &a, void *workspace, cudaStream_t stream) {
  const int P = sm_count();
  TcParams tp{};
  tp.a = a;
  char *ws = static_cast<char *>(workspace);
  tp.pre_out = reinterpret_cast<int *>(ws);
  ws += ((size_t)(a.B + 1) * sizeof(int) + 255) / 256 * 256;
  tp.part_ml = reinterpret_cast<float2 *>(ws);
  ws += ((size_t)2 * P * kM * sizeof(float2) + 255) / 256 * 256;
  tp.part_o = reinterpret_cast<float *>(ws);
  tp.node_pad = (a.N + 15) / 16 * 16;

  CUtensorMap mq, mkc, mvc, mkcr, mvcr, mkt, mvt;
  const uint64_t row_bytes = kD * 2;
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hq, (uint64_t)a.B * a.N};
    const uint64_t str[2] = {row_bytes, row_bytes * a.Hq};
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)a.N};
    if (!make_map(&mq, a.q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t rows = (uint64_t)(a.num_blocks > 0 ? a.num_blocks : 1) * a.Hkv * kBlock;
    const uint64_t dims[2] = {(uint64_t)kD, rows};
    const uint64_t str[1] = {row_bytes};
    const uint32_t box[2] = {64, (uint32_t)kBlock};
    const uint32_t box1[2] = {64, 1};
    if (!make_map(&mkc, a.k_cache, 2, dims, str, box) || !make_map(&mvc, a.v_cache, 2, dims, str, box) ||
        !make_map(&mkcr, a.k_cache, 2, dims, str, box1) || !make_map(&mvcr, a.v_cache, 2, dims, str, box1))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.B * a.N};
    const uint64_t str[2] = {row_bytes, row_bytes * a.Hkv};
    const uint32_t box[3] = {64, 1, (uint32_t)a.N};
    if (!make_map(&mkt, a.k_tree, 3, dims, str, box) || !make_map(&mvt, a.v_tree, 3, dims, str, box))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_tc_kernel<<<P, kThreads, kSmemBytes, stream>>>(mq, mkc, mvc, mkcr, mvcr, mkt, mvt, tp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long rows = (long long)a.B * a.Hkv * a.R;
  const int wpb = 8;
  attn_tc_combine_kernel<<<(unsigned)((rows + wpb - 1) / wpb), wpb * 32, 0, stream>>>(tp, P);
  return cudaGetLastError();
}

}  // namespace tv
