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
// Design (one persistent CTA per SM, 11 warps = 352 threads):
//   warps 0, 10  TMA producers, alternate 64-key tiles: K as eight 2-D boxes
//                (two 64-dim halves x four 16-token paged blocks, 128-byte
//                swizzle), V as four 3-D boxes, one copy per lane so the copies
//                go out together, into a 6-stage 32 KB ring; block ids are read
//                32 slots at a time one window ahead; the tree node K/V rows
//                form one more tile per segment.
//   warp 1       TMEM allocation and the only warp that issues tcgen05.mma (one
//                elected lane per instruction group; the warp polls its
//                barriers warp-uniformly and issues a ready P V before a late
//                S): S_j = Q K_j^T into a double-buffered TMEM S tile (Q read
//                from TMEM), O_x += P_j V_j (P from TMEM, V read as an MN-major
//                shared-memory operand).
//   warps 2-5,   two softmax warpgroups taking alternate tiles, each with its
//   6-9          own running max / sum and O accumulator in TMEM: thread r owns
//                row r, reads S_j, frees it at once, applies the context /
//                window / ancestor mask, writes P_j as bf16 pairs to TMEM.  O is
//                rescaled in TMEM only when the row max grows by more than 2^8
//                (the final division by the running sum makes any reference
//                max exact).  At the end of a (sequence, KV head) segment the
//                two warpgroups exchange (max, sum) and each merges half of the
//                columns of O_0 and O_1; warpgroup 0 writes Q into TMEM at a
//                segment start, warpgroup 1 loads the next segment's Q early.
// TMEM (512 columns): S0, S1 [0,128); O0, O1 [128,384); P0, P1 [384,448); Q [448,512).
// Work balance: the (sequence, KV head, tile) list, ragged in sequence length,
// is cut into equal contiguous ranges, one per CTA, each cut moved to a pair
// boundary when one lies within a few tiles.  A (sequence, KV head) pair that
// falls inside one range is written directly.  A pair cut across ranges leaves
// one (max, sum, O) partial per piece, merged by attn_tc_combine_kernel.
// Programmatic dependent launch: this grid may start while the kernel before
// it on the stream finishes (the ancestor kernel, or the previous layer's
// combine grid), so its prologue, block-id loads and first K/V copies overlap
// that kernel.  Everything read before griddepcontrol.wait is an
// input no earlier kernel of a verify step writes (context lengths, block
// tables, Q, K/V); ancestor masks and positions are read, and status words
// and the scratch (range starts, descriptors, partials) written, only after
// it.  Data errors found before it are kept in a shared-memory bitmap and
// written to status[] at the end.
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

TV_DEBUG_RECORD(attention_tc)

namespace tv {
namespace {

using namespace ptx;

constexpr int kD = 128;
constexpr int kM = 128;                 // UMMA M: rows per tile
constexpr int kBN = 64;                 // keys per context tile (4 paged blocks)
constexpr int kStages = 6;
constexpr int kWarps = 11;               // producer, S issuer, 2 softmax warpgroups, producer
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxB = 1024;             // sequences the in-CTA schedule can hold
constexpr uint32_t kKVChunk = kBN * 64 * 2;            // [64 keys][64 d] bf16 = 8 KB
constexpr uint32_t kStageBytes = 4 * kKVChunk;         // K (16 KB) + V (16 KB)
constexpr uint32_t kHalfStage = 2 * kKVChunk;          // V starts here within a stage
constexpr uint32_t kBlkChunk = kBlock * 64 * 2;        // [16 keys][64 d] bf16 = 2 KB
constexpr uint32_t kBlkBytes = 2 * kBlkChunk;          // one paged block: [2 halves][16][64]
constexpr uint32_t kOffKV = 0;
constexpr uint32_t kOffPre = kOffKV + kStages * kStageBytes;
constexpr uint32_t kOffCtx = kOffPre + 4 * (kMaxB + 1);
constexpr uint32_t kOffMerge = (kOffCtx + 4 * kMaxB + 15) / 16 * 16;   // [2 seg parity][2 wg][128] float2
constexpr uint32_t kOffEpi = kOffMerge + 4 * kM * 8;   // [8 softmax warps][32 rows][64 B] output staging
constexpr uint32_t kSmemBytes = kOffEpi + 8 * 2048 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;     // S0, S1 [0,128); O0, O1 [128,384); P0, P1 [384,448); Q [448,512)
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 384;         // P as bf16 pairs: 64 keys = 32 columns
constexpr uint32_t kColQ = 448;         // Q as bf16 pairs: 128 dims = 64 columns
constexpr float kTau = 8.0f;            // rescale O only when the max grows by > 2^8
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait at most

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct TcParams {
  AttnParams a;
  long long *lo_out;  // [P+1] first flat tile of every CTA's range (and the total)
  longlong2 *desc;    // [P] the (sequence, KV head) pair CTA c starts and that runs
                      // past its range: (first flat tile, end tile | pair << 32),
                      // first = -1 when there is none
  float *part_o;      // [2*P][128 dims][128 rows] unnormalised partial outputs,
                      // dim-major so that a warp's 32 rows store 128 contiguous bytes
  float2 *part_ml;    // [2*P][128]      (max, sum) of each partial
  int node_pad;       // N rounded up to 16
};

struct Bars {
  unsigned long long kv_full[kStages];
  unsigned long long kv_empty[kStages];
  unsigned long long q_full, q_empty;
  unsigned long long s_full[2];
  unsigned long long s_free[2];
  unsigned long long p_full[2];
  unsigned long long pv_done[2];
  unsigned long long merge;
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

__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  return mbar_try_wait(bar, parity) || wait_bar(bar, parity, abort_flag);
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

// Cut points of the work split.  CTA c's range starts at snap_cut(c T / P):
// an even cut, moved to the nearest (sequence, KV head) pair boundary when one
// lies within kSnap tiles.  A pair cut between CTAs costs a partial per piece,
// an extra segment end and a merge, about as much as streaming kSnap tiles, so
// short pairs (sliding windows, short contexts) are no longer cut at all.  The
// function is monotone, so consecutive ranges meet.
constexpr long long kSnap = 5;
__device__ __forceinline__ long long snap_cut(const int *pre, int B, int Hkv, long long x) {
  if (x <= 0 || x >= pre[B]) return x;
  int lo = 0, up = B - 1;
  while (lo < up) {  // largest b with pre[b] <= x
    const int mid = (lo + up + 1) >> 1;
    if (pre[mid] <= x) lo = mid;
    else up = mid - 1;
  }
  const long long tiles = (pre[lo + 1] - pre[lo]) / Hkv;
  const long long below = pre[lo] + (x - pre[lo]) / tiles * tiles, above = below + tiles;
  const long long d_lo = x - below, d_hi = above - x;
  if (d_lo <= d_hi) return d_lo <= kSnap ? below : x;
  return d_hi <= kSnap ? above : x;
}

// One 32-dim chunk of the bf16 output of the 32 rows a warp owns (lane = row
// 32 * quad + lane, its 32 values packed in pk): staged through the warp's own
// 2 KB of shared memory (16-byte units XOR-swizzled by row, so neither the
// writes nor the reads conflict), then stored so that four lanes write one
// row's 64 contiguous bytes.  Row m = t * G + g goes to out + row_base +
// (t * Hq + g) * 128 + col0; rows m >= R are not stored.
__device__ __forceinline__ void stage_store_bf16(uint32_t stg, const uint32_t (&pk)[16], int lane,
                                                 int quad, __nv_bfloat16 *out, size_t row_base,
                                                 int Hq, int G, int R, int col0) {
  const uint32_t f = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
  for (uint32_t u = 0; u < 4; ++u)
    st_shared_v4(stg + (uint32_t)lane * 64u + ((u ^ f) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                 pk[4 * u + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const uint32_t u = (uint32_t)lane & 3u;
    const uint4 v = ld_shared_v4(stg + (uint32_t)r * 64u + ((u ^ ((uint32_t)(r >> 1) & 3u)) << 4));
    const int m = quad * 32 + r;
    if (m < R) {
      const int t = m / G, g = m - t * G;
      *reinterpret_cast<uint4 *>(out + row_base + ((size_t)t * Hq + g) * kD + col0 + u * 8) = v;
    }
  }
  __syncwarp();  // the staging buffer may be refilled
}

// Programmatic dependent launch: wait until the kernels this grid depends on
// have completed and their writes are visible (returns at once otherwise).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int ctx_tiles(int ctx, int window_left) {
  const int blk_lo = first_visible_block(ctx, window_left);
  const int nblk = (ctx + kBlock - 1) / kBlock - blk_lo;
  return nblk > 0 ? (nblk + 3) / 4 : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_kc,
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
  __shared__ uint32_t s_bad[kMaxB / 32];  // sequences with a bad block id or context length

  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  int *s_pre = reinterpret_cast<int *>(smem + kOffPre);
  int *s_ctx = reinterpret_cast<int *>(smem + kOffCtx);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B, Hkv = p.Hkv, N = p.N, G = p.G, R = p.R;
  const int NP = tp.node_pad;

  // ---- schedule: context tiles per sequence, prefix over (sequence, KV head)
  for (int i = tid; i < kMaxB / 32; i += kThreads) s_bad[i] = 0;
  __syncthreads();
  for (int b = tid; b < B; b += kThreads) {
    int ctx = p.ctx_len[b];
    const int cap = p.max_blocks * kBlock;
    if (ctx < 0 || ctx > cap) {
      if (blockIdx.x == 0) atomicOr(&s_bad[b >> 5], 1u << (b & 31));
      ctx = ctx < 0 ? 0 : cap;
    }
    s_ctx[b] = ctx;
    s_pre[b + 1] = (ctx_tiles(ctx, p.window_left) + 1) * Hkv;
  }
  if (tid == 0) {
    s_pre[0] = 0;
    s_abort = 0;
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
      // test hook: one arrival more than the producer makes, in one CTA
      mbar_init(smem_u32(&bars.kv_full[s]), (s == 0 && (int)blockIdx.x == p.withheld_cta) ? 2 : 1);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.q_full), 128);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.s_free[i]), 128);
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars.merge), 256);
    mbar_init(smem_u32(&bars.o_free), 256);
    mbar_init(smem_u32(&bars.fin), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const long long T = s_pre[B];
  const long long P = gridDim.x;
  const long long lo = snap_cut(s_pre, B, Hkv, (long long)blockIdx.x * T / P);
  const long long hi = snap_cut(s_pre, B, Hkv, (long long)(blockIdx.x + 1) * T / P);
  // A grid launched after this one as a programmatic dependent may be
  // scheduled as CTAs of this grid exit; it must wait for this grid's
  // completion (griddepcontrol.wait) before reading its outputs.
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  volatile int *abort_flag = &s_abort;

  Cursor cur{s_pre, B, Hkv, hi, hi, 0, 0, 0, 1};
  if (lo < hi) cur.locate(lo);  // an empty range leaves f == hi: nothing to do

  if (warp == 0 || warp == kWarps - 1) {
    // ======================================================== TMA producers
    // Two warps share the tiles: warp 0 loads even tiles and every Q tile, the
    // last warp loads odd tiles.  Each runs the whole loop (block ids are
    // fetched 32 slots at a time, one per lane, one window ahead) and skips
    // the tiles of the other.
    const int par = warp == 0 ? 0 : 1;
    if (lane == 0 && par == 0) {
      prefetch_tensormap(&tm_kc);
      prefetch_tensormap(&tm_vc);
      prefetch_tensormap(&tm_kt);
      prefetch_tensormap(&tm_vt);
    }
    int j = 0;
    int seg = 0;
    int ctx = 0, blk_lo = 0, nblk_end = 0, nfull = 0;
    int win_base = 0, cur_id = -1, nxt_id = -1;
    bool ok = true;
    auto load_id = [&](int b, int slot) -> int {
      return (slot < nblk_end && TV_CHECK(b < B && slot >= 0 && slot < p.max_blocks))
                 ? __ldg(p.block_table + (size_t)b * p.max_blocks + slot) : -1;
    };
    while (ok && cur.valid()) {
      const int b = cur.b, kvh = cur.kvh;
      if (cur.seg_start(lo)) {
        ctx = s_ctx[b];
        blk_lo = first_visible_block(ctx, p.window_left);
        nblk_end = (ctx + kBlock - 1) / kBlock;
        nfull = ctx / kBlock;
        win_base = blk_lo + 4 * cur.u;  // a CTA's range may start mid-pair
        cur_id = load_id(b, win_base + lane);
        nxt_id = load_id(b, win_base + 32 + lane);
        ++seg;
      }
      const int nct = cur.tiles - 1;
      const int slot0 = blk_lo + 4 * cur.u;
      if (cur.u < nct && slot0 - win_base >= 32) {
        win_base += 32;
        cur_id = nxt_id;
        nxt_id = load_id(b, win_base + 32 + lane);
      }
      if ((j & 1) != par) {  // the other producer's tile
        ++j;
        cur.next();
        continue;
      }
      const int stage = j % kStages;
      const uint32_t empty_parity = (uint32_t)((j / kStages - 1) & 1);
      // every lane waits for the stage itself (no broadcasts)
      if (j >= kStages) {
        ok = __all_sync(0xffffffffu,
                        wait_fast(smem_u32(&bars.kv_empty[stage]), empty_parity, abort_flag));
        if (!ok) break;
      }
      unsigned char *st = smem + kOffKV + stage * kStageBytes;
      const uint32_t st_addr = sbase + kOffKV + stage * kStageBytes;
      const uint32_t fb = smem_u32(&bars.kv_full[stage]);
      if (cur.u < nct) {
        // context tile: paged blocks blk_lo + 4u .. +3
        // fast path: four whole blocks with valid ids.  Lane c < 8 copies K of
        // block c/2 (d half c%2) into [half][64 keys][64], lanes 8-11 copy V of
        // block c-8 whole ([half][16][64]); every lane works out its own copy.
        const int fblk = lane < 8 ? (lane >> 1) : ((lane - 8) & 3);
        const int fid = __shfl_sync(0xffffffffu, cur_id, (slot0 - win_base + fblk) & 31);
        const bool fgood = lane >= 12 || (fid >= 0 && fid < p.num_blocks);
        if (__all_sync(0xffffffffu, fgood) && slot0 + 4 <= nfull) {
          if (lane == 0) mbar_arrive_expect_tx(fb, kStageBytes);
          __syncwarp();
          const int row0 = (fid * Hkv + kvh) * kBlock;
          if (lane < 8)
            tma_load_2d(st_addr + (lane & 1) * kKVChunk + fblk * kBlkChunk, &tm_kc, fb, 64 * (lane & 1),
                        row0);
          else if (lane < 12)
            tma_load_3d(st_addr + kHalfStage + fblk * kBlkBytes, &tm_vc, fb, 0, row0, 0);
        } else {
        int ids[4], rows[4];
        uint32_t bytes = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int slot = slot0 + i;
          int r = ctx - slot * kBlock;
          r = r < 0 ? 0 : (r > kBlock ? kBlock : r);
          int id = __shfl_sync(0xffffffffu, cur_id, slot - win_base);
          if (r > 0 && (id < 0 || id >= p.num_blocks)) {
            if (lane == 0) atomicOr(&s_bad[b >> 5], 1u << (b & 31));
            r = 0;
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
          const int nz = (kBlock - rows[i]) * 8;  // 16-byte words per half
          for (int w = lane; w < 4 * nz; w += 32) {
            const int kc = w / nz, k = w - kc * nz;  // kc: 0,1 = K halves, 2,3 = V halves
            const int r = rows[i] * 128 + k * 16;
            const uint32_t off = kc < 2 ? kc * kKVChunk + i * kBlkChunk + r
                                        : kHalfStage + i * kBlkBytes + (kc - 2) * kBlkChunk + r;
            *reinterpret_cast<uint4 *>(st + off) = make_uint4(0, 0, 0, 0);
          }
        }
        if (zeroed) fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
        __syncwarp();
        // whole blocks: lanes 0-7 copy K (block lane/2, d half lane%2) into the
        // [half][64 keys][64] K tile, lanes 8-11 copy V block lane-8 whole
        // ([half][16][64]); copies issued by several lanes go out together
        if (lane < 12) {
          const int i = lane < 8 ? lane >> 1 : lane - 8;
          if (rows[i] == kBlock) {
            const int row0 = (ids[i] * Hkv + kvh) * kBlock;
            if (lane < 8) {
              const int h = lane & 1;
              tma_load_2d(st_addr + h * kKVChunk + i * kBlkChunk, &tm_kc, fb, 64 * h, row0);
            } else {
              tma_load_3d(st_addr + kHalfStage + i * kBlkBytes, &tm_vc, fb, 0, row0, 0);
            }
          }
        }
        // a partial last block: row by row
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (rows[i] == 0 || rows[i] == kBlock) continue;
            const int row0 = (ids[i] * Hkv + kvh) * kBlock;
            const uint32_t dk = st_addr + i * kBlkChunk, dv = st_addr + kHalfStage + i * kBlkBytes;
            for (int r = 0; r < rows[i]; ++r) {
              tma_load_2d(dk + r * 128, &tm_kc_row, fb, 0, row0 + r);
              tma_load_2d(dk + kKVChunk + r * 128, &tm_kc_row, fb, 64, row0 + r);
              tma_load_2d(dv + r * 128, &tm_vc_row, fb, 0, row0 + r);
              tma_load_2d(dv + kBlkChunk + r * 128, &tm_vc_row, fb, 64, row0 + r);
            }
          }
        }
        }
      } else {
        // node tile: K rows 0..NP-1 per d half (3-D copy of all nodes of the
        // head), V per 16-node group ([half][16][64]); rows past N hold the
        // next sequence's nodes (finite, masked) or zero fill past the end
        if (lane == 0) {
          const int groups = NP / 16;
          mbar_arrive_expect_tx(fb, 2u * groups * kBlkBytes);
          for (int gi = 0; gi < groups; ++gi) {
            tma_load_3d(st_addr + gi * kBlkChunk, &tm_kt, fb, 0, kvh, b * N + 16 * gi);
            tma_load_3d(st_addr + kKVChunk + gi * kBlkChunk, &tm_kt, fb, 64, kvh, b * N + 16 * gi);
            tma_load_4d(st_addr + kHalfStage + gi * kBlkBytes, &tm_vt, fb, 0, kvh, b * N + 16 * gi, 0);
          }
        }
        __syncwarp();
      }
      ++j;
      cur.next();
    }
    if (!ok && lane == 0) {
      // give copies still in flight a bounded chance to land before exit
      int dummy = 0;
      for (int k = j > kStages ? j - kStages : 0; k < j; ++k)
        if ((k & 1) == par) wait_bar(smem_u32(&bars.kv_full[k % kStages]), (uint32_t)((k / kStages) & 1), &dummy);
      grid_dep_wait();
      set_status(p.status, cur.valid() ? cur.b : 0, TV_ERR_CUDA);
    }

  } else if (warp == 1) {
    // ======================================================== MMA issuer
    // The only warp that issues tcgen05.mma (one lane per instruction, chosen
    // by elect.sync).  The whole warp runs this loop with warp-uniform control
    // flow (barrier tests are votes), so operands stay warp-uniform.  It polls
    // for whichever MMA can go next, PV first (it releases a stage), then S,
    // so a late K/V tile never holds up a ready P V product.
    //   S_j  needs its K tile, Q of its segment, and S buffer j&1 read out by
    //        the softmax (s_free of tile j-2, signalled right after the softmax
    //        loaded S, so S of the next tile is ready before it is needed).
    //   PV_k needs P_k (p_full) and, for the first PV of a segment, the
    //        previous segment's O read out by the merge (o_free).
    {
      const uint32_t idesc_pv = make_idesc(kM, kD, true);
      // descriptors: start-address field = address >> 4, so byte offsets
      // (below 256 KB) are added as offset >> 4
      const uint64_t dk = sw128_desc(sbase + kOffKV, 16, 1024);
      const uint64_t dv = sw128_desc(sbase + kOffKV + kHalfStage, kBlkChunk, 1024);
      // S issued, PV not yet: at most kStages tiles (S_j waits for the stage
      // PV_{j-kStages} released).  Packed: blocks | seg_first << 3 |
      // acc_first << 4 | segment << 5, shifted out as PVs are issued.
      uint32_t pend[kStages];
#pragma unroll
      for (int i = 0; i < kStages; ++i) pend[i] = 0;
      bool ok = true;
      int js = 0, jp = 0, seg = 0;
      bool ostart0 = false, ostart1 = false;
      uint64_t t0 = 0;
      // running stage / phase of the next PV and the next S (no divisions)
      int st_p = 0, st_s = 0;
      uint32_t ph_p = 0, ph_s = 0;
      for (uint32_t spin = 0;; ++spin) {
        bool progressed = false;
        // all barrier probes first (independent shared-memory reads), then
        // one vote per candidate MMA
        const uint32_t mt = pend[0];
        const int m_seg = (int)(mt >> 5);
        const bool need_o = ((mt >> 3) & 1) && m_seg > 0;
        const bool s_first = cur.valid() && cur.seg_start(lo);
        const bool t_p = mbar_test_wait(smem_u32(&bars.p_full[jp & 1]), (uint32_t)((jp >> 1) & 1));
        const bool t_o = mbar_test_wait(smem_u32(&bars.o_free), (uint32_t)((m_seg - 1) & 1));
        const bool t_f = mbar_test_wait(smem_u32(&bars.s_free[js & 1]), (uint32_t)(((js - 2) >> 1) & 1));
        const bool t_q = mbar_test_wait(smem_u32(&bars.q_full), (uint32_t)(seg & 1));
        const bool t_k = mbar_test_wait(smem_u32(&bars.kv_full[st_s]), ph_s);
        const bool go_pv = __all_sync(0xffffffffu, (jp < js) & t_p & (t_o | !need_o));
        const bool go_s = __all_sync(0xffffffffu, cur.valid() & (t_f | (js < 2)) & (t_q | !s_first) & t_k);
        if (go_pv) {
          tc_fence_after();
          const int x = jp & 1;
          const uint32_t nblk = mt & 7;
          const bool acc_first = (mt >> 4) & 1;
          const uint32_t ap = tmem + kColP + (uint32_t)x * 32;
          const uint64_t bv = dv + (uint64_t)((st_p * kStageBytes) >> 4);
          const uint32_t od = tmem + kColO + (uint32_t)x * kD;
          // 16 keys (one paged block) per instruction: A = P from TMEM (8
          // columns of bf16 pairs), V block i is [2 d halves][16 keys][64 d],
          // halves kBlkChunk apart (LBO), 8-key groups 1024 B apart (SBO)
          if (nblk == 4) {
            umma_pv4_warp(od, ap, bv, kBlkBytes >> 4, idesc_pv, acc_first ? 0u : 1u,
                          smem_u32(&bars.pv_done[x]), smem_u32(&bars.kv_empty[st_p]));
          } else {
            for (uint32_t i = 0; i < nblk; ++i)
              umma_f16_ta_warp(od, ap + 8 * i, bv + i * (kBlkBytes >> 4), idesc_pv,
                               (i > 0 || !acc_first) ? 1u : 0u);
            umma_commit_warp(smem_u32(&bars.pv_done[x]));
            umma_commit_warp(smem_u32(&bars.kv_empty[st_p]));
          }
#pragma unroll
          for (int i = 0; i + 1 < kStages; ++i) pend[i] = pend[i + 1];
          ++jp;
          if (++st_p == kStages) {
            st_p = 0;
            ph_p ^= 1;
          }
          progressed = true;
        }
        if (go_s) {
          tc_fence_after();
          if (s_first) {
            ++seg;
            ostart0 = ostart1 = false;
          }
          const int keys = cur.u == cur.tiles - 1 ? NP : kBN;
          const uint32_t idesc_s = make_idesc(kM, keys, false);
          const uint64_t bk = dk + (uint64_t)((st_s * kStageBytes) >> 4);
          const uint32_t sc = tmem + (uint32_t)(js & 1) * kBN;
          // A = Q from TMEM (bf16 pairs, 8 columns per 16 dims); K is
          // [2 d halves][keys][64], 128-byte swizzled
          umma_s_tile_warp(sc, tmem + kColQ, bk, kKVChunk >> 4, idesc_s, smem_u32(&bars.s_full[js & 1]));
          if (cur.seg_end()) umma_commit_warp(smem_u32(&bars.q_empty));
          const bool par = js & 1;
          const bool acc_first = par ? !ostart1 : !ostart0;
          if (par) ostart1 = true;
          else ostart0 = true;
          const uint32_t nmt = (uint32_t)(keys >> 4) | ((uint32_t)s_first << 3) |
                               ((uint32_t)acc_first << 4) | ((uint32_t)(seg - 1) << 5);
#pragma unroll
          for (int i = 0; i < kStages; ++i)
            if (i == js - jp) pend[i] = nmt;
          ++js;
          if (++st_s == kStages) {
            st_s = 0;
            ph_s ^= 1;
          }
          cur.next();
          progressed = true;
        }
        if (!cur.valid() && jp == js) break;
        if (progressed) {
          t0 = 0;
        } else if ((spin & 63) == 63) {
          const uint64_t now = globaltimer();
          if (t0 == 0) t0 = now;
          const bool give_up = __any_sync(0xffffffffu, *abort_flag != 0 || now - t0 > kWaitNs);
          if (give_up) {
            if (lane == 0) *abort_flag = 1;
            ok = false;
            break;
          }
        }
      }
      // every MMA issued so far has completed once this arrives
      umma_commit_warp(smem_u32(&bars.fin));
      int dummy = 0;
      wait_bar(smem_u32(&bars.fin), 0, &dummy);
      if (!ok && lane == 0) {
        grid_dep_wait();
        set_status(p.status, cur.valid() ? cur.b : 0, TV_ERR_CUDA);
      }
    }
  } else {
    // ======================================================== softmax / epilogue
    // Masks and positions come from the ancestor kernel, and the scratch may
    // still be read by the previous launch's combine grid: wait for them here
    // (the producers and the MMA warp meanwhile fill the K/V stages).  A wait
    // inside the tile loop instead measurably slowed the loop's code.
    grid_dep_wait();
    // Two warpgroups take alternate tiles (x = parity of the CTA-wide tile
    // counter), each with its own running max / sum and its own O accumulator
    // in TMEM; at the end of a (sequence, KV head) segment warpgroup 0 merges
    // the two.  Thread (warp, lane) owns row 32*(warp%4) + lane == its TMEM lane.
    const int x = (warp - 2) >> 2;                    // warpgroup 0 or 1
    const int quad = warp & 3;
    const int m = quad * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t t_s = tlane + (uint32_t)x * kBN;
    const uint32_t t_o = tlane + kColO + (uint32_t)x * kD;
    const bool row_ok = m < R;
    const int t = row_ok ? m / G : 0;
    const int g = row_ok ? m - t * G : 0;
    const float qscale = p.qscale;
    const int wl = p.window_left;
    long long j = 0, last_j = -1;
    int seg = 0;
    bool ok = true;
    float m_used = -INFINITY, l = 0.f;
    int ctx = 0, blk_lo = 0, pos_t = 0;
    unsigned long long allowed = 0;
    long long seg_f0 = lo;
    bool seg_complete = false;
    bool q_next_loaded = false;  // Q of the coming segment already in TMEM
    // the pair this CTA starts and that runs past its range (merged by the
    // combine grid): its first flat tile, end tile and index b * Hkv + kvh
    long long own_s = -1, own_e = 0;
    int own_pair = 0;
    const uint32_t t_p = tlane + kColP + (uint32_t)x * 32;
    const uint32_t stg = sbase + kOffEpi + (uint32_t)(warp - 2) * 2048u;  // this warp's staging
    while (cur.valid()) {
      const int b = cur.b, kvh = cur.kvh;
      if (cur.seg_start(lo)) {
        m_used = -INFINITY;
        l = 0.f;
        last_j = -1;
        ctx = s_ctx[b];
        blk_lo = first_visible_block(ctx, wl);
        seg_f0 = cur.f;
        seg_complete = cur.u == 0 && cur.f + (cur.tiles - 1) <= hi - 1;
        if (x == 0 && !q_next_loaded) {
          // Q rows of this (sequence, KV head) into TMEM once the previous
          // segment's last S has read the old ones; rows past R are zero
          if (seg > 0) {
            ok = __all_sync(0xffffffffu,
                            wait_fast(smem_u32(&bars.q_empty), (uint32_t)((seg - 1) & 1), abort_flag));
            if (!ok) break;
          }
          uint32_t qr[2][32];
          const uint4 *src = reinterpret_cast<const uint4 *>(
              p.q + (((size_t)b * N + t) * p.Hq + kvh * G + g) * kD);
          const bool q_ok = row_ok && TV_CHECK(b < B && t < N && kvh * G + g < p.Hq);
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            const uint4 w = q_ok ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
            qr[v >> 3][(v & 7) * 4 + 0] = w.x;
            qr[v >> 3][(v & 7) * 4 + 1] = w.y;
            qr[v >> 3][(v & 7) * 4 + 2] = w.z;
            qr[v >> 3][(v & 7) * 4 + 3] = w.w;
          }
          tmem_st32(tlane + kColQ, qr[0]);
          tmem_st32(tlane + kColQ + 32, qr[1]);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.q_full));
        }
        q_next_loaded = false;
        allowed = 0;
        if (row_ok && TV_CHECK(b < B && t < N)) {
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
      if ((int)(j & 1) == x) {
        // every wait is made warp-uniform: the tcgen05.ld/st that follow are
        // warp-collective
        ok = __all_sync(0xffffffffu,
                        wait_fast(smem_u32(&bars.s_full[x]), (uint32_t)((j >> 1) & 1), abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[2][32];
        tmem_ld32(t_s, sr[0]);
        tmem_ld32(t_s + 32, sr[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.s_free[x]));  // the S buffer may be refilled
        const bool node = cur.u == cur.tiles - 1;
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
          const int kb = (blk_lo + 4 * cur.u) * kBlock;
          const int c0 = wl >= 0 ? pos_t - wl - kb : 0;
          const int c1 = ctx - kb;
          if (c0 > 0 || c1 < 64) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c < c0 || c >= c1) s[c] = -INFINITY;
          }
        }
        float mt[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          mt[i] = fmaxf(fmaxf(s[i], s[i + 16]), fmaxf(s[i + 32], s[i + 48]));
#pragma unroll
        for (int w = 8; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) mt[i] = fmaxf(mt[i], mt[i + w]);
        const float mxs = mt[0] * qscale;
        const bool need = m_used != -INFINITY && mxs > m_used + kTau;
        // the factor for O and l, and the new running max (raised to this
        // tile's max when the old one is too low by 2^kTau, or set by the
        // first tile); a running max of -inf means every score so far is
        // -inf: 2^(-inf) = 0
        const float alpha = need ? ex2(m_used - mxs) : 1.f;
        const float m_new = (need || m_used == -INFINITY) ? mxs : m_used;
        const float neg_m = m_new != -INFINITY ? -m_new : 0.f;
        // P_j and its row sum need only the new max: they are formed while
        // PV_{j-2} may still run
        float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = ex2(fmaf(s[c], qscale, neg_m));
          const float p1 = ex2(fmaf(s[c + 1], qscale, neg_m));
          ps[(c >> 1) & 7] += p0 + p1;
          pk[c >> 1] = pack_bf16(p0, p1);
        }
        if (j >= 2) {
          // PV_{j-2} done: P buffer x is free and O_x is quiescent
          ok = __all_sync(0xffffffffu, wait_fast(smem_u32(&bars.pv_done[x]),
                                                 (uint32_t)(((j - 2) >> 1) & 1), abort_flag));
          if (!ok) break;
        }
        // Rescale this warpgroup's O only when some row's max grew by more than
        // 2^kTau; decided per warp (tcgen05.ld/st are warp-collective), rows
        // that do not need it scale by 1.  A finite running max means this
        // warpgroup had an earlier tile in the segment: PV_{j-2} wrote O last.
        if (__any_sync(0xffffffffu, need)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(t_o + c * 32, o);
          }
          tmem_wait_st();
        }
        if (need) l *= alpha;
        m_used = m_new;
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        // P_j as bf16 pairs into this warpgroup's P columns of TMEM (the A
        // operand of the P V product): key 2c in the low half of column c
        tmem_st32(t_p, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[x]));  // the MMA thread issues O_x += P_j V_j
        last_j = j;
      }
      if (cur.seg_end()) {
        // this warpgroup's last PV of the segment must have landed in O_x
        if (last_j >= 0) {
          ok = __all_sync(0xffffffffu, wait_fast(smem_u32(&bars.pv_done[x]),
                                                 (uint32_t)((last_j >> 1) & 1), abort_flag));
          if (!ok) break;
        }
        // is there a next segment in this CTA's range (then warpgroup 1 loads
        // its Q rows into TMEM now, before the merge, so that the next
        // segment's first S does not wait for the merge)
        const bool q_next = cur.f + 1 < hi && cur.b + (cur.kvh + 1 == p.Hkv ? 1 : 0) < B;
        q_next_loaded = q_next;
        // both warpgroups hand over (running max, running sum) ...
        float2 *mrg = reinterpret_cast<float2 *>(smem + kOffMerge) + (seg & 1) * 2 * kM;
        mrg[x * kM + m] = make_float2(m_used, l);
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.merge));
        if (x == 1 && q_next) {
          // once this segment's last S has read the old Q rows (q_empty)
          const int nb = cur.kvh + 1 < p.Hkv ? cur.b : cur.b + 1;
          const int nk = cur.kvh + 1 < p.Hkv ? cur.kvh + 1 : 0;
          const uint4 *src = reinterpret_cast<const uint4 *>(
              p.q + (((size_t)nb * N + t) * p.Hq + nk * G + g) * kD);
          ok = __all_sync(0xffffffffu,
                          wait_fast(smem_u32(&bars.q_empty), (uint32_t)(seg & 1), abort_flag));
          if (!ok) break;
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {  // 64 dims at a time
            uint32_t qn[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const uint4 w = row_ok ? __ldg(src + 8 * hf + v) : make_uint4(0, 0, 0, 0);
              qn[v * 4 + 0] = w.x;
              qn[v * 4 + 1] = w.y;
              qn[v * 4 + 2] = w.z;
              qn[v * 4 + 3] = w.w;
            }
            tmem_st32(tlane + kColQ + 32 * hf, qn);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&bars.q_full));
        }
        // ... then each merges its share of the 32-column chunks of O_0 and
        // O_1: warpgroup 0 chunks 0-2, warpgroup 1 (which loaded Q) chunk 3
        ok = __all_sync(0xffffffffu,
                        wait_fast(smem_u32(&bars.merge), (uint32_t)(seg & 1), abort_flag));
        if (!ok) break;
        tc_fence_after();
        const float2 h0 = mrg[m], h1 = mrg[kM + m];
        const float M = fmaxf(h0.x, h1.x);
        const float w0 = h0.x == -INFINITY ? 0.f : ex2(h0.x - M);
        const float w1 = h1.x == -INFINITY ? 0.f : ex2(h1.x - M);
        const float L = h0.y * w0 + h1.y * w1;
        const uint32_t t_o0 = tlane + kColO, t_o1 = tlane + kColO + kD;
        const int c_lo = x == 0 ? 0 : 3, c_hi = x == 0 ? 3 : 4;
        if (seg_complete) {
          const float inv = L > 0.f ? 1.f / L : 0.f;
          const float a0 = w0 * inv, a1 = w1 * inv;
          const size_t row_base = ((size_t)b * N * p.Hq + (size_t)kvh * G) * kD;
#pragma unroll 1
          for (int c = c_lo; c < c_hi; ++c) {
            uint32_t o0[32], o1[32];
            tmem_ld32(t_o0 + c * 32, o0);
            tmem_ld32(t_o1 + c * 32, o1);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float f0 = (w0 > 0.f ? __uint_as_float(o0[e]) * a0 : 0.f) +
                               (w1 > 0.f ? __uint_as_float(o1[e]) * a1 : 0.f);
              const float f1 = (w0 > 0.f ? __uint_as_float(o0[e + 1]) * a0 : 0.f) +
                               (w1 > 0.f ? __uint_as_float(o1[e + 1]) * a1 : 0.f);
              pk[e >> 1] = pack_bf16(f0, f1);
            }
            stage_store_bf16(stg, pk, lane, quad, p.out, row_base, p.Hq, G, R, c * 32);
          }
        } else {
          const int slot = 2 * (int)blockIdx.x + (seg_f0 == lo ? 0 : 1);
          float *dst = tp.part_o + (size_t)slot * kD * kM + m;  // dim-major: dim d at d * 128
#pragma unroll 1
          for (int c = c_lo; c < c_hi && TV_CHECK(slot < 2 * (int)gridDim.x); ++c) {
            uint32_t o0[32], o1[32];
            tmem_ld32(t_o0 + c * 32, o0);
            tmem_ld32(t_o1 + c * 32, o1);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              dst[(size_t)(c * 32 + e) * kM] = (w0 > 0.f ? __uint_as_float(o0[e]) * w0 : 0.f) +
                                               (w1 > 0.f ? __uint_as_float(o1[e]) * w1 : 0.f);
          }
          if (x == 0 && TV_CHECK(slot < 2 * (int)gridDim.x)) tp.part_ml[(size_t)slot * kM + m] = make_float2(M, L);
          if (seg_f0 == cur.f - cur.u) {  // the piece holds the pair's first tile
            own_s = seg_f0;
            own_e = seg_f0 + cur.tiles;
            own_pair = b * p.Hkv + kvh;
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.o_free));  // O_0 and O_1 may be overwritten
        ++seg;
      }
      ++j;
      cur.next();
    }
    // every CTA writes its range start and descriptor (the workspace is not
    // cleared between calls); the combine grid reads them once this grid has
    // completed
    if (warp == 2 && lane == 0) {
      tp.lo_out[blockIdx.x] = lo;
      if (blockIdx.x + 1 == gridDim.x) tp.lo_out[gridDim.x] = hi;
      tp.desc[blockIdx.x] = make_longlong2(own_s, own_s < 0 ? 0 : (own_e | ((long long)own_pair << 32)));
    }
    if (!ok && lane == 0) set_status(p.status, cur.valid() ? cur.b : 0, TV_ERR_CUDA);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  } else if (warp == 0) {
    // the data errors every warp of this CTA found, once the ancestor kernel
    // has initialised the status words
    grid_dep_wait();
    for (int i = lane; i < (B + 31) / 32; i += 32) {
      uint32_t bits = s_bad[i];
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        set_status(p.status, 32 * i + bit, TV_ERR_BLOCK);
      }
    }
  }
}

// Merge the partials of the pairs cut between CTAs.  Block (c, y) takes the
// pair CTA c starts and that runs past its range (CTA c's descriptor; most
// blocks find none and exit) and its dims 64y .. 64y+63: thread i owns row
// i % 128 and 32 dims.  The pieces are in CTAs c, c+1, ... up to the one whose
// range holds the pair's last tile; slot 2d (a piece that starts a CTA's
// range) or 2c + 1 (CTA c's piece, when the pair starts inside its range).
// The range starts are read 32 CTAs at a time; the (max, sum) and data of up
// to kCombBatch pieces are loaded together, then merged in piece order.
// Launched as a programmatic dependent of the attention grid: it waits for
// that grid's completion before any read.
constexpr int kCombBatch = 2;

__global__ void __launch_bounds__(256) attn_tc_combine_kernel(const TcParams tp, int P) {
  // the next attention launch may start now: it waits for this grid before it
  // touches the scratch read here
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  grid_dep_wait();
  const AttnParams &p = tp.a;
  const int c = blockIdx.x;
  const longlong2 dsc = tp.desc[c];
  if (dsc.x < 0) return;
  const long long S = dsc.x, E = dsc.y & 0xffffffffll;
  const int pair = (int)(dsc.y >> 32);
  const int b = pair / p.Hkv, kvh = pair - b * p.Hkv;
  __shared__ long long s_lo[33];
  __shared__ int s_slot[32];
  __shared__ int s_n;
  const int m = threadIdx.x & 127, d0 = 64 * blockIdx.y + 32 * (threadIdx.x >> 7);
  float Mx = -INFINITY, Lx = 0.f, acc[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) acc[k] = 0.f;
  // windows of 32 CTAs: their range starts, the pieces they hold, then the
  // pieces' partials kCombBatch at a time
  for (int w0 = c; w0 < P; w0 += 32) {
    __syncthreads();
    if (threadIdx.x < 33) s_lo[threadIdx.x] = w0 + (int)threadIdx.x <= P ? tp.lo_out[w0 + threadIdx.x] : E;
    __syncthreads();
    if (threadIdx.x == 0) {
      int n = 0;
      for (int i = 0; i < 32 && w0 + i < P; ++i) {
        const int d = w0 + i;
        const long long ld = s_lo[i], hd = s_lo[i + 1];
        if (ld >= E) {
          n = -1 - n;  // the pair ends in this window
          break;
        }
        if (ld == hd) continue;  // an empty range holds no piece
        s_slot[n++] = 2 * d + ((d == c && ld < S) ? 1 : 0);
      }
      s_n = n;
    }
    __syncthreads();
    const int nraw = s_n;
    const bool done = nraw < 0;
    const int n = done ? -1 - nraw : nraw;
    for (int i0 = 0; i0 < n; i0 += kCombBatch) {
      float2 ml[kCombBatch];
      float o[kCombBatch][32];
#pragma unroll
      for (int i = 0; i < kCombBatch; ++i) {
        ml[i] = make_float2(-INFINITY, 0.f);
        if (i0 + i < n && TV_CHECK(s_slot[i0 + i] < 2 * P && d0 + 32 <= kD)) {
          const int slot = s_slot[i0 + i];
          ml[i] = __ldcg(tp.part_ml + (size_t)slot * kM + m);
          const float *src = tp.part_o + ((size_t)slot * kD + d0) * kM + m;
#pragma unroll
          for (int k = 0; k < 32; ++k) o[i][k] = __ldcg(src + (size_t)k * kM);
        }
      }
#pragma unroll
      for (int i = 0; i < kCombBatch; ++i) {
        if (ml[i].x == -INFINITY) continue;  // no piece, or no key seen: O = 0
        const float Mn = fmaxf(Mx, ml[i].x);
        const float a = Mx == -INFINITY ? 0.f : exp2f(Mx - Mn), w = exp2f(ml[i].x - Mn);
        Lx = Lx * a + ml[i].y * w;
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] = acc[k] * a + o[i][k] * w;
        Mx = Mn;
      }
    }
    if (done) break;
  }
  if (m >= p.R) return;
  const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
  const int t = m / p.G, g = m - t * p.G;
  __nv_bfloat16 *dst = p.out + (((size_t)b * p.N + t) * p.Hq + kvh * p.G + g) * kD + d0;
#pragma unroll
  for (int e = 0; e < 32; e += 8) {
    uint4 v;
    v.x = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    v.y = pack_bf16(acc[e + 2] * inv, acc[e + 3] * inv);
    v.z = pack_bf16(acc[e + 4] * inv, acc[e + 5] * inv);
    v.w = pack_bf16(acc[e + 6] * inv, acc[e + 7] * inv);
    *reinterpret_cast<uint4 *>(dst + e) = v;
  }
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
  const uint32_t estr[4] = {1, 1, 1, 1};
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
  (void)B;
  const size_t lo = ((size_t)(P + 1) * sizeof(long long) + 255) / 256 * 256;
  const size_t desc = ((size_t)P * sizeof(longlong2) + 255) / 256 * 256;
  const size_t ml = ((size_t)2 * P * kM * sizeof(float2) + 255) / 256 * 256;
  const size_t o = (size_t)2 * P * kM * kD * sizeof(float);
  return lo + desc + ml + o;
}

cudaError_t launch_attention_tc(const AttnParams &a, void *workspace, cudaStream_t stream) {
  const int P = a.ctas > 0 && a.ctas < sm_count() ? a.ctas : sm_count();
  TcParams tp{};
  tp.a = a;
  char *ws = static_cast<char *>(workspace);
  tp.lo_out = reinterpret_cast<long long *>(ws);
  ws += ((size_t)(P + 1) * sizeof(long long) + 255) / 256 * 256;
  tp.desc = reinterpret_cast<longlong2 *>(ws);
  ws += ((size_t)P * sizeof(longlong2) + 255) / 256 * 256;
  tp.part_ml = reinterpret_cast<float2 *>(ws);
  ws += ((size_t)2 * P * kM * sizeof(float2) + 255) / 256 * 256;
  tp.part_o = reinterpret_cast<float *>(ws);
  tp.node_pad = (a.N + 15) / 16 * 16;

  CUtensorMap mkc, mvc, mkcr, mvcr, mkt, mvt;
  const uint64_t row_bytes = kD * 2;
  {
    // cache rows (block, head, token) of 128 d, viewed as [d half][row][64]:
    // one copy moves a whole 16-token block as [2][16][64]
    const uint64_t rows = (uint64_t)(a.num_blocks > 0 ? a.num_blocks : 1) * a.Hkv * kBlock;
    const uint64_t dims3[3] = {64, rows, 2};
    const uint64_t str3[2] = {row_bytes, 128};
    const uint32_t box3[3] = {64, (uint32_t)kBlock, 2};
    const uint64_t dims2[2] = {(uint64_t)kD, rows};
    const uint64_t str2[1] = {row_bytes};
    const uint32_t box16[2] = {64, (uint32_t)kBlock};
    const uint32_t box1[2] = {64, 1};
    if (!make_map(&mkc, a.k_cache, 2, dims2, str2, box16) ||
        !make_map(&mvc, a.v_cache, 3, dims3, str3, box3) ||
        !make_map(&mkcr, a.k_cache, 2, dims2, str2, box1) ||
        !make_map(&mvcr, a.v_cache, 2, dims2, str2, box1))
      return cudaErrorInvalidValue;
  }
  {
    // tree K [B*N][Hkv][128]: 16 consecutive nodes of one head, one d half;
    // tree V viewed as [d half][node][head][64]: 16 nodes as [2][16][64]
    const uint64_t dimsk[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.B * a.N};
    const uint64_t strk[2] = {row_bytes, row_bytes * a.Hkv};
    const uint32_t boxk[3] = {64, 1, 16};
    const uint64_t dims[4] = {64, (uint64_t)a.Hkv, (uint64_t)a.B * a.N, 2};
    const uint64_t str[3] = {row_bytes, row_bytes * a.Hkv, 128};
    const uint32_t box[4] = {64, 1, 16, 2};
    if (!make_map(&mkt, a.k_tree, 3, dimsk, strk, boxk) || !make_map(&mvt, a.v_tree, 4, dims, str, box))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // both grids are programmatic dependents of the kernel before them on the
  // stream: each may start while it finishes, and waits for it
  // (griddepcontrol.wait) before touching what it may write
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel, mkc, mvc, mkcr, mvcr, mkt, mvt, tp);
  if (e != cudaSuccess) return e;
  if (P > 1) {
    cfg.gridDim = dim3(P, 2);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, attn_tc_combine_kernel, tp, (int)P);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace tv
