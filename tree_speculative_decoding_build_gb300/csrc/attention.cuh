// Internal interface between the tree-attention entry point and its kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace tv {

// Everything a tree-attention kernel needs, resolved on the host.
//
// Rows: the G = Hq/Hkv query heads that share KV head kvh are packed with the
// N nodes into R = G*N rows, row r = t*G + g (node t, head kvh*G + g), so one
// pass over a KV tile serves every row of the group.
struct AttnParams {
  const __nv_bfloat16 *q, *k_tree, *v_tree, *k_cache, *v_cache;
  const int32_t *block_table, *ctx_len, *pos;
  const uint64_t *anc;
  int B, N, Hq, Hkv, G, R, D;
  int max_blocks, num_blocks;
  int window_left;       // -1 = global
  float qscale;          // sm_scale * log2(e): scores live in the base-2 domain
  int splits;            // context splits per (sequence, KV head)
  int bps;               // 16-token context blocks per split
  float *part_o;         // [B*Hkv][splits][R][D]  unnormalised partial outputs
  float2 *part_ml;       // [B*Hkv][splits][R]     (running max, running sum)
  __nv_bfloat16 *out;    // [B, N, Hq, D]
  int32_t *status;       // [B]
  int ctas;              // tensor-core kernel: persistent CTAs (0 = one per SM)
  int withheld_cta;      // test hook: CTA whose first K/V barrier expects an extra arrival (-1: none)
};

// First visible context block of a sequence: rows sit at positions
// >= ctx_len (depth >= 1), so the union of their windows starts at
// ctx_len - window_left.
__host__ __device__ inline int first_visible_block(int ctx, int window_left) {
  if (window_left < 0) return 0;
  int lo = ctx - window_left;
  return lo > 0 ? lo / TV_BLOCK_SIZE : 0;
}

// Context blocks a split grid must cover for any ctx_len <= max_blocks*16.
inline int visible_blocks_bound(int max_blocks, int window_left) {
  if (window_left < 0) return max_blocks;
  int w = (window_left + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE + 1;
  return w < max_blocks ? w : max_blocks;
}

// Merge split partials into the bf16 output (one warp per row).
void launch_combine(const AttnParams &p, cudaStream_t stream);

// CUDA-core kernel: any supported D and row count.
void launch_attention_generic(const AttnParams &p, cudaStream_t stream);

// Tensor-core (tcgen05) kernel for D = 128 and R <= 128 rows per KV head.
bool attention_tc_supported(const AttnParams &p);
// Scratch of the tensor-core kernel: schedule offsets and split partials.
size_t attention_tc_workspace(int B, int num_ctas);
// Launches the kernel (one CTA per SM) and its partial combine.
cudaError_t launch_attention_tc(const AttnParams &p, void *workspace, cudaStream_t stream);

// Tensor-core kernel for D = 256 and R <= 128: one CTA per (sequence, KV
// head, split) with the split plan's partials (merged by launch_combine).
bool attention_tc256_supported(const AttnParams &p);
cudaError_t launch_attention_tc256(const AttnParams &p, cudaStream_t stream);

}  // namespace tv
