// Shared device/host helpers of libtv (CUDA, sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tv.h"

namespace tv {

constexpr int kBlock = TV_BLOCK_SIZE;
constexpr int kMaxNodes = TV_MAX_NODES;

// Record a data error for sequence b without overwriting an earlier one.
__device__ __forceinline__ void set_status(int32_t *status, int b, int code) {
  if (status) atomicCAS(status + b, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Host side: translate the last CUDA error into a status code.
inline tv_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

inline cudaStream_t as_stream(tv_stream s) { return reinterpret_cast<cudaStream_t>(s); }

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Test hook (tv_debug.h): the CTA, by linear index, whose first-copy barrier
// the tensor-core kernels set to expect one arrival more than it gets; -1
// (the default) for none.  Host state, read at every launch.
int debug_withheld_cta();

}  // namespace tv
