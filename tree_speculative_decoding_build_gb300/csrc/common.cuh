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

// Programmatic dependent launch.  A kernel launched by launch_pdl may be
// scheduled while the grid before it on the stream is still running, once
// that grid's blocks have all executed pdl_launch_dependents (or exited); it
// must call pdl_wait before it reads anything that grid (or any earlier work)
// writes.  pdl_wait returns at once when the kernel was launched normally.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Index checks of the TV_DEBUG build (a stand-in for a memory checker).
// TV_CHECK(cond) guards one access: in a build with -DTV_DEBUG a false
// condition is recorded in this translation unit's fault record (the number
// of failed checks and the source line of the first) and the access is
// skipped; without TV_DEBUG it is the constant true and the compiled code is
// that of the plain build.  Each .cu file that uses it names its record once
// with TV_DEBUG_RECORD(name); tv_debug_check_failures() (tv_debug.h) reads
// them all.
#ifdef TV_DEBUG
#define TV_DEBUG_RECORD(name)                                                   \
  namespace tv {                                                                \
  static __device__ unsigned int g_check_record[2];                             \
  static __device__ __noinline__ bool check_failed(int line) {                  \
    if (atomicAdd(&g_check_record[0], 1u) == 0u) g_check_record[1] = (unsigned)line; \
    return false;                                                               \
  }                                                                             \
  unsigned debug_record_##name(unsigned *first_line, bool clear) {              \
    unsigned r[2] = {0u, 0u};                                                   \
    if (cudaMemcpyFromSymbol(r, g_check_record, sizeof(r)) != cudaSuccess) return ~0u; \
    if (clear) {                                                                \
      const unsigned z[2] = {0u, 0u};                                           \
      cudaMemcpyToSymbol(g_check_record, z, sizeof(z));                         \
    }                                                                           \
    if (first_line) *first_line = r[1];                                         \
    return r[0];                                                                \
  }                                                                             \
  }
#define TV_CHECK(cond) ((cond) || tv::check_failed(__LINE__))
#else
#define TV_DEBUG_RECORD(name)                                                   \
  namespace tv {                                                                \
  unsigned debug_record_##name(unsigned *first_line, bool) {                    \
    if (first_line) *first_line = 0u;                                           \
    return 0u;                                                                  \
  }                                                                             \
  }
#define TV_CHECK(cond) true
#endif

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
