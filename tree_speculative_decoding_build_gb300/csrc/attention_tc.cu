// Tensor-core tree attention (tcgen05); not yet available in this build.
#include "attention.cuh"

namespace tv {

bool attention_tc_supported(const AttnParams &) { return false; }

cudaError_t launch_attention_tc(const AttnParams &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tv
