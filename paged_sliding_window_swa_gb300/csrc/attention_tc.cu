// tcgen05 prefill attention (placeholder until the tensor-core kernel lands).
#include "common.cuh"
#include "launch.h"

namespace swa {

bool tc_supported(const AttnArgs &) { return false; }
cudaError_t launch_attention_tc(const AttnArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace swa
