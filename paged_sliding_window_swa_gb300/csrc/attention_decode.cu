// Split-KV decode attention (placeholder until the TMA-staged kernel lands).
#include "common.cuh"
#include "launch.h"

namespace swa {

bool decode_supported(const AttnArgs &) { return false; }
cudaError_t launch_attention_decode(const AttnArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace swa
