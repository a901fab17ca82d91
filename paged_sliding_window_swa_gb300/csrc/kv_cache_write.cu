// A step's new K/V rows -> the paged KV cache, by slot id (vllm-ascend
// slot-mapping article, section 1 and its closing summary: the cache-write and
// attention operators consume the slot ids).
//
// A token's row (num_heads_kv x head_dim elements) is contiguous both in the
// new tensors [T, Hkv, D] and in the slot-major cache [num_slots, Hkv, D], so
// the scatter is a copy of whole rows: one warp per token, every lane moving
// 16-byte vectors of the K row and then of the V row, all loads of a lane in
// flight before its stores.
#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr int kWarps = 8;
constexpr int kInFlight = 4;                    // 16-byte vectors per lane per batch

__global__ void __launch_bounds__(kWarps * 32)
kv_cache_write_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                      const int32_t *__restrict__ slots, int64_t num_tokens, int64_t row_vecs,
                      uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int64_t num_slots,
                      int32_t *__restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  for (int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); t < num_tokens; t += warps) {
    const int32_t slot = __ldg(slots + t);
    if (slot < 0) continue;                     // padding token
    if (slot >= num_slots) {
      if (lane == 0) report(err, SWA_ERR_SLOT);
      continue;
    }
    const uint4 *srcs[2] = {k_new + t * row_vecs, v_new + t * row_vecs};
    uint4 *dsts[2] = {k_cache + (int64_t)slot * row_vecs, v_cache + (int64_t)slot * row_vecs};
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      for (int64_t base = 0; base < row_vecs; base += 32 * kInFlight) {
        uint4 v[kInFlight];
#pragma unroll
        for (int i = 0; i < kInFlight; ++i) {
          const int64_t j = base + i * 32 + lane;
          if (j < row_vecs) v[i] = __ldcs(srcs[kv] + j);
        }
#pragma unroll
        for (int i = 0; i < kInFlight; ++i) {
          const int64_t j = base + i * 32 + lane;
          if (j < row_vecs) dsts[kv][j] = v[i];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_cache_write(const void *k_new, const void *v_new, const int32_t *slots,
                                  int64_t num_tokens, int64_t row_bytes, void *k_cache, void *v_cache,
                                  int64_t num_slots, int32_t *err, cudaStream_t st) {
  if (num_tokens == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  // enough warps to keep every SM's load queue full; tokens are walked grid-stride
  const int64_t blocks = min(ceil_div(num_tokens, kWarps), (int64_t)sms * 8);
  kv_cache_write_kernel<<<(unsigned)blocks, kWarps * 32, 0, st>>>(
      static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slots, num_tokens, row_bytes / 16,
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), num_slots, err);
  return cudaGetLastError();
}

}  // namespace swa
