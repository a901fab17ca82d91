// Device helpers shared by the kernels of the library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "swa.h"

namespace swa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

__device__ inline void report(int32_t *err, int32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

// Nanosecond clock shared by all SMs; used to bound every spin-wait.
__device__ inline uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ inline float to_f(float x) { return x; }
  static __device__ inline float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ inline float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ inline __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Query blocks: sequence s owns the block indices
//   [qsl[s] / bq + s, qsl[s+1] / bq + s + 1),
// which is at least ceil(query_len / bq) indices, so a grid of
// num_tokens / bq + num_seqs blocks covers every sequence without a host-side
// scan.  Returns the sequence of `block` (largest s whose first index <= block).
__device__ inline int find_seq(const int32_t *qsl, int num_seqs, int64_t block, int bq) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((int64_t)__ldg(qsl + mid) / bq + mid <= block) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Visible keys of the query at absolute position q form one interval:
// [max(0, q-W+1), min(seq_len-1, max(right(q), max{e : valid range [s,e] holds q}))]
// (right(q) = q causal, q+W-1 non-causal; with W <= 0 the left edge is 0 and a
// non-causal right edge is the sequence end).  Every range holding q starts at
// or before q, so its clamped part [max(s, q-W+1), e] joins the base window
// without a gap.  Returns lo > hi when nothing is visible.  `ranges` may point
// to global or shared memory (plain generic loads).
struct Span { int lo, hi; };

__device__ inline Span visible_span(int q, int seq_len, int window, bool causal,
                                    const int32_t *ranges, int num_ranges) {
  Span sp;
  if (window > 0) {
    sp.lo = max(0, q - window + 1);
    sp.hi = causal ? q : q + window - 1;
  } else {
    sp.lo = 0;
    sp.hi = causal ? q : seq_len - 1;
  }
  for (int i = 0; i < num_ranges; ++i) {
    const int s = ranges[2 * i], e = ranges[2 * i + 1];
    if (s < e && s <= q && q <= e) sp.hi = max(sp.hi, e);
  }
  sp.hi = min(sp.hi, seq_len - 1);
  return sp;
}

// Split-KV partition of a sequence: keys [p*L, min((p+1)*L, seq_len)),
// L = SWA_SPLIT_ALIGN * ceil(ceil(seq_len / parts) / SWA_SPLIT_ALIGN).
__device__ inline Span split_span(int seq_len, int parts, int p) {
  int per = (int)ceil_div(seq_len, parts);
  int len = (int)ceil_div(per, SWA_SPLIT_ALIGN) * SWA_SPLIT_ALIGN;
  Span sp;
  sp.lo = min(p * len, seq_len);
  sp.hi = min((p + 1) * len, seq_len) - 1;
  return sp;
}

__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace swa
