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

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the kernel before it in the
// stream is still running; pdl_wait() blocks until that kernel has completed
// and its writes are visible (a no-op without the attribute).  The earlier
// kernel lets it start early with pdl_launch_dependents().
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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

// The base window of the query at absolute position q, before the image union
// and the clamp to the sequence.  Left edge: q-W+1, or with chunked lookback
// (lookback L >= 0, chunk size C, only with W > 0) the start of the chunk L
// chunks before q's, ((q / C) - L) * C; 0 without a window.  Right edge: q
// (causal), q+W-1 (non-causal), the sequence end without a window.  Edges are
// clamped to [0, seq_len - 1] in 64-bit arithmetic, so no window or lookback
// overflows.
__device__ inline int base_lo(int q, int window, int chunk_size, int chunk_lookback) {
  if (window <= 0) return 0;
  int64_t lo = chunk_lookback >= 0 ? ((int64_t)(q / chunk_size) - chunk_lookback) * chunk_size
                                   : (int64_t)q - window + 1;
  return lo < 0 ? 0 : (int)lo;
}
__device__ inline int base_hi(int q, int window, bool causal, int seq_len) {
  if (causal) return q;
  if (window <= 0) return seq_len - 1;
  return (int)min((int64_t)q + window - 1, (int64_t)seq_len - 1);
}

// Visible keys of the query at absolute position q form one interval:
//   lo = max(0, min(base_lo(q), min{max(s, q-W+1) : valid range [s,e] holds q}))
//   hi = min(seq_len-1, max(base_hi(q), max{e : valid range [s,e] holds q}))
// (the image terms' left edge only with W > 0).  The base window and every
// range holding q contain q itself, so their union has no gap: the image mask
// keeps the ordinary window clamp even where the chunk start is later, and so
// reaches keys before the chunk.  Returns lo > hi when nothing is visible.
// `ranges` may point to global or shared memory (plain generic loads).
struct Span { int lo, hi; };

__device__ inline Span visible_span(int q, int seq_len, int window, bool causal, int chunk_size,
                                    int chunk_lookback, const int32_t *ranges, int num_ranges) {
  Span sp;
  sp.lo = base_lo(q, window, chunk_size, chunk_lookback);
  sp.hi = base_hi(q, window, causal, seq_len);
  const int clamp = window > 0 ? q - window + 1 : INT_MIN;
  for (int i = 0; i < num_ranges; ++i) {
    const int s = ranges[2 * i], e = ranges[2 * i + 1];
    if (s < e && s <= q && q <= e) {
      sp.hi = max(sp.hi, e);
      sp.lo = min(sp.lo, max(s, clamp));
    }
  }
  sp.lo = max(sp.lo, 0);
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
