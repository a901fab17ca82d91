// Token position -> physical KV-cache slot
// (vllm-ascend article on _compute_slot_mapping_kernel, sections 1-2).
//
// Token-flat grid: every thread maps 8 consecutive tokens, so positions are
// read as four 16-byte vectors and slots written as two, with streaming cache
// hints (each byte is touched once) that leave L1 to query_start_loc and the
// block table; the padded tail [num_tokens, max_num_tokens) is filled by the
// same threads.  A thread finds its request by binary search over
// query_start_loc once and walks forward.
// Neighbouring tokens share block-table entries, so each entry is fetched from
// DRAM once and served from L1/L2 afterwards -- the job of the page's bounded
// block-table window, without staging it by hand.
#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr int kTokPerThread = 8;
constexpr int kThreads = 256;

__device__ inline int find_req(const int32_t *qsl, int num_reqs, int64_t t) {
  // largest r in [0, num_reqs) with qsl[r] <= t
  int lo = 0, hi = num_reqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// kPow2: block_size == 1 << shift, the usual case -- a shift and a mask
// instead of a 64-bit division, which the GPU does in software.
template <bool kVec, bool kPow2>
__global__ void __launch_bounds__(kThreads)
slot_mapping_kernel(const int32_t *__restrict__ qsl, const int64_t *__restrict__ pos,
                    const int32_t *__restrict__ bt, int64_t stride, int32_t block_size, int32_t shift,
                    int32_t num_reqs, int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                    int32_t *__restrict__ out, int32_t *__restrict__ err) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // query_start_loc sanity: monotone, starts >= 0, ends <= num_tokens
  if (tid < num_reqs) {
    int32_t a = __ldg(qsl + tid), b = __ldg(qsl + tid + 1);
    if (a > b || a < 0 || b > num_tokens) report(err, SWA_ERR_QSL);
  }
  const int64_t t0 = tid * kTokPerThread;
  if (t0 >= max_num_tokens) return;

  int32_t res[kTokPerThread];
  if (t0 >= num_tokens || num_reqs == 0) {
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) res[i] = pad_id;
  } else {
    int64_t p[kTokPerThread];
    if (kVec && t0 + kTokPerThread <= num_tokens) {
      const longlong2 *src = reinterpret_cast<const longlong2 *>(pos + t0);
#pragma unroll
      for (int i = 0; i < kTokPerThread / 2; ++i) {
        const longlong2 a = __ldcs(src + i);
        p[2 * i] = a.x;
        p[2 * i + 1] = a.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kTokPerThread; ++i) p[i] = (t0 + i < num_tokens) ? __ldg(pos + t0 + i) : 0;
    }
    int r = find_req(qsl, num_reqs, t0);
    int32_t r_end = __ldg(qsl + r + 1);
    int64_t last = -1;                                       // (request, page) of the last lookup
    int32_t blk = 0;
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i) {
      const int64_t t = t0 + i;
      res[i] = pad_id;
      if (t >= num_tokens) continue;
      while (r + 1 < num_reqs && t >= r_end) { ++r; r_end = __ldg(qsl + r + 1); }
      if (t < __ldg(qsl + r) || t >= r_end) continue;        // outside every request
      const int64_t ps = p[i];
      const int64_t page = kPow2 ? (ps >> shift) : ps / block_size;
      if (ps < 0 || page >= stride) { report(err, SWA_ERR_POSITION); continue; }
      const int64_t idx = (int64_t)r * stride + page;
      if (idx != last) {                                     // neighbouring tokens mostly share a page
        blk = __ldg(bt + idx);
        last = idx;
      }
      const int64_t off = kPow2 ? (ps & (block_size - 1)) : ps - page * block_size;
      res[i] = (int32_t)((int64_t)blk * block_size + off);
    }
  }
  if (kVec && t0 + kTokPerThread <= max_num_tokens) {
    int4 *dst = reinterpret_cast<int4 *>(out + t0);
#pragma unroll
    for (int i = 0; i < kTokPerThread / 4; ++i)
      __stcs(dst + i, make_int4(res[4 * i], res[4 * i + 1], res[4 * i + 2], res[4 * i + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < kTokPerThread; ++i)
      if (t0 + i < max_num_tokens) out[t0 + i] = res[i];
  }
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t *qsl, const int64_t *pos, const int32_t *bt,
                                int64_t stride, int32_t block_size, int32_t num_reqs,
                                int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                                int32_t *out, int32_t *err, cudaStream_t st) {
  const int64_t work = max(ceil_div(max_num_tokens, kTokPerThread), (int64_t)num_reqs);
  if (work == 0) return cudaSuccess;
  const unsigned grid = (unsigned)ceil_div(work, kThreads);
  const bool vec = ((uintptr_t)pos % 16 == 0) && ((uintptr_t)out % 16 == 0);   // t0 is a multiple of 8
  int shift = 0;
  while (shift < 30 && (1 << shift) < block_size) ++shift;
  const bool pow2 = (1 << shift) == block_size;
  auto k = vec ? (pow2 ? slot_mapping_kernel<true, true> : slot_mapping_kernel<true, false>)
               : (pow2 ? slot_mapping_kernel<false, true> : slot_mapping_kernel<false, false>);
  k<<<grid, kThreads, 0, st>>>(qsl, pos, bt, stride, block_size, shift, num_reqs, num_tokens, max_num_tokens,
                               pad_id, out, err);
  return cudaGetLastError();
}

}  // namespace swa
