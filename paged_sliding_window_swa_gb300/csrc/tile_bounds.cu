// Per-query-block KV-tile loop range after sliding-window pruning with the
// window-clamped image union (vLLM PR #53147 summary, compute_tile_loop_bounds
// excerpt, with its chunked-lookback left edge and per-sequence causal right
// edge).
#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr int kWarpsPerBlock = 4;

// One warp per (sequence, query block): the lanes split the sequence's image
// ranges and the warp reduces the edges.  Each edge is clamped to the range it
// ends up in before the reduction (left edge >= 0, right edge <= seq_len - 1),
// which keeps it in 32 bits and leaves min/max unchanged after the clamp.
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
tile_bounds_kernel(const int32_t *__restrict__ qsl, const int32_t *__restrict__ seq_lens,
                   const int32_t *__restrict__ ctx_lens, const int32_t *__restrict__ mm, int32_t max_mm,
                   int32_t num_seqs, int32_t window, int32_t causal, int32_t per_seq_causal, int32_t chunk_size,
                   int32_t chunk_lookback, int32_t tile, int32_t bq, int32_t max_qblocks,
                   int32_t *__restrict__ out, int32_t *__restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.y;
  const int b = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (s >= num_seqs || b >= max_qblocks) return;             // uniform per warp
  int32_t *o = out + ((int64_t)s * max_qblocks + b) * 3;
  const int qlen = __ldg(qsl + s + 1) - __ldg(qsl + s);
  const int seq_len = __ldg(seq_lens + s);
  int ctx = seq_len - qlen;
  if (qlen < 0 || ctx < 0 || (ctx_lens != nullptr && __ldg(ctx_lens + s) != ctx)) {
    if (lane == 0) {
      if (b == 0) report(err, SWA_ERR_LENS);
      o[0] = o[1] = o[2] = 0;
    }
    return;
  }
  const int qpos_lo = b * bq;
  if (qpos_lo >= qlen) {
    if (lane == 0) o[0] = o[1] = o[2] = 0;
    return;
  }
  const int qpos_hi = min(qpos_lo + bq - 1, qlen - 1);
  const bool use_mm = (mm != nullptr) && (max_mm > 0);
  // the per-sequence causal mode is bounded as non-causal (the flags are not read here)
  const bool right_causal = causal && !per_seq_causal;
  const int q_lo = ctx + qpos_lo, q_hi = ctx + qpos_hi;
  const int max_prefix = (use_mm || !right_causal) ? seq_len : min(q_hi + 1, seq_len);
  const int num_tiles = (int)ceil_div(max_prefix, tile);
  int lo = 0, hi = num_tiles;
  if (window > 0) {
    // 64-bit edges: a large window or lookback reaches past the int range
    const int64_t first0 = chunk_lookback >= 0 ? ((int64_t)(q_lo / chunk_size) - chunk_lookback) * chunk_size
                                               : (int64_t)q_lo - window + 1;
    const int64_t last0 = right_causal ? (int64_t)q_hi : (int64_t)q_hi + window - 1;
    int first = (int)max(first0, (int64_t)0);                // in [0, q_lo]
    int last = (int)min(last0, (int64_t)seq_len - 1);        // in [q_hi, seq_len - 1]
    if (use_mm) {
      const int clamp_lo = (int)max((int64_t)q_lo - window + 1, (int64_t)0);
      const int32_t *r = mm + (int64_t)s * max_mm * 2;
      for (int i = lane; i < max_mm; i += 32) {
        const int rs = __ldg(r + 2 * i), re = __ldg(r + 2 * i + 1);
        if (rs < re && rs <= q_hi && re >= q_lo) {
          first = min(first, max(rs, clamp_lo));
          last = max(last, min(re, seq_len - 1));
        }
      }
      first = __reduce_min_sync(0xffffffffu, first);
      last = __reduce_max_sync(0xffffffffu, last);
    }
    lo = first / tile;
    hi = min(last / tile + 1, num_tiles);
  }
  if (lane == 0) {
    o[0] = lo;
    o[1] = hi;
    o[2] = max_prefix;
  }
}

}  // namespace

cudaError_t launch_tile_bounds(const int32_t *qsl, const int32_t *seq_lens, const int32_t *ctx,
                               const int32_t *mm, int32_t max_mm, int32_t num_seqs, int32_t window,
                               int32_t causal, int32_t per_seq_causal, int32_t chunk_size,
                               int32_t chunk_lookback, int32_t tile, int32_t bq, int32_t max_qblocks,
                               int32_t *out, int32_t *err, cudaStream_t st) {
  if (num_seqs == 0 || max_qblocks == 0) return cudaSuccess;
  dim3 grid((unsigned)ceil_div(max_qblocks, kWarpsPerBlock), (unsigned)num_seqs);
  tile_bounds_kernel<<<grid, 32 * kWarpsPerBlock, 0, st>>>(qsl, seq_lens, ctx, mm, max_mm, num_seqs, window, causal,
                                               per_seq_causal, chunk_size, chunk_lookback, tile, bq,
                                               max_qblocks, out, err);
  return cudaGetLastError();
}

}  // namespace swa
