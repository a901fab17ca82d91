// Internal launchers behind the C ABI (host side).  Arguments are validated
// by the ABI layer before these are called.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace swa {

struct AttnArgs {
  const void *q, *k_cache, *v_cache;
  int64_t num_blocks;
  const int32_t *block_table;
  int64_t bt_stride;
  const int32_t *qsl, *seq_lens, *ctx_lens, *mm_ranges;
  int32_t max_mm_ranges, num_seqs;
  int64_t num_tokens;
  int32_t max_query_len, hq, hkv, head_dim, block_size, window, causal;
  const int32_t *seq_causal;            // per-sequence causal flags (replace `causal`) or null
  int32_t chunk_size, chunk_lookback;   // chunked lookback; chunk_lookback < 0: off
  float scale;
  int32_t dtype, num_splits;
  const int32_t *splits_per_seq;
  void *out;
  float *lse;
  void *partial_out;
  float *partial_lse;
  int32_t *err;
  uint64_t wait_ns;                     // bound of each pipeline wait in the tensor-core kernels
  int32_t stall;                        // watchdog test: the PV issuer waits on a barrier nothing signals
};

// Default bound of a pipeline wait: far above any real stall.
constexpr uint64_t kDefaultWaitNs = 200000000ull;

// Host-side checks of swa_mm_paged_attention.  Returns SWA_OK and fills `a`,
// or a negative SWA_E_* code; an empty call (no tokens or no sequences) passes
// with attention_is_empty(a).  Launches nothing.
int prepare_attention(const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
                      const int32_t *block_table, int64_t block_table_stride, const int32_t *query_start_loc,
                      const int32_t *seq_lens, const int32_t *context_lens, const int32_t *mm_ranges,
                      int32_t max_mm_ranges, int32_t num_seqs, int64_t num_tokens, int32_t max_query_len,
                      int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t block_size,
                      int32_t window, int32_t causal, const int32_t *seq_causal, int32_t chunk_size,
                      int32_t chunk_lookback, float scale, int32_t dtype, int32_t num_splits,
                      const int32_t *splits_per_seq, void *out, float *lse, void *partial_out,
                      float *partial_lse, int32_t *err, AttnArgs &a);
bool attention_is_empty(const AttnArgs &a);
// Picks the attention kernel for checked arguments and launches it.
cudaError_t dispatch_attention(const AttnArgs &a, cudaStream_t st);
// Host-side checks of lse_combine (SWA_OK or a negative code); launches nothing.
int check_lse_combine(const void *partial_out, const float *partial_lse, int32_t num_splits,
                      int64_t num_tokens, int32_t num_heads, int32_t head_dim, int32_t dtype, const void *out);

// Context-parallel geometry of swa_slot_mapping_cp (validated by the caller).
struct CpArgs {
  int32_t kv_cache_block_size, world, rank, interleave;
};

// pos == nullptr: token i of request r sits at ctx[r] + i.
cudaError_t launch_slot_mapping(const int32_t *qsl, const int64_t *pos, const int32_t *ctx, const int32_t *bt,
                                int64_t stride, int32_t block_size, int32_t num_reqs,
                                int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                                int32_t *out, int32_t *err, cudaStream_t st, const CpArgs *cp = nullptr);

// Scatter of new K/V rows into the paged cache by slot id.
cudaError_t launch_kv_cache_write(const void *k_new, const void *v_new, const int32_t *slots,
                                  int64_t num_tokens, int64_t row_bytes, void *k_cache, void *v_cache,
                                  int64_t num_slots, int32_t *err, cudaStream_t st);

cudaError_t launch_tile_bounds(const int32_t *qsl, const int32_t *seq_lens, const int32_t *ctx,
                               const int32_t *mm, int32_t max_mm, int32_t num_seqs, int32_t window,
                               int32_t causal, int32_t per_seq_causal, int32_t chunk_size,
                               int32_t chunk_lookback, int32_t tile, int32_t bq, int32_t max_qblocks,
                               int32_t *out, int32_t *err, cudaStream_t st);

cudaError_t launch_lse_combine(const void *po, const float *pl, int32_t num_splits,
                               int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                               int32_t dtype, void *out, float *out_lse, cudaStream_t st);

// General CUDA-core attention: any supported dtype / head_dim, split or not
// (what no tensor-core kernel takes: a GQA group that does not divide 128).
cudaError_t launch_attention_simt(const AttnArgs &a, cudaStream_t st);

// Split-KV decode: bf16, few query tokens per sequence, K/V staged with cp.async.
bool decode_supported(const AttnArgs &a);
cudaError_t launch_attention_decode(const AttnArgs &a, cudaStream_t st);

// tcgen05 / TMEM / TMA prefill: bf16, head_dim 256, no split.
bool tc_supported(const AttnArgs &a);
cudaError_t launch_attention_tc(const AttnArgs &a, cudaStream_t st);

// The same for head_dim 128 and 64 with two query tiles per work item.
bool tc_pair_supported(const AttnArgs &a);
cudaError_t launch_attention_tc_pair(const AttnArgs &a, cudaStream_t st);

// tcgen05 / TMEM attention for everything else: bf16 or fp32 (fp32 as bf16
// hi + lo operand pairs), head_dim 64, 128 or 256, split or not.
bool tc_small_supported(const AttnArgs &a);
cudaError_t launch_attention_tc_small(const AttnArgs &a, cudaStream_t st);

}  // namespace swa
