// The C ABI (include/swa.h): host-side argument checks, then one launch per
// call on the caller's stream.  Nothing here allocates device memory.
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }
inline bool block_size_ok(int b) { return b == 16 || b == 32 || b == 64 || b == 128; }
inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }
inline int finish(cudaError_t e) { return e == cudaSuccess ? SWA_OK : SWA_E_CUDA; }
// chunked lookback replaces the sliding window's left edge: it needs a window and a chunk size
inline bool chunk_ok(int window, int chunk_size, int chunk_lookback) {
  return chunk_lookback < 0 || (window > 0 && chunk_size > 0);
}

// swa_set_watchdog: process-wide settings read by every later attention call.
std::atomic<uint64_t> g_wait_ns{0};      // 0: the default bound
std::atomic<int32_t> g_stall{0};

}  // namespace

namespace swa {

int prepare_attention(const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
                      const int32_t *block_table, int64_t block_table_stride, const int32_t *query_start_loc,
                      const int32_t *seq_lens, const int32_t *context_lens, const int32_t *mm_ranges,
                      int32_t max_mm_ranges, int32_t num_seqs, int64_t num_tokens, int32_t max_query_len,
                      int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t block_size,
                      int32_t window, int32_t causal, const int32_t *seq_causal, int32_t chunk_size,
                      int32_t chunk_lookback, float scale, int32_t dtype, int32_t num_splits,
                      const int32_t *splits_per_seq, void *out, float *lse, void *partial_out,
                      float *partial_lse, int32_t *err, AttnArgs &a) {
  a = AttnArgs{};
  if (num_seqs < 0 || num_tokens < 0 || num_blocks < 0 || block_table_stride < 1 ||
      max_mm_ranges < 0 || num_heads_q < 1 || num_heads_kv < 1 || num_splits < 1 ||
      max_query_len < 0)
    return SWA_E_SIZE;
  if (num_heads_q % num_heads_kv != 0 || num_heads_q / num_heads_kv > 32) return SWA_E_SIZE;
  if (num_heads_kv > 65535 || num_splits > 65535) return SWA_E_SIZE;
  if (dtype != SWA_DTYPE_BF16 && dtype != SWA_DTYPE_FP32) return SWA_E_UNSUPPORTED;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return SWA_E_UNSUPPORTED;
  if (!std::isfinite(scale)) return SWA_E_SIZE;
  if (!chunk_ok(window, chunk_size, chunk_lookback)) return SWA_E_SIZE;
  if (num_tokens == 0 || num_seqs == 0) return SWA_OK;     // nothing to do: `a` stays empty
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      query_start_loc == nullptr || seq_lens == nullptr)
    return SWA_E_NULL;
  if (num_splits > 1) {
    if (partial_out == nullptr || partial_lse == nullptr) return SWA_E_NULL;
    if (!aligned16(partial_out)) return SWA_E_ALIGN;
  } else {
    if (out == nullptr) return SWA_E_NULL;
    if (!aligned16(out)) return SWA_E_ALIGN;
  }
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return SWA_E_ALIGN;

  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.num_blocks = num_blocks;
  a.block_table = block_table; a.bt_stride = block_table_stride;
  a.qsl = query_start_loc; a.seq_lens = seq_lens; a.ctx_lens = context_lens;
  a.mm_ranges = (max_mm_ranges > 0) ? mm_ranges : nullptr;
  a.max_mm_ranges = (mm_ranges != nullptr) ? max_mm_ranges : 0;
  a.num_seqs = num_seqs; a.num_tokens = num_tokens; a.max_query_len = max_query_len;
  a.hq = num_heads_q; a.hkv = num_heads_kv; a.head_dim = head_dim; a.block_size = block_size;
  a.window = window; a.causal = causal != 0; a.scale = scale; a.dtype = dtype;
  a.seq_causal = seq_causal;
  a.chunk_size = chunk_size; a.chunk_lookback = chunk_lookback < 0 ? -1 : chunk_lookback;
  a.num_splits = num_splits; a.splits_per_seq = (num_splits > 1) ? splits_per_seq : nullptr;
  a.out = out; a.lse = lse; a.partial_out = partial_out; a.partial_lse = partial_lse; a.err = err;
  const uint64_t wait_ns = g_wait_ns.load();
  a.wait_ns = wait_ns != 0 ? wait_ns : kDefaultWaitNs;
  a.stall = g_stall.load();
  return SWA_OK;
}

bool attention_is_empty(const AttnArgs &a) { return a.num_tokens == 0 || a.num_seqs == 0; }

cudaError_t dispatch_attention(const AttnArgs &a, cudaStream_t st) {
  if (tc_pair_supported(a)) return launch_attention_tc_pair(a, st);
  if (tc_supported(a)) return launch_attention_tc(a, st);
  if (decode_supported(a)) return launch_attention_decode(a, st);
  if (tc_small_supported(a)) return launch_attention_tc_small(a, st);
  return launch_attention_simt(a, st);
}

int check_lse_combine(const void *partial_out, const float *partial_lse, int32_t num_splits,
                      int64_t num_tokens, int32_t num_heads, int32_t head_dim, int32_t dtype, const void *out) {
  if (num_splits < 1 || num_tokens < 0 || num_heads < 1) return SWA_E_SIZE;
  if (!head_dim_ok(head_dim)) return SWA_E_UNSUPPORTED;
  if (dtype != SWA_DTYPE_BF16 && dtype != SWA_DTYPE_FP32) return SWA_E_UNSUPPORTED;
  if (num_tokens == 0) return SWA_OK;
  if (partial_out == nullptr || partial_lse == nullptr || out == nullptr) return SWA_E_NULL;
  if (!aligned16(partial_out) || !aligned16(out)) return SWA_E_ALIGN;
  return SWA_OK;
}

}  // namespace swa

extern "C" {

const char *swa_version(void) { return "swa-gb300 0.1 sm_103a"; }

int swa_set_watchdog(uint64_t wait_limit_ns, int32_t stall) {
  if (wait_limit_ns != 0 && (wait_limit_ns < 1000ull || wait_limit_ns > 10000000000ull)) return SWA_E_SIZE;
  g_wait_ns.store(wait_limit_ns);
  g_stall.store(stall != 0 ? 1 : 0);
  return SWA_OK;
}

int swa_slot_mapping(const int32_t *query_start_loc, const int64_t *positions,
                     const int32_t *context_lens, const int32_t *block_table, int64_t block_table_stride,
                     int32_t block_size, int32_t num_reqs, int64_t num_tokens, int64_t max_num_tokens,
                     int32_t pad_id, int32_t *slot_mapping, int32_t *err, void *stream) {
  if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens || block_size <= 0 ||
      block_table_stride < 1)
    return SWA_E_SIZE;
  if (max_num_tokens == 0) return SWA_OK;
  if (slot_mapping == nullptr || query_start_loc == nullptr) return SWA_E_NULL;
  if (num_tokens > 0 && ((positions == nullptr && context_lens == nullptr) || block_table == nullptr))
    return SWA_E_NULL;
  if (max_num_tokens > INT32_MAX) return SWA_E_SIZE;
  return finish(swa::launch_slot_mapping(query_start_loc, positions, positions ? nullptr : context_lens, block_table,
                                         block_table_stride, block_size, num_reqs, num_tokens, max_num_tokens, pad_id,
                                         slot_mapping, err, as_stream(stream)));
}

int swa_slot_mapping_cp(const int32_t *query_start_loc, const int64_t *positions,
                        const int32_t *block_table, int64_t block_table_stride, int32_t block_size,
                        int32_t num_reqs, int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                        int32_t kv_cache_block_size, int32_t cp_world_size, int32_t cp_rank,
                        int32_t cp_interleave, int32_t *slot_mapping, int32_t *err, void *stream) {
  if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens || block_size <= 0 ||
      block_table_stride < 1)
    return SWA_E_SIZE;
  if (cp_world_size < 1 || cp_rank < 0 || cp_rank >= cp_world_size || cp_interleave < 1 ||
      kv_cache_block_size < 1 || kv_cache_block_size % block_size != 0 ||
      kv_cache_block_size % cp_interleave != 0 || (int64_t)kv_cache_block_size * cp_world_size > INT32_MAX)
    return SWA_E_SIZE;
  if (max_num_tokens == 0) return SWA_OK;
  if (slot_mapping == nullptr || query_start_loc == nullptr) return SWA_E_NULL;
  if (num_tokens > 0 && (positions == nullptr || block_table == nullptr)) return SWA_E_NULL;
  if (max_num_tokens > INT32_MAX) return SWA_E_SIZE;
  const swa::CpArgs cp{kv_cache_block_size, cp_world_size, cp_rank, cp_interleave};
  return finish(swa::launch_slot_mapping(query_start_loc, positions, nullptr, block_table, block_table_stride,
                                         block_size, num_reqs, num_tokens, max_num_tokens, pad_id,
                                         slot_mapping, err, as_stream(stream), &cp));
}

int swa_kv_cache_write(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                       int64_t num_tokens, int32_t num_heads_kv, int32_t head_dim, int32_t dtype,
                       void *k_cache, void *v_cache, int64_t num_slots, int32_t *err, void *stream) {
  if (num_tokens < 0 || num_heads_kv < 1 || head_dim < 1 || head_dim % 8 != 0 || num_slots < 0)
    return SWA_E_SIZE;
  if (dtype != SWA_DTYPE_BF16 && dtype != SWA_DTYPE_FP32) return SWA_E_UNSUPPORTED;
  if (num_tokens == 0) return SWA_OK;
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr || k_cache == nullptr ||
      v_cache == nullptr)
    return SWA_E_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache)) return SWA_E_ALIGN;
  const int64_t row_bytes = (int64_t)num_heads_kv * head_dim * (dtype == SWA_DTYPE_BF16 ? 2 : 4);
  return finish(swa::launch_kv_cache_write(k_new, v_new, slot_mapping, num_tokens, row_bytes, k_cache, v_cache,
                                           num_slots, err, as_stream(stream)));
}

int swa_tile_bounds(const int32_t *query_start_loc, const int32_t *seq_lens,
                    const int32_t *context_lens, const int32_t *mm_ranges, int32_t max_mm_ranges,
                    int32_t num_seqs, int32_t window, int32_t causal, int32_t per_seq_causal,
                    int32_t chunk_size, int32_t chunk_lookback, int32_t tile_size, int32_t block_q,
                    int32_t max_qblocks_per_seq, int32_t *out, int32_t *err, void *stream) {
  if (tile_size <= 0 || block_q <= 0 || num_seqs < 0 || max_qblocks_per_seq < 0 || max_mm_ranges < 0)
    return SWA_E_SIZE;
  if (!chunk_ok(window, chunk_size, chunk_lookback)) return SWA_E_SIZE;
  if (num_seqs == 0 || max_qblocks_per_seq == 0) return SWA_OK;
  if (query_start_loc == nullptr || seq_lens == nullptr || out == nullptr) return SWA_E_NULL;
  if (num_seqs > 65535) return SWA_E_SIZE;
  return finish(swa::launch_tile_bounds(query_start_loc, seq_lens, context_lens, mm_ranges,
                                        max_mm_ranges, num_seqs, window, causal != 0, per_seq_causal != 0,
                                        chunk_size, chunk_lookback < 0 ? -1 : chunk_lookback, tile_size,
                                        block_q, max_qblocks_per_seq, out, err, as_stream(stream)));
}

int swa_mm_paged_attention(const void *q, const void *k_cache, const void *v_cache,
                           int64_t num_blocks, const int32_t *block_table,
                           int64_t block_table_stride, const int32_t *query_start_loc,
                           const int32_t *seq_lens, const int32_t *context_lens,
                           const int32_t *mm_ranges, int32_t max_mm_ranges, int32_t num_seqs,
                           int64_t num_tokens, int32_t max_query_len, int32_t num_heads_q,
                           int32_t num_heads_kv, int32_t head_dim, int32_t block_size,
                           int32_t window, int32_t causal, const int32_t *seq_causal,
                           int32_t chunk_size, int32_t chunk_lookback, float scale, int32_t dtype,
                           int32_t num_splits, const int32_t *splits_per_seq, void *out,
                           float *lse, void *partial_out, float *partial_lse, int32_t *err,
                           void *stream) {
  swa::AttnArgs a;
  const int rc = swa::prepare_attention(q, k_cache, v_cache, num_blocks, block_table, block_table_stride,
                                        query_start_loc, seq_lens, context_lens, mm_ranges, max_mm_ranges,
                                        num_seqs, num_tokens, max_query_len, num_heads_q, num_heads_kv, head_dim,
                                        block_size, window, causal, seq_causal, chunk_size, chunk_lookback, scale,
                                        dtype, num_splits, splits_per_seq, out, lse, partial_out, partial_lse,
                                        err, a);
  if (rc != SWA_OK || swa::attention_is_empty(a)) return rc;
  return finish(swa::dispatch_attention(a, as_stream(stream)));
}

int lse_combine(const void *partial_out, const float *partial_lse, int32_t num_splits,
                int64_t num_tokens, int32_t num_heads, int32_t head_dim, int32_t dtype, void *out,
                float *out_lse, void *stream) {
  const int rc = swa::check_lse_combine(partial_out, partial_lse, num_splits, num_tokens, num_heads, head_dim,
                                        dtype, out);
  if (rc != SWA_OK || num_tokens == 0) return rc;
  return finish(swa::launch_lse_combine(partial_out, partial_lse, num_splits, num_tokens, num_heads,
                                        head_dim, dtype, out, out_lse, as_stream(stream)));
}

}  // extern "C"
