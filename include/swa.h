/*
 * swa.h -- C ABI of the GB300 paged sliding-window attention library.
 *
 * Varlen prefill/decode attention over a paged KV cache with a sliding window
 * (SWA) and a window-clamped bidirectional image-prefix mask, plus the two
 * feeders around it: token -> KV-slot mapping and the log-sum-exp merge of
 * split-KV partial outputs.  Hand-written CUDA for sm_103a (GB300).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership.  Every array argument is a DEVICE pointer owned by the caller.
 *   The library allocates no memory and keeps no pointer after a call returns
 *   (swa_mm_paged_attention_split_static works in a fixed array of its own
 *   instead, placed on a device by the first call there; see there).
 * Streams.  `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *   default stream.  Each call only enqueues work on `stream` and never
 *   synchronises the host.
 * Errors.  The return value is SWA_OK (0), or a negative SWA_E_* code when the
 *   host-side argument checks fail -- in that case nothing is launched.  Data
 *   errors that can only be seen on the device (a block id outside the cache,
 *   a position outside the block-table row, inconsistent lengths, a stalled
 *   pipeline) set SWA_ERR_* bits in the optional device word `err` with
 *   atomicOr; the affected entries get PAD / zero / -inf and the kernel keeps
 *   going.  Kernels never trap.  Pass err = NULL to skip the report.
 * Layouts (row-major, innermost last):
 *   q            [num_tokens, num_heads_q, head_dim]            (bf16 or fp32)
 *   k/v cache    [num_blocks, block_size, num_heads_kv, head_dim] (slot-major:
 *                slot = block * block_size + offset)
 *   block_table  [num_seqs, block_table_stride] int32, logical page -> block
 *   mm_ranges    [num_seqs, max_mm_ranges, 2] int32, inclusive [start, end]
 *                in absolute sequence positions; start >= end is padding
 *   out          [num_tokens, num_heads_q, head_dim]   lse [num_tokens, num_heads_q] fp32
 *   partial_out  [num_splits, num_tokens, num_heads_q, head_dim]
 *   partial_lse  [num_splits, num_tokens, num_heads_q] fp32
 * Query token i of sequence s sits at absolute position
 *   context_lens[s] + i,  with context_lens[s] = seq_lens[s] - query_len[s];
 * the KV cache already holds all seq_lens[s] keys of the sequence.
 * Query head h reads kv head h / (num_heads_q / num_heads_kv).
 */
#ifndef SWA_GB300_H
#define SWA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- host-side return codes ------------------------------------------- */
#define SWA_OK             0
#define SWA_E_NULL        -1   /* a required pointer is NULL                      */
#define SWA_E_SIZE        -2   /* a size is negative, zero where it must not be,
                                  or sizes disagree (e.g. Hq % Hkv != 0)          */
#define SWA_E_UNSUPPORTED -3   /* dtype / head_dim / block_size not built         */
#define SWA_E_ALIGN       -4   /* a pointer is not 16-byte aligned               */
#define SWA_E_CUDA        -5   /* the CUDA runtime or driver reported an error    */
#define SWA_E_SCRATCH     -6   /* the call needs more than the library's fixed
                                  scratch array holds (see below)                 */

/* ---- device-side error bits (atomicOr into *err) ------------------------ */
#define SWA_ERR_BLOCK_ID   0x01  /* block_table entry outside [0, num_blocks)      */
#define SWA_ERR_POSITION   0x02  /* position < 0 or its page beyond the table row  */
#define SWA_ERR_QSL        0x04  /* query_start_loc not monotone / past num_tokens */
#define SWA_ERR_LENS       0x08  /* seq_lens / context_lens inconsistent           */
#define SWA_ERR_TIMEOUT    0x10  /* a bounded pipeline wait gave up                */
#define SWA_ERR_SPLITS     0x20  /* splits_per_seq entry outside [1, num_splits]   */
#define SWA_ERR_INTERNAL   0x40  /* a kernel could not set up its pipeline (its
                                    outputs are not written)                      */
#define SWA_ERR_SLOT       0x80  /* a slot id at or past the end of the KV cache   */

/* ---- element types ------------------------------------------------------ */
#define SWA_DTYPE_BF16 0
#define SWA_DTYPE_FP32 1

/* Split-KV partitions start on multiples of this many keys (see below). */
#define SWA_SPLIT_ALIGN 128

/*
 * swa_slot_mapping -- logical token position -> physical KV-cache slot.
 *
 * Defined by the vllm-ascend article on _compute_slot_mapping_kernel,
 * section 2 ("non-CP path") and section 1 (the padded tail): for token t of
 * request r, with pos = positions[t] (or, when positions is NULL,
 * pos = context_lens[r] + (t - query_start_loc[r]): the request's cached
 * context followed by its new tokens),
 *     slot_mapping[t] = block_table[r][pos / block_size] * block_size
 *                       + pos % block_size,
 * and slot_mapping[t] = pad_id for t in [num_tokens, max_num_tokens), which
 * keeps the output shape fixed for graph capture.
 *
 *   query_start_loc  int32[num_reqs + 1], CSR offsets of each request's tokens
 *   positions        int64[num_tokens], or NULL to derive them
 *   context_lens     int32[num_reqs]; read only when positions is NULL
 *   block_table      int32[num_reqs, block_table_stride]
 *   slot_mapping     int32[max_num_tokens] (output)
 * Host errors: NULL pointers (except err, and one of positions /
 *   context_lens), num_reqs < 0, num_tokens < 0,
 *   max_num_tokens < num_tokens, block_size <= 0, stride < 1.
 * Device errors: a position < 0 or whose page index >= block_table_stride
 *   sets SWA_ERR_POSITION and writes pad_id; query_start_loc that decreases or
 *   passes num_tokens sets SWA_ERR_QSL (tokens outside every request get pad_id).
 */
int swa_slot_mapping(const int32_t *query_start_loc, const int64_t *positions,
                     const int32_t *context_lens, const int32_t *block_table,
                     int64_t block_table_stride, int32_t block_size, int32_t num_reqs,
                     int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                     int32_t *slot_mapping, int32_t *err, void *stream);

/*
 * swa_slot_mapping_cp -- swa_slot_mapping on one rank of a context-parallel
 * group whose KV cache is interleaved across the ranks.
 *
 * Defined by the same article, section 3 ("multi-CP domains", steps 1-5):
 * token i of a sequence lives on rank (i / cp_interleave) % cp_world_size.
 * With W = cp_world_size, I = cp_interleave, pos = positions[t]:
 *     v_idx = pos / (kv_cache_block_size * W),  v_off = pos % (kv_cache_block_size * W)
 *     token is local   iff (v_off / I) % W == cp_rank
 *     local_off        = (v_off / (W * I)) * I + v_off % I
 *     block_index      = v_idx * (kv_cache_block_size / block_size) + local_off / block_size
 *     slot_mapping[t]  = block_table[r][block_index] * block_size + local_off % block_size
 * and pad_id for tokens owned by another rank and for the padded tail.  A
 * rank's segments are thus concatenated: its j-th token of a sequence sits at
 * local offset j.  With W = 1 and I = 1 this is swa_slot_mapping.
 *
 *   arguments as for swa_slot_mapping, plus
 *   kv_cache_block_size   a multiple of block_size and of cp_interleave
 *   cp_world_size >= 1, 0 <= cp_rank < cp_world_size, cp_interleave >= 1
 * Host errors: those of swa_slot_mapping, and a geometry that breaks the
 *   rules above (SWA_E_SIZE).
 * Device errors: as swa_slot_mapping (a block index >= block_table_stride sets
 *   SWA_ERR_POSITION).
 */
int swa_slot_mapping_cp(const int32_t *query_start_loc, const int64_t *positions,
                        const int32_t *block_table, int64_t block_table_stride,
                        int32_t block_size, int32_t num_reqs, int64_t num_tokens,
                        int64_t max_num_tokens, int32_t pad_id, int32_t kv_cache_block_size,
                        int32_t cp_world_size, int32_t cp_rank, int32_t cp_interleave,
                        int32_t *slot_mapping, int32_t *err, void *stream);

/*
 * swa_kv_cache_write -- store a step's new K and V rows in the paged cache.
 *
 * The slot ids of swa_slot_mapping are what the cache-write and attention
 * operators consume (the slot-mapping article, section 1 and its closing
 * summary): for every token t with 0 <= slot_mapping[t] < num_slots,
 *     k_cache[slot_mapping[t]] = k_new[t],   v_cache[slot_mapping[t]] = v_new[t]
 * (all num_heads_kv x head_dim elements of the row).  A negative slot is a
 * padding token and writes nothing.  When two tokens carry the same slot, which
 * one lands is unspecified.
 *
 *   k_new, v_new      [num_tokens, num_heads_kv, head_dim] (dtype), 16-byte aligned
 *   slot_mapping      int32[num_tokens]
 *   k_cache, v_cache  [num_slots, num_heads_kv, head_dim] (dtype) -- the
 *                     [num_blocks, block_size, Hkv, D] caches with
 *                     num_slots = num_blocks * block_size
 * Host errors: NULL pointers (except err), num_tokens < 0, num_heads_kv < 1,
 *   head_dim not a positive multiple of 8, unsupported dtype, misaligned pointers.
 * Device errors: a slot >= num_slots sets SWA_ERR_SLOT and writes nothing.
 */
int swa_kv_cache_write(const void *k_new, const void *v_new, const int32_t *slot_mapping,
                       int64_t num_tokens, int32_t num_heads_kv, int32_t head_dim, int32_t dtype,
                       void *k_cache, void *v_cache, int64_t num_slots, int32_t *err,
                       void *stream);

/*
 * swa_tile_bounds -- per query block, the KV-tile loop range after pruning.
 *
 * Defined by the vLLM PR #53147 summary, the compute_tile_loop_bounds excerpt
 * (with its CHUNK_LOOKBACK and USE_PER_SEQ_CAUSAL branches) and its geometry
 * tests.  Query block b of sequence s holds query rows
 * qpos_lo = b*block_q .. qpos_hi = min(qpos_lo + block_q - 1, query_len - 1);
 * q_lo = ctx + qpos_lo, q_hi = ctx + qpos_hi;  rc = causal && !per_seq_causal.
 *   max_seq_prefix_len = seq_len if image ranges are enabled (mm_ranges != NULL
 *     and max_mm_ranges > 0) or !rc, else min(q_hi + 1, seq_len);
 *   num_tiles = ceil(max_seq_prefix_len / tile_size);
 *   window <= 0: [lo, hi) = [0, num_tiles);
 *   window  > 0: first = q_lo - window + 1, or with chunk_lookback >= 0
 *       first = ((q_lo / chunk_size) - chunk_lookback) * chunk_size;
 *     last = rc ? q_hi : q_hi + window - 1;
 *     every valid range [s, e] (s < e) with s <= q_hi and e >= q_lo gives
 *     first = min(first, max(s, q_lo - window + 1)), last = max(last, e);
 *     last = min(last, seq_len - 1);
 *     lo = max(0, floor(first / tile_size)), hi = min(last / tile_size + 1, num_tiles).
 * (The page takes the block's last row for the window's and the chunk's left
 * edge; this library takes the first row, which keeps every visible key of the
 * block's earlier rows inside [lo, hi) and gives the printed [3, 72) and
 * [3, 68).)  per_seq_causal (0/1) is the per-sequence causal mode: the flags
 * themselves are not read, every sequence is bounded with the non-causal
 * right edge, as the excerpt does.  chunk_lookback < 0 turns chunking off
 * (chunk_size is then ignored).
 *
 *   context_lens  int32[num_seqs] or NULL (then seq_len - query_len)
 *   out           int32[num_seqs, max_qblocks_per_seq, 3] = {lo, hi,
 *                 max_seq_prefix_len}; blocks past the query length get {0,0,0}
 * Host errors: NULL (except context_lens, mm_ranges, err), tile_size <= 0,
 *   block_q <= 0, num_seqs < 0, max_qblocks_per_seq < 0, max_mm_ranges < 0,
 *   chunk_lookback >= 0 with window <= 0 or chunk_size <= 0 (SWA_E_SIZE).
 * Device errors: context_lens[s] != seq_len - query_len or query_len > seq_len
 *   sets SWA_ERR_LENS and writes {0, 0, 0} for the sequence.
 */
int swa_tile_bounds(const int32_t *query_start_loc, const int32_t *seq_lens,
                    const int32_t *context_lens, const int32_t *mm_ranges,
                    int32_t max_mm_ranges, int32_t num_seqs, int32_t window, int32_t causal,
                    int32_t per_seq_causal, int32_t chunk_size, int32_t chunk_lookback,
                    int32_t tile_size, int32_t block_q, int32_t max_qblocks_per_seq,
                    int32_t *out, int32_t *err, void *stream);

/*
 * swa_mm_paged_attention -- paged attention with SWA and the clamped image mask.
 *
 * Key k of sequence s is visible to the query at absolute position q when
 * (vLLM PR #53147 summary, implementation items 1-2, "OR semantics"):
 *     base(q,k): window > 0: k >= left(q) and (causal ? k <= q : k <= q+window-1)
 *                window <= 0: causal ? k <= q : true
 *  OR mm(q,k):   some valid range [s0,e0] holds both q and k, and
 *                (window > 0) k >= q - window + 1
 *  AND 0 <= k < seq_lens[s].
 * left(q) = q - window + 1, or with chunked lookback (chunk_lookback >= 0,
 * compute_tile_loop_bounds excerpt) the start of the chunk chunk_lookback
 * chunks before q's: ((q / chunk_size) - chunk_lookback) * chunk_size.  The
 * image term keeps the window clamp, so it can reach keys before the chunk
 * (the reviewer's note on the same summary).  `causal` is sequence s's flag
 * seq_causal[s] != 0 when seq_causal is not NULL (the per-sequence causal
 * mode), else the argument.
 * With sc = scale * dot(q, k) over the visible keys:
 *     out = sum_k exp(sc - m) v_k / sum_k exp(sc - m),  lse = m + ln sum_k exp(sc - m)
 * (m = max sc, natural log).  Tiles outside the pruned loop range of
 * swa_tile_bounds are never read.
 *
 * Split-KV (num_splits > 1): sequence s uses P_s = splits_per_seq[s] (or
 * num_splits when splits_per_seq is NULL) partitions.  Partition p covers the
 * keys [p*L, min((p+1)*L, seq_len)), L = SWA_SPLIT_ALIGN *
 * ceil(ceil(seq_len / P_s) / SWA_SPLIT_ALIGN).  Each (p, token, head) gets the
 * normalised partial output over the visible keys of its partition and their
 * LSE; when the partition holds no visible key for the row (including p >= P_s)
 * partial_lse = -inf and that partial_out row is NOT written (lse_combine never
 * reads it).  out / lse are not written in split mode; merge with lse_combine.
 *
 *   q, k_cache, v_cache   see layouts; dtype SWA_DTYPE_BF16 or SWA_DTYPE_FP32
 *   num_blocks            first dimension of the caches (block ids are checked)
 *   query_start_loc       int32[num_seqs + 1]
 *   seq_lens              int32[num_seqs]
 *   context_lens          int32[num_seqs] or NULL (derived)
 *   mm_ranges             int32[num_seqs, max_mm_ranges, 2] or NULL
 *   seq_causal            int32[num_seqs] or NULL (per-sequence causal flags)
 *   chunk_size, chunk_lookback  chunked lookback; chunk_lookback < 0: off
 *                         (chunk_size ignored), >= 0 needs window > 0 and
 *                         chunk_size > 0 (else SWA_E_SIZE)
 *   max_query_len         host-side upper bound of every query length (it
 *                         selects the decode or the prefill kernel; a value
 *                         below a sequence's query length sets SWA_ERR_LENS
 *                         for that sequence in the decode kernel)
 *   head_dim              64, 128 or 256;  block_size 16, 32, 64 or 128
 *   out                   [num_tokens, Hq, D] same dtype as q  (num_splits == 1)
 *   lse                   fp32 [num_tokens, Hq] or NULL          (num_splits == 1)
 *   partial_out/partial_lse  required when num_splits > 1, else ignored
 * Host errors: NULL pointers, non-positive sizes, Hq % Hkv != 0, an unsupported
 *   dtype/head_dim/block_size, misaligned (not 16-byte) q/k/v/out pointers.
 * Device errors: SWA_ERR_BLOCK_ID (rows that see such a page get unspecified
 *   but finite outputs), SWA_ERR_LENS and SWA_ERR_QSL (the sequence's rows are
 *   not written), SWA_ERR_SPLITS, SWA_ERR_TIMEOUT, SWA_ERR_INTERNAL.
 */
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
                           void *stream);

/*
 * lse_combine -- merge split-KV partial outputs with their log-sum-exp.
 *
 * Defined by the MLA DCP decode study notes, section 1.1 and the LSE glossary
 * entry (partial results merged by their LSE equal one softmax over the whole
 * sequence).  Per (token, head):
 *     L = max_p lse_p;  w_p = exp(lse_p - L);
 *     out = sum_p w_p * o_p / sum_p w_p;   out_lse = L + ln(sum_p w_p).
 * Partitions with lse_p = -inf have weight 0 and o_p is not read.  When every
 * partition is -inf, out = 0 and out_lse = -inf.  Accumulation is fp32.
 *
 *   partial_out  [num_splits, num_tokens, num_heads, head_dim] (dtype)
 *   partial_lse  fp32 [num_splits, num_tokens, num_heads]
 *   out          [num_tokens, num_heads, head_dim] (dtype)
 *   out_lse      fp32 [num_tokens, num_heads] or NULL
 * Host errors: NULL pointers, num_splits < 1, num_tokens < 0, num_heads < 1,
 *   head_dim not in {64, 128, 256}, unsupported dtype, misaligned pointers.
 * Launch: as a programmatic dependent of the work enqueued before it on the
 *   stream (it may start during the tail of a preceding kernel and waits for
 *   that kernel's completion before reading the partials); the ordering
 *   towards everything else in the stream is unchanged, inside CUDA graphs too.
 */
int lse_combine(const void *partial_out, const float *partial_lse, int32_t num_splits,
                int64_t num_tokens, int32_t num_heads, int32_t head_dim, int32_t dtype,
                void *out, float *out_lse, void *stream);

/*
 * swa_mm_paged_attention_split_static -- split-KV attention followed by its
 * LSE merge, with no device allocation by anyone.
 *
 * The pages have no counterpart of this call; it is a convenience for callers
 * that cannot allocate device memory when they run attention: an engine whose
 * allocator reserved the device up front, a plugin host that hands its kernels
 * fixed buffers and forbids allocation while enqueuing, or a loop that cannot
 * take the device-wide synchronisation of cudaMalloc / cudaFree.  The split
 * partials (partial_out, partial_lse of swa_mm_paged_attention) live in a
 * library-owned array of SWA_STATIC_SCRATCH_BYTES bytes that every GPU loading
 * the library holds until the process exits.  The result equals
 * swa_mm_paged_attention with num_splits > 1 followed by lse_combine.
 *
 *   arguments as swa_mm_paged_attention, without partial_out / partial_lse;
 *   num_splits >= 2; out [num_tokens, Hq, D] (dtype) and lse fp32
 *   [num_tokens, Hq] (or NULL) are the caller's, as there.
 * Scratch needed: round_up(num_splits * num_tokens * Hq * D * elem, 256)
 *   + num_splits * num_tokens * Hq * 4 bytes (elem 2 for bf16, 4 for fp32);
 *   more than SWA_STATIC_SCRATCH_BYTES returns SWA_E_SCRATCH and launches
 *   nothing.
 * First call on a device: it looks up the array's device address with that
 *   device current and caches it.  CUDA loads device code lazily by default,
 *   so that lookup is also when the array and this call's kernels are placed
 *   on the device (with CUDA_MODULE_LOADING=EAGER: when the context is
 *   created).  Make the first call on each device before reserving the rest
 *   of its memory and before any stream capture.  Later calls do no set-up.
 * Checks: every host-side check of swa_mm_paged_attention and lse_combine runs
 *   before anything is launched or the array is touched.
 * Sharing: every call on a device uses the same array and leaves its contents
 *   behind.  Calls whose work overlaps on the GPU (two streams, or two host
 *   threads) race on it; serialise them.  The LSE part is reset to -inf at the
 *   start of each call.
 * Errors: those of swa_mm_paged_attention and lse_combine, plus
 *   SWA_E_SCRATCH; num_splits < 2 is SWA_E_SIZE.  Rows of a sequence rejected
 *   on the device, and tokens that no sequence covers, come out as 0 with
 *   lse = -inf.
 */
#define SWA_STATIC_SCRATCH_BYTES (16u << 20)
int swa_mm_paged_attention_split_static(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_table, int64_t block_table_stride, const int32_t *query_start_loc,
    const int32_t *seq_lens, const int32_t *context_lens, const int32_t *mm_ranges,
    int32_t max_mm_ranges, int32_t num_seqs, int64_t num_tokens, int32_t max_query_len,
    int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t block_size, int32_t window,
    int32_t causal, const int32_t *seq_causal, int32_t chunk_size, int32_t chunk_lookback, float scale,
    int32_t dtype, int32_t num_splits, const int32_t *splits_per_seq, void *out, float *lse,
    int32_t *err, void *stream);

/*
 * swa_set_watchdog -- bound of the pipeline waits in the tensor-core
 * attention kernels, and a switch that makes those waits run out on purpose.
 *
 * The pages have no counterpart of this call.  Every wait of the tcgen05
 * prefill kernels (a TMA copy landing, an MMA completing, a softmax warpgroup
 * publishing its probabilities) is bounded in time; when a bound runs out the
 * kernel sets SWA_ERR_TIMEOUT in `err`, lets its own copies and MMAs finish,
 * frees its tensor memory and returns, so the CUDA context stays usable.
 *   wait_limit_ns  bound of each such wait for the attention calls made after
 *                  this one; 0 restores the default (200 ms); otherwise it must
 *                  lie in [1 us, 10 s] (else SWA_E_SIZE, nothing changes).
 *                  The final drains always keep the default bound.
 *   stall          nonzero: in every later tensor-core attention call the PV
 *                  issuer first waits on a barrier that nothing signals, so
 *                  that wait runs out after wait_limit_ns and the whole
 *                  pipeline of every CTA stops through the timeout path (the
 *                  call returns SWA_OK, `err` gets SWA_ERR_TIMEOUT, the
 *                  outputs are unspecified).  0: normal operation.  This is
 *                  for failure-detection tests of callers and of this library.
 * Settings are process-wide (all devices, all host threads) and apply to
 * calls enqueued after this one; the CUDA-core and decode kernels have no
 * pipeline waits and ignore them.  Returns SWA_OK or SWA_E_SIZE.
 */
int swa_set_watchdog(uint64_t wait_limit_ns, int32_t stall);

/* Library version string, e.g. "swa-gb300 0.1 sm_103a". */
const char *swa_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* SWA_GB300_H */
