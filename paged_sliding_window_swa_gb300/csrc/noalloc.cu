// swa_mm_paged_attention_split_static: split-KV attention and its LSE merge in
// one call, with the split partials held in a fixed array that the library
// owns, so the call allocates nothing.
//
// The ordinary split-KV path needs two caller-allocated intermediates,
// partial_out [P, T, Hq, D] and partial_lse [P, T, Hq].  Some callers cannot
// allocate device memory at the point of the call: an engine whose allocator
// reserved all device memory up front and hands out nothing afterwards, a
// plugin host that gives its kernels fixed buffers and forbids allocation
// inside its enqueue hook, or a latency-critical loop that cannot afford the
// device-wide synchronisation cudaMalloc / cudaFree imply.  For them this entry
// point keeps the partials in a file-scope __device__ array of
// SWA_STATIC_SCRATCH_BYTES bytes.
//
// When the array is reserved: CUDA loads this library's device code lazily by
// default, so the array (and this file's kernels) are placed on a device when
// the first call on that device looks up the array's address.  That first
// call must therefore come before the caller reserves the rest of the device,
// and before any stream capture; with CUDA_MODULE_LOADING=EAGER the array is
// placed when the CUDA context is created instead.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

// Every GPU that loads this code holds the array until the process exits.
static __device__ __align__(256) uint8_t g_split_scratch[SWA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};   // device address of g_split_scratch, per device ordinal

// The host-side name g_split_scratch is only a stand-in; the kernels need the
// array's device address, looked up once per device with that device current.
int scratch_address(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWA_E_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SWA_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || p == nullptr) return SWA_E_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return SWA_OK;
}

__global__ void fill_neg_inf(float *x, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    x[i] = -INFINITY;
}

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return 0;
  return n;
}

}  // namespace

extern "C" int swa_mm_paged_attention_split_static(
    const void *q, const void *k_cache, const void *v_cache, int64_t num_blocks,
    const int32_t *block_table, int64_t block_table_stride, const int32_t *query_start_loc,
    const int32_t *seq_lens, const int32_t *context_lens, const int32_t *mm_ranges,
    int32_t max_mm_ranges, int32_t num_seqs, int64_t num_tokens, int32_t max_query_len,
    int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim, int32_t block_size, int32_t window,
    int32_t causal, const int32_t *seq_causal, int32_t chunk_size, int32_t chunk_lookback, float scale,
    int32_t dtype, int32_t num_splits, const int32_t *splits_per_seq, void *out, float *lse,
    int32_t *err, void *stream) {
  if (num_splits < 2 || num_tokens < 0 || num_heads_q < 1 || head_dim < 1) return SWA_E_SIZE;
  if (dtype != SWA_DTYPE_BF16 && dtype != SWA_DTYPE_FP32) return SWA_E_UNSUPPORTED;
  if (num_tokens == 0 || num_seqs == 0) return SWA_OK;
  if (out == nullptr) return SWA_E_NULL;

  // partial_out first, then partial_lse on the next 256-byte boundary
  const int64_t rows = (int64_t)num_splits * num_tokens * num_heads_q;
  const int64_t elem = dtype == SWA_DTYPE_BF16 ? 2 : 4;
  if (rows > INT64_MAX / (head_dim * elem + 4 + 256)) return SWA_E_SCRATCH;
  const int64_t po_bytes = round_up(rows * head_dim * elem, 256);
  const int64_t need = po_bytes + rows * 4;
  if (need > (int64_t)SWA_STATIC_SCRATCH_BYTES) return SWA_E_SCRATCH;

  void *base = nullptr;
  int rc = scratch_address(&base);
  if (rc != SWA_OK) return rc;
  void *partial_out = base;
  float *partial_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(base) + po_bytes);

  // Every host-side check of both steps runs before anything is launched.
  swa::AttnArgs a;
  rc = swa::prepare_attention(q, k_cache, v_cache, num_blocks, block_table, block_table_stride, query_start_loc,
                              seq_lens, context_lens, mm_ranges, max_mm_ranges, num_seqs, num_tokens,
                              max_query_len, num_heads_q, num_heads_kv, head_dim, block_size, window, causal,
                              seq_causal, chunk_size, chunk_lookback, scale, dtype, num_splits, splits_per_seq,
                              nullptr, nullptr, partial_out, partial_lse, err, a);
  if (rc != SWA_OK) return rc;
  rc = swa::check_lse_combine(partial_out, partial_lse, num_splits, num_tokens, num_heads_q, head_dim, dtype, out);
  if (rc != SWA_OK) return rc;
  const int sms = device_sm_count();
  if (sms <= 0) return SWA_E_CUDA;

  // The array keeps the previous call's contents.  A partition row the
  // attention kernel leaves unwritten (a token no sequence covers, a sequence
  // it rejects on the device) must read as "no keys" (-inf), so the LSE part
  // is reset on every call; partial_out rows behind a -inf are never read.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t max_blocks = (int64_t)sms * 8, want = swa::ceil_div(rows, 256);
  const int64_t blocks = want < max_blocks ? want : max_blocks;
  fill_neg_inf<<<(unsigned)blocks, 256, 0, st>>>(partial_lse, rows);
  if (cudaGetLastError() != cudaSuccess) return SWA_E_CUDA;
  if (swa::dispatch_attention(a, st) != cudaSuccess) return SWA_E_CUDA;
  if (swa::launch_lse_combine(partial_out, partial_lse, num_splits, num_tokens, num_heads_q, head_dim, dtype, out,
                              lse, st) != cudaSuccess)
    return SWA_E_CUDA;
  return SWA_OK;
}
