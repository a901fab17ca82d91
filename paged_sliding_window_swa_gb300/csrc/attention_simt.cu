// General CUDA-core paged attention with the sliding window and the
// window-clamped image mask (vLLM PR #53147 summary, implementation items
// 1-2).  It serves every dtype / head_dim / split combination the ABI accepts
// and is the path for fp32 inputs and for the cases the tensor-core and
// decode kernels do not take.
//
// One CTA of 4 warps owns BQ query positions x G query heads of one kv head
// (GQA packing: each K/V tile is staged once for the whole group) and one
// split partition.  K/V tiles of 32 keys are gathered page by page through the
// block table into shared memory (fp32); each warp runs an online softmax for
// its rows, one key per lane.  The key loop covers only the union of the
// rows' visible intervals (the pruned tile range), and the per-key test is the
// interval check, which is the same set as the per-pair rule.
#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kKeys = 32;          // keys per tile (one per lane)
constexpr int kMaxRows = 32;       // query rows (positions x heads) per CTA
constexpr int kRowsPerWarp = kMaxRows / kWarps;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
attn_simt_kernel(AttnArgs a, int bq) {
  constexpr int KS = D + 1;                                   // padded K row: no bank conflicts
  constexpr int C = D / 32;                                   // output columns per lane
  constexpr int VE = 16 / sizeof(T);                          // elements per 16-byte vector
  extern __shared__ float smem[];
  const int G = a.hq / a.hkv;
  const int rows = bq * G;
  float *Qs = smem;                                           // [rows][D]
  float *Ks = Qs + kMaxRows * D;                              // [kKeys][KS]
  float *Vs = Ks + kKeys * KS;                                // [kKeys][D]
  int *kval = reinterpret_cast<int *>(Vs + kKeys * D);        // [kKeys]
  __shared__ int s_lo[kMaxRows], s_hi[kMaxRows];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hk = blockIdx.y;
  const int split = blockIdx.z;
  const int s = find_seq(a.qsl, a.num_seqs, blockIdx.x, bq);
  const int64_t first_blk = (int64_t)__ldg(a.qsl + s) / bq + s;
  const int local = (int)(blockIdx.x - first_blk);
  const int qstart = __ldg(a.qsl + s);
  const int qlen = __ldg(a.qsl + s + 1) - qstart;
  const int qpos_lo = local * bq;
  if (local < 0 || qpos_lo >= qlen) return;
  if (qstart < 0 || (int64_t)qstart + qlen > a.num_tokens) {
    if (threadIdx.x == 0) report(a.err, SWA_ERR_QSL);
    return;
  }
  const int seq_len = __ldg(a.seq_lens + s);
  const int ctx = seq_len - qlen;
  const bool causal = a.seq_causal != nullptr ? __ldg(a.seq_causal + s) != 0 : a.causal != 0;
  if (ctx < 0 || (a.ctx_lens != nullptr && __ldg(a.ctx_lens + s) != ctx)) {
    if (threadIdx.x == 0) report(a.err, SWA_ERR_LENS);
    return;
  }

  // split partition of this CTA
  Span part{0, seq_len - 1};
  if (a.num_splits > 1) {
    int parts = a.splits_per_seq ? __ldg(a.splits_per_seq + s) : a.num_splits;
    if (parts < 1 || parts > a.num_splits) {
      if (threadIdx.x == 0) report(a.err, SWA_ERR_SPLITS);
      parts = min(max(parts, 1), a.num_splits);
    }
    if (split >= parts) {
      part.lo = 1; part.hi = 0;                                // nothing visible
    } else {
      part = split_span(seq_len, parts, split);
    }
  }

  const int32_t *ranges = a.mm_ranges ? a.mm_ranges + (int64_t)s * a.max_mm_ranges * 2 : nullptr;
  const int nr = a.mm_ranges ? a.max_mm_ranges : 0;
  for (int r = threadIdx.x; r < kMaxRows; r += kThreads) {
    int lo = 1, hi = 0;
    if (r < rows && qpos_lo + r / G < qlen) {
      Span sp = visible_span(ctx + qpos_lo + r / G, seq_len, a.window, causal, a.chunk_size, a.chunk_lookback,
                             ranges, nr);
      lo = max(sp.lo, part.lo);
      hi = min(sp.hi, part.hi);
    }
    s_lo[r] = lo;
    s_hi[r] = hi;
  }
  // scaled queries (log2 domain)
  const float qscale = a.scale * kLog2e;
  const T *qg = static_cast<const T *>(a.q);
  for (int i = threadIdx.x; i < rows * D; i += kThreads) {
    const int r = i / D, d = i % D;
    const int qpos = qpos_lo + r / G;
    float v = 0.f;
    if (qpos < qlen)
      v = Elem<T>::to_f(qg[((int64_t)(qstart + qpos) * a.hq + hk * G + r % G) * D + d]) * qscale;
    Qs[i] = v;
  }
  __syncthreads();
  int kmin = INT_MAX, kmax = -1;
  for (int r = 0; r < rows; ++r)
    if (s_lo[r] <= s_hi[r]) { kmin = min(kmin, s_lo[r]); kmax = max(kmax, s_hi[r]); }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][C];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    m[i] = -INFINITY; l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) acc[i][c] = 0.f;
  }

  const T *kc = static_cast<const T *>(a.k_cache);
  const T *vc = static_cast<const T *>(a.v_cache);
  const int32_t *bt = a.block_table + (int64_t)s * a.bt_stride;
  for (int kt = (kmin / kKeys) * kKeys; kt <= kmax; kt += kKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kKeys * (D / VE); i += kThreads) {
      const int j = i / (D / VE), vcol = (i % (D / VE)) * VE;
      const int k = kt + j;
      bool ok = k <= kmax;
      int64_t base = 0;
      if (ok) {
        const int page = k / a.block_size;
        const int32_t blk = (page < a.bt_stride) ? __ldg(bt + page) : -1;
        if (blk < 0 || blk >= a.num_blocks) {
          ok = false;
          if (vcol == 0) report(a.err, SWA_ERR_BLOCK_ID);
        } else {
          base = (((int64_t)blk * a.block_size + k % a.block_size) * a.hkv + hk) * D + vcol;
        }
      }
      if (vcol == 0) kval[j] = ok;
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        Ks[j * KS + vcol + e] = ok ? Elem<T>::to_f(kc[base + e]) : 0.f;
        Vs[j * D + vcol + e] = ok ? Elem<T>::to_f(vc[base + e]) : 0.f;
      }
    }
    __syncthreads();
    const int k = kt + lane;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int r = warp + kWarps * i;
      if (r >= rows) continue;
      const int lo = s_lo[r], hi = s_hi[r];
      if (lo > hi || hi < kt || lo >= kt + kKeys) continue;      // warp-uniform
      float sc = -INFINITY;
      if (k >= lo && k <= hi && kval[lane]) {
        float dot = 0.f;
        const float *qr = Qs + r * D;
        const float *kr = Ks + lane * KS;
#pragma unroll 8
        for (int d = 0; d < D; ++d) dot = fmaf(qr[d], kr[d], dot);
        sc = dot;
      }
      const float tmax = warp_max(sc);
      if (tmax == -INFINITY) continue;
      const float mnew = fmaxf(m[i], tmax);
      const float alpha = exp2f(m[i] - mnew);                  // m = -inf -> 0
      const float p = exp2f(sc - mnew);
      l[i] = l[i] * alpha + warp_sum(p);
#pragma unroll
      for (int c = 0; c < C; ++c) acc[i][c] *= alpha;
      for (int j = 0; j < kKeys; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
        if (pj == 0.f) continue;                                // warp-uniform
#pragma unroll
        for (int c = 0; c < C; ++c) acc[i][c] = fmaf(pj, Vs[j * D + lane + 32 * c], acc[i][c]);
      }
      m[i] = mnew;
    }
  }

  // epilogue
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int r = warp + kWarps * i;
    if (r >= rows) continue;
    const int qpos = qpos_lo + r / G;
    if (qpos >= qlen) continue;
    const int64_t row = (int64_t)(qstart + qpos) * a.hq + hk * G + r % G;
    const bool any = l[i] > 0.f;
    const float inv = any ? 1.f / l[i] : 0.f;
    const float lse = any ? (m[i] + log2f(l[i])) * kLn2 : -INFINITY;
    if (a.num_splits > 1) {
      if (lane == 0) a.partial_lse[(int64_t)split * a.num_tokens * a.hq + row] = lse;
      if (any) {
        T *po = static_cast<T *>(a.partial_out) + ((int64_t)split * a.num_tokens * a.hq + row) * D;
#pragma unroll
        for (int c = 0; c < C; ++c) po[lane + 32 * c] = Elem<T>::from_f(acc[i][c] * inv);
      }
    } else {
      T *o = static_cast<T *>(a.out) + row * D;
#pragma unroll
      for (int c = 0; c < C; ++c) o[lane + 32 * c] = Elem<T>::from_f(acc[i][c] * inv);
      if (a.lse != nullptr && lane == 0) a.lse[row] = lse;
    }
  }
}

template <typename T, int D>
cudaError_t run(const AttnArgs &a, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  const int bq = max(1, 16 / G);
  const size_t smem = sizeof(float) * (kMaxRows * D + kKeys * (D + 1) + kKeys * D) + sizeof(int) * kKeys;
  cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = a.num_tokens / bq + a.num_seqs;
  if (blocks == 0) return cudaSuccess;
  dim3 grid((unsigned)blocks, (unsigned)a.hkv, (unsigned)max(1, a.num_splits));
  attn_simt_kernel<T, D><<<grid, kThreads, smem, st>>>(a, bq);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt(const AttnArgs &a, cudaStream_t st) {
  if (a.hq / a.hkv > kMaxRows) return cudaErrorInvalidValue;
  if (a.dtype == SWA_DTYPE_BF16) {
    switch (a.head_dim) {
      case 64: return run<__nv_bfloat16, 64>(a, st);
      case 128: return run<__nv_bfloat16, 128>(a, st);
      case 256: return run<__nv_bfloat16, 256>(a, st);
    }
  } else {
    switch (a.head_dim) {
      case 64: return run<float, 64>(a, st);
      case 128: return run<float, 128>(a, st);
      case 256: return run<float, 256>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace swa
