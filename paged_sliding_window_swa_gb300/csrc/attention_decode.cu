// Split-KV decode attention over the paged KV cache (few query tokens per
// sequence), with the same visibility rule as the prefill kernels (vLLM PR
// #53147 summary, implementation items 1-2) and the partition convention of
// the split-KV partial outputs merged by LSE (MLA DCP decode study notes,
// section 1.1).
//
// Decode is bound by HBM: every visible K and V row is read once and used by
// at most 16 query rows (query positions x the heads of one kv head).  One
// CTA owns one (sequence, kv head, partition).  Each of its 4 warps streams
// 16-key chunks of K and V through its own cp.async ring in shared memory --
// a chunk never crosses a page, so one block-table lookup serves it; keys
// outside the rows' union, past the sequence or on a bad page are zero-filled
// without a global read -- and the warps never wait on each other until the
// final merge.  A warp computes S = Q K^T and O += P V for its chunk with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate): at 16 rows the 128-row tcgen05
// tile would be nearly empty, and at this size the tensor work is tiny
// against the K/V stream.  P is reused from the S accumulators as the A
// operand of P V without leaving registers; the online softmax keeps its max
// in the log2 domain and rescales only when it grows by more than 2^8.  The
// warps' states merge through shared memory at the end.
#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 16;          // keys per ring stage (never crosses a page)
constexpr int kMaxRows = 16;        // query rows per CTA: the M of one mma.sync tile
constexpr int kStages = 3;

__device__ inline void cp_async16(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ inline void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ inline void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ inline void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ inline void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ inline void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ inline uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ inline float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct DecShape {
  static constexpr int ROW = D * 2 + 16;                 // padded smem row: conflict-free ldmatrix
  static constexpr int TILE = kChunk * ROW;              // one K or V chunk
  static constexpr int STAGE = 2 * TILE;
  static constexpr int RING = kStages * STAGE;           // per warp
  static constexpr int MERGE = kWarps * kMaxRows * (D + 2) * 4;
  static constexpr int SMEM = (kWarps * RING > MERGE ? kWarps * RING : MERGE);
};

template <int D>
__global__ void __launch_bounds__(kThreads)
attn_decode_kernel(AttnArgs a) {
  using Sh = DecShape<D>;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_lo[kMaxRows], s_hi[kMaxRows];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, i4 = lane & 3;                // mma fragment coordinates
  const int s = blockIdx.x, hk = blockIdx.y, split = blockIdx.z;
  const int G = a.hq / a.hkv;
  const int qstart = __ldg(a.qsl + s);
  const int qlen = __ldg(a.qsl + s + 1) - qstart;
  if (qlen <= 0) return;
  const int rows = qlen * G;
  if (rows > kMaxRows || qstart < 0 || (int64_t)qstart + qlen > a.num_tokens) {
    if (threadIdx.x == 0) report(a.err, rows > kMaxRows ? SWA_ERR_LENS : SWA_ERR_QSL);
    return;
  }
  const int seq_len = __ldg(a.seq_lens + s);
  const int ctx = seq_len - qlen;
  const bool causal = a.seq_causal != nullptr ? __ldg(a.seq_causal + s) != 0 : a.causal != 0;
  if (ctx < 0 || (a.ctx_lens != nullptr && __ldg(a.ctx_lens + s) != ctx)) {
    if (threadIdx.x == 0) report(a.err, SWA_ERR_LENS);
    return;
  }
  // this CTA's partition of the keys
  Span part{0, seq_len - 1};
  bool live = true;
  if (a.num_splits > 1) {
    int parts = a.splits_per_seq ? __ldg(a.splits_per_seq + s) : a.num_splits;
    if (parts < 1 || parts > a.num_splits) {
      if (threadIdx.x == 0) report(a.err, SWA_ERR_SPLITS);
      parts = min(max(parts, 1), a.num_splits);
    }
    if (split >= parts) live = false;
    else part = split_span(seq_len, parts, split);
  }
  // a dependent kernel (the LSE merge of the partials) may be launched now; it
  // waits for this grid to complete before it reads anything
  pdl_launch_dependents();
  // rows' visible intervals inside the partition (rows >= `rows` see nothing)
  if (threadIdx.x < kMaxRows) {
    int lo = 1, hi = 0;
    const int r = threadIdx.x;
    if (live && r < rows) {
      const int32_t *ranges = a.mm_ranges ? a.mm_ranges + (int64_t)s * a.max_mm_ranges * 2 : nullptr;
      const Span sp = visible_span(ctx + r / G, seq_len, a.window, causal, a.chunk_size, a.chunk_lookback,
                                   ranges, a.mm_ranges ? a.max_mm_ranges : 0);
      lo = max(sp.lo, part.lo);
      hi = min(sp.hi, part.hi);
    }
    s_lo[r] = lo;
    s_hi[r] = hi;
  }
  __syncthreads();
  int umin = INT_MAX, umax = -1;
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r)
    if (s_lo[r] <= s_hi[r]) { umin = min(umin, s_lo[r]); umax = max(umax, s_hi[r]); }
  // this thread's two fragment rows: g and g + 8
  const int lo0 = s_lo[g], hi0 = s_hi[g], lo1 = s_lo[g + 8], hi1 = s_hi[g + 8];

  // Q as the A operand of S = Q K^T, for every 16-column step of head_dim
  const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(a.q);
  uint32_t qa[D / 16][4];
  {
    const bool v0 = g < rows, v1 = g + 8 < rows;
    const uint32_t *q0 = reinterpret_cast<const uint32_t *>(
        qg + ((int64_t)(qstart + (v0 ? g / G : 0)) * a.hq + hk * G + (v0 ? g % G : 0)) * D);
    const uint32_t *q1 = reinterpret_cast<const uint32_t *>(
        qg + ((int64_t)(qstart + (v1 ? (g + 8) / G : 0)) * a.hq + hk * G + (v1 ? (g + 8) % G : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = v0 ? __ldg(q0 + kk * 8 + i4) : 0u;
      qa[kk][1] = v1 ? __ldg(q1 + kk * 8 + i4) : 0u;
      qa[kk][2] = v0 ? __ldg(q0 + kk * 8 + 4 + i4) : 0u;
      qa[kk][3] = v1 ? __ldg(q1 + kk * 8 + 4 + i4) : 0u;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int db = 0; db < D / 8; ++db) o[db][0] = o[db][1] = o[db][2] = o[db][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = a.scale * kLog2e;

  const __nv_bfloat16 *kc = static_cast<const __nv_bfloat16 *>(a.k_cache);
  const __nv_bfloat16 *vc = static_cast<const __nv_bfloat16 *>(a.v_cache);
  const int32_t *bt = a.block_table + (int64_t)s * a.bt_stride;
  const int kbase = umax >= umin ? (umin / kChunk) * kChunk : 0;
  const int n_chunks = umax >= umin ? (umax - kbase) / kChunk + 1 : 0;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + warp * Sh::RING;

  // stage one 16-key chunk of K and V (one page, one block-table lookup)
  auto load_chunk = [&](int c, int stage) {
    const int k0 = kbase + c * kChunk;
    const int page = k0 / a.block_size;
    const int32_t blk = page < a.bt_stride ? __ldg(bt + page) : -1;
    const bool page_ok = blk >= 0 && blk < a.num_blocks;
    if (!page_ok && lane == 0 && k0 <= umax) report(a.err, SWA_ERR_BLOCK_ID);
    const int64_t row0 = page_ok ? (((int64_t)blk * a.block_size + (k0 - page * a.block_size)) * a.hkv + hk) * D : 0;
    const uint32_t dst = ring + stage * Sh::STAGE;
#pragma unroll
    for (int p = lane; p < 2 * kChunk * (D / 8); p += 32) {
      const int kv = p / (kChunk * (D / 8));                // 0 = K, 1 = V
      const int rem = p - kv * (kChunk * (D / 8));
      const int kr = rem / (D / 8), col = (rem % (D / 8)) * 8;
      const int k = k0 + kr;
      const bool ok = page_ok && k >= umin && k <= umax;
      const __nv_bfloat16 *src = (kv ? vc : kc) + (ok ? row0 + (int64_t)kr * a.hkv * D + col : 0);
      cp_async16(dst + kv * Sh::TILE + kr * Sh::ROW + col * 2, src, ok ? 16u : 0u);
    }
  };

  int issued = 0;                                   // chunks of this warp staged so far
  for (int it = 0; it < kStages - 1; ++it) {
    const int c = warp + kWarps * issued;
    if (c < n_chunks) load_chunk(c, issued % kStages);
    cp_async_commit();
    ++issued;
  }
  for (int it = 0;; ++it) {
    const int c = warp + kWarps * it;
    if (c >= n_chunks) break;
    {
      const int cn = warp + kWarps * issued;
      if (cn < n_chunks) load_chunk(cn, issued % kStages);
      cp_async_commit();
      ++issued;
    }
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint32_t ks = ring + (it % kStages) * Sh::STAGE;
    const uint32_t vs = ks + Sh::TILE;
    const int k0 = kbase + c * kChunk;

    // S = Q K^T: two n8 blocks of keys (0-7, 8-15); B fragments by ldmatrix
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int lm = lane >> 3, lr = lane & 7;          // ldmatrix: matrix, row
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(ks + ((lm >> 1) * 8 + lr) * Sh::ROW + (kk * 16 + (lm & 1) * 8) * 2, b00, b01, b10, b11);
      mma16816(sacc[0], qa[kk], b00, b01);
      mma16816(sacc[1], qa[kk], b10, b11);
    }
    // mask, scale into the log2 domain; this thread holds keys nb*8 + 2*i4 + e
    float x[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = k0 + nb * 8 + 2 * i4 + e;
        x[nb][e] = (k >= lo0 && k <= hi0) ? sacc[nb][e] * sl2 : -INFINITY;
        x[nb][2 + e] = (k >= lo1 && k <= hi1) ? sacc[nb][2 + e] * sl2 : -INFINITY;
      }
    float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
    float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (mx0 > m0 + 8.f) {                              // lazy rescale of row g
      const float al = m0 == -INFINITY ? 0.f : ex2f(m0 - mx0);
      l0 *= al;
#pragma unroll
      for (int db = 0; db < D / 8; ++db) { o[db][0] *= al; o[db][1] *= al; }
      m0 = mx0;
    }
    if (mx1 > m1 + 8.f) {                              // and of row g + 8
      const float al = m1 == -INFINITY ? 0.f : ex2f(m1 - mx1);
      l1 *= al;
#pragma unroll
      for (int db = 0; db < D / 8; ++db) { o[db][2] *= al; o[db][3] *= al; }
      m1 = mx1;
    }
    const float ms0 = m0 == -INFINITY ? 0.f : m0, ms1 = m1 == -INFINITY ? 0.f : m1;
    float p[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      p[nb][0] = ex2f(x[nb][0] - ms0);
      p[nb][1] = ex2f(x[nb][1] - ms0);
      p[nb][2] = ex2f(x[nb][2] - ms1);
      p[nb][3] = ex2f(x[nb][3] - ms1);
    }
    l0 += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
    l1 += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
    // P as the A operand of O += P V (rows g, g+8; keys 2*i4 (+1), +8)
    const uint32_t pa[4] = {pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(p[0][2], p[0][3]),
                            pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(p[1][2], p[1][3])};
    // V fragments by transposed ldmatrix: two n8 blocks of head_dim per load
#pragma unroll
    for (int db = 0; db < D / 8; db += 2) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4_t(vs + ((lm & 1) * 8 + lr) * Sh::ROW + (db + (lm >> 1)) * 8 * 2, b00, b01, b10, b11);
      mma16816(o[db], pa, b00, b01);
      mma16816(o[db + 1], pa, b10, b11);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();                                   // rings are free: reuse them for the merge

  // per-warp row sums over the four lanes of a fragment row, then the merge
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  float *mrg = reinterpret_cast<float *>(smem);      // [warp][row][D + 2]: O, then m, l
  {
    float *r0 = mrg + (warp * kMaxRows + g) * (D + 2);
    float *r1 = mrg + (warp * kMaxRows + g + 8) * (D + 2);
#pragma unroll
    for (int db = 0; db < D / 8; ++db) {
      r0[db * 8 + 2 * i4] = o[db][0];
      r0[db * 8 + 2 * i4 + 1] = o[db][1];
      r1[db * 8 + 2 * i4] = o[db][2];
      r1[db * 8 + 2 * i4 + 1] = o[db][3];
    }
    if (i4 == 0) {
      r0[D] = m0; r0[D + 1] = l0;
      r1[D] = m1; r1[D + 1] = l1;
    }
  }
  __syncthreads();
  // warp w finishes rows w, w + 4, ...: merge the 4 warps' states and store
  for (int r = warp; r < rows; r += kWarps) {
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, mrg[(w * kMaxRows + r) * (D + 2) + D]);
    float wgt[kWarps], ll = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = mrg[(w * kMaxRows + r) * (D + 2) + D];
      wgt[w] = mw == -INFINITY ? 0.f : ex2f(mw - mm);
      ll += mrg[(w * kMaxRows + r) * (D + 2) + D + 1] * wgt[w];
    }
    const bool any = ll > 0.f;
    const float inv = any ? 1.f / ll : 0.f;
    const float lse = any ? (mm + log2f(ll)) * kLn2 : -INFINITY;
    const int64_t row = (int64_t)(qstart + r / G) * a.hq + hk * G + r % G;
    __nv_bfloat16 *dst;
    if (a.num_splits > 1) {
      if (lane == 0) a.partial_lse[(int64_t)split * a.num_tokens * a.hq + row] = lse;
      dst = any ? static_cast<__nv_bfloat16 *>(a.partial_out) + ((int64_t)split * a.num_tokens * a.hq + row) * D
                : nullptr;
    } else {
      if (lane == 0 && a.lse != nullptr) a.lse[row] = lse;
      dst = static_cast<__nv_bfloat16 *>(a.out) + row * D;
    }
    if (dst != nullptr)
      for (int d = 2 * lane; d < D; d += 64) {
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          v0 = fmaf(mrg[(w * kMaxRows + r) * (D + 2) + d], wgt[w], v0);
          v1 = fmaf(mrg[(w * kMaxRows + r) * (D + 2) + d + 1], wgt[w], v1);
        }
        *reinterpret_cast<__nv_bfloat162 *>(dst + d) = __floats2bfloat162_rn(v0 * inv, v1 * inv);
      }
  }
}

template <int D>
cudaError_t run(const AttnArgs &a, cudaStream_t st) {
  using Sh = DecShape<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
  if (e != cudaSuccess) return e;
  // prefer the largest shared-memory carveout so two CTAs fit on an SM
  e = cudaFuncSetAttribute(attn_decode_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)a.num_seqs, (unsigned)a.hkv, (unsigned)max(1, a.num_splits));
  attn_decode_kernel<D><<<grid, kThreads, Sh::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(const AttnArgs &a) {
  const int G = a.hq / a.hkv;
  // a 16-key chunk must never cross a page: block sizes are multiples of 16
  return a.dtype == SWA_DTYPE_BF16 && (a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256) &&
         a.block_size % kChunk == 0 && a.max_query_len >= 1 && (int64_t)a.max_query_len * G <= kMaxRows;
}

cudaError_t launch_attention_decode(const AttnArgs &a, cudaStream_t st) {
  switch (a.head_dim) {
    case 64: return run<64>(a, st);
    case 128: return run<128>(a, st);
    case 256: return run<256>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace swa
