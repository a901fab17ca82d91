// Tensor-core (tcgen05 / TMEM) attention for the shapes the two fast kernels
// do not take: fp32 inputs, split-KV partitions with many query rows, and GQA
// groups of 32 to 128 (head_dim 64, 128 or 256).  Same mask and pruning as
// attention_tc.cu (vLLM PR #53147 summary, implementation items 1-2 and the
// compute_tile_loop_bounds excerpt); split partitions as in the split-KV
// decode (MLA DCP decode study notes, section 1.1).
//
// One CTA of four warps per 128-row query tile (128 / G positions x the G
// query heads of one kv head) and split partition; thread i owns row i (TMEM
// lane i).  Per key tile of N keys, in order and without overlap: the warps
// stage K and V from the paged cache into shared memory (bf16, 128-byte
// swizzled, the layouts the MMA descriptors read), one thread issues
// S = Q K^T, every thread masks and exponentiates its row of S and writes P
// to TMEM, one thread issues O += P V.
//
// fp32 inputs keep fp32 accuracy on the bf16 tensor cores: every operand x is
// split into x_hi = bf16(x) and x_lo = bf16(x - x_hi), and each product as
// x_hi y_hi + x_hi y_lo + x_lo y_hi (the dropped x_lo y_lo term and the
// rounding of x_lo are below 2^-16 of |x y|), accumulated in fp32 in TMEM.
// P is split the same way.
//
// Every mbarrier wait is bounded; on expiry the CTA reports SWA_ERR_TIMEOUT,
// waits (bounded) for its own MMAs, frees TMEM and exits.
#include "attn_tc_common.cuh"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr int kSmallThreads = 128;

constexpr uint32_t pow2_cols(int n) {
  uint32_t c = 32;
  while ((int)c < n) c <<= 1;
  return c;
}

template <typename T, int D_>
struct SmallCfg {
  static constexpr int D = D_;
  static constexpr bool SPLIT = sizeof(T) == 4;        // fp32 operands as bf16 hi + lo
  static constexpr int NC = SPLIT ? 2 : 1;             // bf16 copies of every operand
  static constexpr int N = (SPLIT && D == 256) ? 32 : 128;   // keys per tile (shared-memory budget)
  static constexpr int M = 128;
  static constexpr int CH = D / 64;                    // 64-column chunks (128 bytes of bf16)
  static constexpr int Q_CHUNK = M * 128;
  static constexpr int Q_BYTES = CH * Q_CHUNK;         // one bf16 copy of the Q tile
  static constexpr int KV_CHUNK = N * 128;
  static constexpr int KV_BYTES = CH * KV_CHUNK;       // one bf16 copy of a K or V tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NC * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NC * KV_BYTES;
  static constexpr int OFF_CTRL = OFF_V + NC * KV_BYTES;
  static constexpr int TM_O = 0;                       // TMEM: O [0, D), S [D, D+N), P copies after S
  static constexpr int TM_S = D;
  static constexpr int TM_P = D + N;                   // copy i at TM_P + i * N / 2 (bf16 pairs)
  static constexpr uint32_t TM_COLS = pow2_cols(D + N + NC * N / 2);
  static constexpr int PIECE = 16 / (int)sizeof(T);    // elements per 16-byte source piece
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, N, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
};

struct SmallCtrl {
  uint64_t bar_s, bar_o, bar_drain;     // S complete, PV complete, drain
  uint32_t tmem_base;
  int red_lo[4], red_hi[4];
};

template <class C>
constexpr int small_smem() { return C::OFF_CTRL + (int)sizeof(SmallCtrl); }

// Byte offset of bf16 column c (a multiple of 4) of row r in a tile stored as
// 64-column chunks of `rows` rows x 128 bytes, 128-byte swizzled.
__device__ inline uint32_t sw_off(int r, int c, int rows) {
  const int cc = c & 63;
  return (uint32_t)((c >> 6) * rows * 128 + r * 128 + ((((cc >> 3) ^ (r & 7))) << 4) + ((cc & 7) << 1));
}

// Stores one 16-byte source piece (PIECE elements starting at column c) of
// row r: bf16 as it is, fp32 as its hi and lo bf16 copies.
template <class C, typename T>
__device__ inline void stage_piece(uint8_t *base, int copy_bytes, int r, int c, int rows, const uint4 &v) {
  const uint32_t off = sw_off(r, c, rows);
  if constexpr (C::SPLIT) {
    const float *f = reinterpret_cast<const float *>(&v);
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(f[2 * i]), h1 = __float2bfloat16_rn(f[2 * i + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(f[2 * i] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(f[2 * i + 1] - __bfloat162float(h1));
      hi[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    *reinterpret_cast<uint2 *>(base + off) = make_uint2(hi[0], hi[1]);
    *reinterpret_cast<uint2 *>(base + copy_bytes + off) = make_uint2(lo[0], lo[1]);
  } else {
    *reinterpret_cast<uint4 *>(base + off) = v;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kSmallThreads, 1)
attn_tc_small_kernel(const AttnArgs a, const int G, const int bq) {
  using C = SmallCfg<T, D>;
  constexpr int N = C::N;
  static_assert(C::TM_COLS <= 512 && small_smem<C>() <= 227 * 1024, "TMEM and shared-memory budgets");
  // everything in dynamic shared memory, which starts 1024-byte aligned when a
  // kernel has no static shared data (checked below; the swizzled tiles need it)
  extern __shared__ __align__(1024) uint8_t dsm[];
  SmallCtrl &ctl = *reinterpret_cast<SmallCtrl *>(dsm + C::OFF_CTRL);
  uint64_t &bar_s = ctl.bar_s, &bar_o = ctl.bar_o, &bar_drain = ctl.bar_drain;
  int *red_lo = ctl.red_lo, *red_hi = ctl.red_hi;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  Item it;
  int32_t eb;
  if (!decode_item(a, (int)blockIdx.x, bq, it, eb)) {
    if (eb != 0 && tid == 0 && blockIdx.y == 0) report(a.err, eb);
    return;
  }
  if ((smem_u32(dsm) & 1023u) != 0) {
    if (tid == 0) report(a.err, SWA_ERR_INTERNAL);
    return;
  }
  // the CTA's split partition of the keys
  const int split = (int)blockIdx.y;
  Span part{0, it.seq_len - 1};
  bool live = true;
  if (a.num_splits > 1) {
    int parts = a.splits_per_seq ? __ldg(a.splits_per_seq + it.s) : a.num_splits;
    if (parts < 1 || parts > a.num_splits) {
      if (tid == 0) report(a.err, SWA_ERR_SPLITS);
      parts = min(max(parts, 1), a.num_splits);
    }
    if (split >= parts) live = false;
    else part = split_span(it.seq_len, parts, split);
  }
  // this thread's row and its visible keys inside the partition
  const int qpos = it.qpos_lo + tid / G;
  const bool row_valid = qpos < it.qlen;
  const int64_t out_row = (int64_t)(it.qstart + qpos) * a.hq + it.hk * G + tid % G;
  int klo = 1, khi = 0;
  if (row_valid && live) {
    const int32_t *ranges = a.mm_ranges ? a.mm_ranges + (int64_t)it.s * a.max_mm_ranges * 2 : nullptr;
    const Span sp = visible_span(it.ctx + qpos, it.seq_len, a.window, it.causal, a.chunk_size, a.chunk_lookback,
                                 ranges, a.mm_ranges ? a.max_mm_ranges : 0);
    klo = max(sp.lo, part.lo);
    khi = min(sp.hi, part.hi);
  }
  {
    int lo = klo <= khi ? klo : INT_MAX, hi = klo <= khi ? khi : -1;
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
      red_lo[warp] = lo;
      red_hi[warp] = hi;
    }
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar_s), 1);
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&ctl.tmem_base), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t lane_t = (uint32_t)(32 * warp) << 16;
  int kmin = INT_MAX, kmax = -1;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    kmin = min(kmin, red_lo[w]);
    kmax = max(kmax, red_hi[w]);
  }
  const int tile_lo = kmax >= 0 ? kmin / N : 0;
  const int n_tiles = kmax >= 0 ? kmax / N - tile_lo + 1 : 0;

  const uint32_t s_base = smem_u32(dsm);
  const T *qg = static_cast<const T *>(a.q);
  const T *kc = static_cast<const T *>(a.k_cache);
  const T *vc = static_cast<const T *>(a.v_cache);
  constexpr int PPR = D / C::PIECE;                      // 16-byte pieces per row
  // Q tile: row r = position r / G, head it.hk * G + r % G; rows past the
  // query length are zero
  for (int i = tid; i < C::M * PPR; i += kSmallThreads) {
    const int r = i / PPR, c = (i % PPR) * C::PIECE;
    uint4 v = make_uint4(0, 0, 0, 0);
    const int qp = it.qpos_lo + r / G;
    if (qp < it.qlen)
      v = __ldg(reinterpret_cast<const uint4 *>(qg + ((int64_t)(it.qstart + qp) * a.hq + it.hk * G + r % G) * D + c));
    stage_piece<C, T>(dsm + C::OFF_Q, C::Q_BYTES, r, c, C::M, v);
  }

  const float sl2 = a.scale * kLog2e;                    // scores in the log2 domain (any sign)
  const int32_t *bt = a.block_table + (int64_t)it.s * a.bt_stride;
  float m_used = -INFINITY, l = 0.f;
  bool ok = true;
  for (int t = 0; t < n_tiles && ok; ++t) {
    const int k0 = (tile_lo + t) * N;
    if (t > 0) {
      // PV(t-1) done: V, P and O are free
      ok = __syncthreads_and(mbar_wait(smem_u32(&bar_o), (uint32_t)((t - 1) & 1), nullptr, a.wait_ns));
      if (!ok) break;
      tc_fence_after();
    }
    // K and V rows of the tile; keys past the sequence (or on a bad page) are zero
    for (int i = tid; i < N * PPR; i += kSmallThreads) {
      const int n = i / PPR, c = (i % PPR) * C::PIECE;
      const int k = k0 + n;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (k < it.seq_len) {
        const int page = k / a.block_size;
        const int32_t blk = page < a.bt_stride ? __ldg(bt + page) : -1;
        if (blk >= 0 && blk < a.num_blocks) {
          const int64_t off = ((int64_t)blk * a.block_size + k % a.block_size) * a.hkv * D + (int64_t)it.hk * D + c;
          kv = __ldg(reinterpret_cast<const uint4 *>(kc + off));
          vv = __ldg(reinterpret_cast<const uint4 *>(vc + off));
        } else if (c == 0) {
          report(a.err, SWA_ERR_BLOCK_ID);
        }
      }
      stage_piece<C, T>(dsm + C::OFF_K, C::KV_BYTES, n, c, N, kv);
      stage_piece<C, T>(dsm + C::OFF_V, C::KV_BYTES, n, c, N, vv);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32, ko = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
        const uint32_t qh = s_base + C::OFF_Q + qo, kh = s_base + C::OFF_K + ko;
        mma_ss(tmem + C::TM_S, smem_desc_sw128(qh, 16, 1024), smem_desc_sw128(kh, 16, 1024), C::IDESC_QK,
               kk > 0 ? 1u : 0u);
        if constexpr (C::SPLIT) {
          mma_ss(tmem + C::TM_S, smem_desc_sw128(qh, 16, 1024), smem_desc_sw128(kh + C::KV_BYTES, 16, 1024),
                 C::IDESC_QK, 1u);
          mma_ss(tmem + C::TM_S, smem_desc_sw128(qh + C::Q_BYTES, 16, 1024), smem_desc_sw128(kh, 16, 1024),
                 C::IDESC_QK, 1u);
        }
      }
      mma_commit(smem_u32(&bar_s));
    }
    ok = __syncthreads_and(mbar_wait(smem_u32(&bar_s), (uint32_t)(t & 1), nullptr, a.wait_ns));
    if (!ok) break;
    tc_fence_after();
    // this row of S: the masked maximum (a first pass over S in TMEM), the
    // rescale of O, then P (a second pass)
    float mx = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < N / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_t + C::TM_S + 32 * c, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int k = k0 + 32 * c + e;
        if (k >= klo && k <= khi) mx = fmaxf(mx, __uint_as_float(r[e]) * sl2);
      }
    }
    const float m_new = fmaxf(m_used, mx);
    const bool grow = m_new > m_used;
    if (__any_sync(0xffffffffu, grow)) {
      const float alpha = (!grow || m_used == -INFINITY) ? (grow ? 0.f : 1.f) : ex2(m_used - m_new);
      if (t > 0) {
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_t + C::TM_O + 32 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tmem + lane_t + C::TM_O + 32 * c, r);
        }
        tmem_wait_st();
      }
      l *= alpha;
      if (grow) m_used = m_new;
    }
    const float ms = m_used == -INFINITY ? 0.f : m_used;
#pragma unroll 1
    for (int c = 0; c < N / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_t + C::TM_S + 32 * c, r);
      tmem_wait_ld();
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int k = k0 + 32 * c + 2 * e;
        const float x0 = (k >= klo && k <= khi) ? __uint_as_float(r[2 * e]) * sl2 : -INFINITY;
        const float x1 = (k + 1 >= klo && k + 1 <= khi) ? __uint_as_float(r[2 * e + 1]) * sl2 : -INFINITY;
        const float p0 = ex2(x0 - ms), p1 = ex2(x1 - ms);
        l += p0 + p1;
        const __nv_bfloat16 h0 = __float2bfloat16_rn(p0), h1 = __float2bfloat16_rn(p1);
        ph[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        if constexpr (C::SPLIT)
          pl[e] = pack_bf16(p0 - __bfloat162float(h0), p1 - __bfloat162float(h1));
      }
      tmem_st16(tmem + lane_t + C::TM_P + 16 * c, ph);
      if constexpr (C::SPLIT) tmem_st16(tmem + lane_t + C::TM_P + N / 2 + 16 * c, pl);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      for (int kk = 0; kk < N / 16; ++kk) {
        const uint32_t vb = s_base + C::OFF_V + kk * 16 * 128;
        const uint32_t ph = tmem + C::TM_P + kk * 8;
        mma_ts(tmem + C::TM_O, ph, smem_desc_sw128(vb, C::KV_CHUNK, 1024), C::IDESC_PV, (t > 0 || kk > 0) ? 1u : 0u);
        if constexpr (C::SPLIT) {
          mma_ts(tmem + C::TM_O, ph, smem_desc_sw128(vb + C::KV_BYTES, C::KV_CHUNK, 1024), C::IDESC_PV, 1u);
          mma_ts(tmem + C::TM_O, ph + N / 2, smem_desc_sw128(vb, C::KV_CHUNK, 1024), C::IDESC_PV, 1u);
        }
      }
      mma_commit(smem_u32(&bar_o));
    }
  }
  if (ok && n_tiles > 0) {
    ok = __syncthreads_and(mbar_wait(smem_u32(&bar_o), (uint32_t)((n_tiles - 1) & 1), nullptr, a.wait_ns));
    tc_fence_after();
  }
  if (ok) {
    // epilogue: O / l (zero for a row with no visible key), LSE
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    T *dst = nullptr;
    if (a.num_splits > 1) {
      if (row_valid) a.partial_lse[(int64_t)split * a.num_tokens * a.hq + out_row] = lse;
      if (row_valid && l > 0.f) dst = static_cast<T *>(a.partial_out) + ((int64_t)split * a.num_tokens * a.hq + out_row) * D;
    } else {
      if (row_valid && a.lse != nullptr) a.lse[out_row] = lse;
      if (row_valid) dst = static_cast<T *>(a.out) + out_row * D;
    }
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      if (n_tiles > 0) {
        tmem_ld32(tmem + lane_t + C::TM_O + 32 * c, r);
        tmem_wait_ld();
      }
      if (dst != nullptr) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          float o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = n_tiles > 0 ? __uint_as_float(r[e + i]) * inv : 0.f;
          if constexpr (sizeof(T) == 4) {
            reinterpret_cast<float4 *>(dst + 32 * c + e)[0] = make_float4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<float4 *>(dst + 32 * c + e)[1] = make_float4(o[4], o[5], o[6], o[7]);
          } else {
            *reinterpret_cast<uint4 *>(dst + 32 * c + e) =
                make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
          }
        }
      }
    }
  } else {
    if (tid == 0) report(a.err, SWA_ERR_TIMEOUT);
    // the MMAs this CTA issued must be done before TMEM is released
    if (tid == 0) {
      mma_commit(smem_u32(&bar_drain));
      mbar_wait(smem_u32(&bar_drain), 0, nullptr, kWaitLimitNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <typename T, int D>
cudaError_t run_small(const AttnArgs &a, cudaStream_t st) {
  using C = SmallCfg<T, D>;
  const int G = a.hq / a.hkv;
  const int bq = C::M / G;
  constexpr int smem = small_smem<C>();
  cudaError_t e = cudaFuncSetAttribute(attn_tc_small_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (a.num_tokens / bq + a.num_seqs) * (int64_t)a.hkv;
  dim3 grid((unsigned)items, (unsigned)max(1, a.num_splits));
  attn_tc_small_kernel<T, D><<<grid, kSmallThreads, smem, st>>>(a, G, bq);
  return cudaGetLastError();
}

}  // namespace

// Any head_dim of the library, bf16 or fp32, split or not; a GQA group that
// divides the 128-row tile; 32-bit token indices.
bool tc_small_supported(const AttnArgs &a) {
  const int G = a.hq / a.hkv;
  const int64_t items = (a.num_tokens / (128 / max(G, 1)) + a.num_seqs) * (int64_t)a.hkv;
  return (a.head_dim == 64 || a.head_dim == 128 || a.head_dim == 256) && G >= 1 && G <= 128 && (G & (G - 1)) == 0 &&
         a.num_tokens < (int64_t)INT32_MAX && items < (int64_t)INT32_MAX && a.num_splits <= 65535;
}

cudaError_t launch_attention_tc_small(const AttnArgs &a, cudaStream_t st) {
  if (a.dtype == SWA_DTYPE_BF16) {
    switch (a.head_dim) {
      case 64: return run_small<__nv_bfloat16, 64>(a, st);
      case 128: return run_small<__nv_bfloat16, 128>(a, st);
      case 256: return run_small<__nv_bfloat16, 256>(a, st);
    }
  } else {
    switch (a.head_dim) {
      case 64: return run_small<float, 64>(a, st);
      case 128: return run_small<float, 128>(a, st);
      case 256: return run_small<float, 256>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace swa
