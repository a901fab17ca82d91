// Pieces shared by the tensor-core attention kernels (attention_tc.cu,
// attention_tc_pair.cu, attention_tc_small.cu): the work items (a query block,
// or a pair of consecutive query blocks, of one sequence and one kv head), the
// union of their rows' visible intervals, the item records the scheduler warps
// publish, the per-row interval a softmax thread needs, and the host-side TMA
// descriptor helpers.
#pragma once

#include <climits>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace swa {
namespace {

constexpr uint64_t kWaitLimitNs = kDefaultWaitNs;  // drain waits: every copy and MMA must land before exit
constexpr int kMaxUnits = 8;                       // ring slots per operand

struct Item {
  int s, hk, qstart, qlen, qpos_lo, seq_len, ctx;
  int q_lo, q_hi;                        // absolute positions of the block's first and last rows
  bool causal;                           // the sequence's flag, or the call's
};

// Item -> (query block, kv head).  False for blocks past their sequence's
// query length (nothing to do) and for inconsistent metadata (err bits set).
__device__ inline bool decode_item(const AttnArgs &a, int item, int bq, Item &it, int32_t &errbits) {
  const int bx = item / a.hkv;
  it.hk = item - bx * a.hkv;
  it.s = find_seq(a.qsl, a.num_seqs, bx, bq);
  const int64_t first = (int64_t)__ldg(a.qsl + it.s) / bq + it.s;
  const int local = (int)(bx - first);
  it.qstart = __ldg(a.qsl + it.s);
  it.qlen = __ldg(a.qsl + it.s + 1) - it.qstart;
  it.qpos_lo = local * bq;
  errbits = 0;
  if (local < 0 || it.qpos_lo >= it.qlen) return false;
  if (it.qstart < 0 || (int64_t)it.qstart + it.qlen > a.num_tokens) {
    errbits = SWA_ERR_QSL;
    return false;
  }
  it.seq_len = __ldg(a.seq_lens + it.s);
  it.ctx = it.seq_len - it.qlen;
  if (it.ctx < 0 || (a.ctx_lens != nullptr && __ldg(a.ctx_lens + it.s) != it.ctx)) {
    errbits = SWA_ERR_LENS;
    return false;
  }
  it.q_lo = it.ctx + it.qpos_lo;
  it.q_hi = it.ctx + min(it.qpos_lo + bq - 1, it.qlen - 1);
  it.causal = a.seq_causal != nullptr ? __ldg(a.seq_causal + it.s) != 0 : a.causal != 0;
  return true;
}

// The union of the block's rows' visible intervals.  Right edge: the larger of
// the last row's base window and the end of every valid image range that meets
// the block (largest such end: `emax`, -1 if none).  Left edge: the smaller of
// the first row's base window (the base left edge never decreases with q) and
// every such range's clamped start max(s, q_lo-W+1) (smallest: `smin`,
// INT_MAX if none; a range meeting the block holds its row max(s, q_lo), whose
// clamped start that is).  A range meets the block exactly when it holds one
// of its rows, so this equals the union of the per-row intervals.
__device__ inline void union_keys(const AttnArgs &a, const Item &it, int emax, int smin, int &kmin, int &kmax) {
  kmin = max(0, min(base_lo(it.q_lo, a.window, a.chunk_size, a.chunk_lookback), smin));
  kmax = min(max(base_hi(it.q_hi, a.window, it.causal, it.seq_len), emax), it.seq_len - 1);
}

// What a softmax thread needs for one item: the item's tile range and its
// row's visible interval [klo, khi] (empty for rows past the query length).
struct RowSetup {
  Item it;
  int key_lo, n_tiles;
  int klo, khi;
  int64_t out_row;
  bool row_valid;
};

// An item as the scheduler warp decoded it, published in a ring of
// kRecSlots records in shared memory for the MMA issuers and the softmax, so
// that they do not repeat the decode (a chain of dependent global loads) at
// every item boundary.  n_tiles 0 marks the end of the CTA's stream.  The
// record also holds the image ranges that meet the item's rows (nr of them;
// -1 when more than kRecRanges do, and the softmax scans them itself).
constexpr int kRecSlots = 4;
constexpr int kRecRanges = 4;
struct ItemRec {
  Item it;
  int key_lo, n_tiles;                 // key tiles [key_lo + j N, key_lo + (j + 1) N), j < n_tiles
  int half_last;                       // 1: no row sees a key in the last tile's second half
  int nr;
  int rs[kRecRanges], re[kRecRanges];
};

// Whole warp, warp-uniform item: the item's key tiles (N keys each, covering
// the union of its rows' intervals, union_keys) and the image ranges that meet
// its rows, the i-th of them kept by lane i < kRecRanges in (rs, re); nr counts
// all of them.  The first tile starts at the union's first key rounded down to
// min(page size, N), not to a multiple of N: every page box a tile loads then
// still lies in one page, and a window of W keys seen from b positions takes
// ceil((W + b - 1 + page - 1) / N) tiles instead of up to one more.
// `half_last`: the union ends in the first N / 2 keys of the last tile, so its
// MMAs need only those (the softmax masks the rest of the tile anyway).
template <int N>
__device__ inline void block_keys_rec(const AttnArgs &a, const Item &it, int lane, int &key_lo, int &n_tiles,
                                      int &half_last, int &nr, int &rs, int &re) {
  int emax = -1, smin = INT_MAX;
  nr = 0;
  rs = 0;
  re = -1;
  if (a.mm_ranges != nullptr) {
    const int32_t *rg = a.mm_ranges + (int64_t)it.s * a.max_mm_ranges * 2;
    const int clamp = a.window > 0 ? it.q_lo - a.window + 1 : INT_MIN;
    for (int b = 0; b < a.max_mm_ranges; b += 32) {
      int s0 = 0, e0 = -1;
      if (b + lane < a.max_mm_ranges) {
        s0 = __ldg(rg + 2 * (b + lane));
        e0 = __ldg(rg + 2 * (b + lane) + 1);
      }
      const bool meets = s0 < e0 && s0 <= it.q_hi && e0 >= it.q_lo;
      if (meets) {
        emax = max(emax, e0);
        smin = min(smin, max(s0, clamp));
      }
      uint32_t m = __ballot_sync(0xffffffffu, meets);
      while (m != 0 && nr < kRecRanges) {              // warp-uniform
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const int s1 = __shfl_sync(0xffffffffu, s0, src), e1 = __shfl_sync(0xffffffffu, e0, src);
        if (lane == nr) {
          rs = s1;
          re = e1;
        }
        ++nr;
      }
      nr += __popc(m);                                 // the ones past kRecRanges are only counted
    }
    emax = __reduce_max_sync(0xffffffffu, emax);
    smin = __reduce_min_sync(0xffffffffu, smin);
  }
  int kmin, kmax;
  union_keys(a, it, emax, smin, kmin, kmax);
  key_lo = kmin & -min(a.block_size, N);             // page sizes are powers of two
  n_tiles = (kmax - key_lo) / N + 1;
  half_last = kmax - (key_lo + (n_tiles - 1) * N) < N / 2 ? 1 : 0;
}

// Whole warp: writes the record (n_tiles 0: the end of the stream).  The
// caller publishes it afterwards with one release (an mbarrier arrive).
__device__ inline void write_rec(ItemRec &r, const Item &it, int key_lo, int n_tiles, int half_last, int nr,
                                 int rs, int re, int lane) {
  if (lane < nr && lane < kRecRanges) {
    r.rs[lane] = rs;
    r.re[lane] = re;
  }
  if (lane == 0) {
    r.it = it;
    r.key_lo = key_lo;
    r.half_last = half_last;
    r.n_tiles = n_tiles;
    r.nr = nr <= kRecRanges ? nr : -1;
  }
  __threadfence_block();
  __syncwarp();
}

// A softmax thread's RowSetup from a record: its row's interval from the
// record's ranges, or, for a record that could not hold them all, from a scan
// of the sequence's ranges by the warp: a range is tested against the warp's
// 32 rows only when it meets their span (ballot).  Same rule as the visible
// interval of a single query: a valid range holding q moves the right edge to
// its end and the left edge to its clamped start.  `qoff`: the
// position of the thread's query tile within the item (0, or bq for the
// second tile of a pair).
__device__ inline void row_setup_rec(const AttnArgs &a, const ItemRec &r, int row, int G, int lane,
                                     RowSetup &rs, int qoff = 0) {
  rs.it = r.it;
  rs.it.qpos_lo += qoff;
  rs.key_lo = r.key_lo;
  rs.n_tiles = r.n_tiles;
  const Item &it = rs.it;
  const int qpos = it.qpos_lo + row / G;
  const int q = it.ctx + qpos;
  const int rclamp = a.window > 0 ? q - a.window + 1 : INT_MIN;
  int rhi = -1, rlo = INT_MAX;
  const int nr = r.nr;
  if (nr >= 0) {
    for (int i = 0; i < nr; ++i) {
      const int s1 = r.rs[i], e1 = r.re[i];
      if (s1 <= q && q <= e1) {
        rhi = max(rhi, e1);
        rlo = min(rlo, max(s1, rclamp));
      }
    }
  } else {
    const int32_t *rg = a.mm_ranges + (int64_t)it.s * a.max_mm_ranges * 2;
    const int wrow0 = row - lane;
    const int wq_lo = it.ctx + it.qpos_lo + wrow0 / G;
    const int wq_hi = it.ctx + it.qpos_lo + (wrow0 + 31) / G;
    for (int b = 0; b < a.max_mm_ranges; b += 32) {
      int s0 = 0, e0 = -1;
      if (b + lane < a.max_mm_ranges) {
        s0 = __ldg(rg + 2 * (b + lane));
        e0 = __ldg(rg + 2 * (b + lane) + 1);
      }
      uint32_t m = __ballot_sync(0xffffffffu, s0 < e0 && s0 <= wq_hi && e0 >= wq_lo);
      while (m != 0) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const int s1 = __shfl_sync(0xffffffffu, s0, src), e1 = __shfl_sync(0xffffffffu, e0, src);
        if (s1 <= q && q <= e1) {
          rhi = max(rhi, e1);
          rlo = min(rlo, max(s1, rclamp));
        }
      }
    }
  }
  rs.row_valid = qpos < it.qlen;
  if (rs.row_valid) {
    rs.klo = max(0, min(base_lo(q, a.window, a.chunk_size, a.chunk_lookback), rlo));
    rs.khi = min(max(base_hi(q, a.window, it.causal, it.seq_len), rhi), it.seq_len - 1);
    rs.out_row = (int64_t)(it.qstart + qpos) * a.hq + it.hk * G + row % G;
  } else {
    rs.klo = 1;
    rs.khi = 0;
    rs.out_row = 0;
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiled>(nullptr);
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

bool make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
              uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiled enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// What both tensor-core prefill kernels need besides their head_dim: bf16, no
// split, more than one query row per sequence somewhere, a GQA group that
// divides the 128-row tile, 32-bit slot and token indices, and the TMA
// descriptor encoder of the driver.
inline bool tc_prefill_ok(const AttnArgs &a) {
  const int G = a.hq / a.hkv;
  const int64_t items = (a.num_tokens / (128 / max(G, 1)) + a.num_seqs) * (int64_t)a.hkv;
  return a.dtype == SWA_DTYPE_BF16 && a.num_splits == 1 && (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) &&
         a.max_query_len > 1 && a.num_blocks * a.block_size < (int64_t)INT32_MAX &&
         a.num_tokens < (int64_t)INT32_MAX && items < (int64_t)INT32_MAX && encoder() != nullptr;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return 0;
  return n;
}

}  // namespace
}  // namespace swa
