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

// How a position becomes (page, offset).  kPlainPow2: block_size == 1 << shift,
// the usual case -- a shift and a mask instead of a 64-bit division, which the
// GPU does in software.  kPlain: any block size.  kCp: one rank of an
// interleaved context-parallel cache (the article's section 3.1, steps 1-5).
// kCpPow2: the same with every CP size a power of two (shifts and masks).
enum Mode { kPlainPow2 = 0, kPlain = 1, kCp = 2, kCpPow2 = 3 };

struct Geom {
  int32_t block_size, shift;
  int64_t vbs;                          // CP: kv_cache_block_size * world size (< 2^31)
  int32_t world, rank, interleave, blocks_per_kv_block;
  int32_t vbs_shift, inter_shift, wi_shift;   // kCpPow2: log2 of vbs, interleave, world * interleave
};

template <bool kVec, int kMode, bool kDerive>
__global__ void __launch_bounds__(kThreads)
slot_mapping_kernel(const int32_t *__restrict__ qsl, const int64_t *__restrict__ pos,
                    const int32_t *__restrict__ ctx, const int32_t *__restrict__ bt, int64_t stride, const Geom g,
                    int32_t num_reqs, int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                    int32_t *__restrict__ out, int32_t *__restrict__ err) {
  const int32_t block_size = g.block_size;
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
    // positions: given, or (kDerive) the request's context length plus the
    // token's index in the request (filled below, once the request is known)
    int64_t p[kTokPerThread];
    if (kDerive) {
#pragma unroll
      for (int i = 0; i < kTokPerThread; ++i) p[i] = 0;
    } else if (kVec && t0 + kTokPerThread <= num_tokens) {
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
    int32_t r_start = __ldg(qsl + r), r_end = __ldg(qsl + r + 1);
    int32_t r_ctx = kDerive ? __ldg(ctx + r) : 0;
    if (kDerive) {
#pragma unroll
      for (int i = 0; i < kTokPerThread; ++i) p[i] = (int64_t)r_ctx + (t0 + i - r_start);
    }
    // Fast path: the 8 tokens are consecutive positions of one request that
    // stay inside one page (and, for a CP cache, one interleave run of one
    // rank): one ownership test and one block-table read serve all of them.
    bool done = false;
    if (t0 >= r_start && t0 + kTokPerThread <= r_end && p[0] >= 0 && p[kTokPerThread - 1] - p[0] == kTokPerThread - 1) {
      bool consecutive = true;
#pragma unroll
      for (int i = 1; i < kTokPerThread - 1; ++i) consecutive &= p[i] == p[0] + i;
      if (consecutive) {
        const int64_t ps = p[0];
        int64_t page = -1, off = 0;
        bool mine = true, one_page = false;
        if (kMode == kCpPow2) {
          const int64_t v_idx = ps >> g.vbs_shift;
          const int32_t v_off = (int32_t)(ps & (g.vbs - 1));
          if ((v_off & (g.interleave - 1)) + kTokPerThread <= g.interleave) {
            mine = ((v_off >> g.inter_shift) & (g.world - 1)) == g.rank;
            const int32_t local = ((v_off >> g.wi_shift) << g.inter_shift) | (v_off & (g.interleave - 1));
            page = v_idx * g.blocks_per_kv_block + (local >> g.shift);
            off = local & (block_size - 1);
            one_page = off + kTokPerThread <= block_size;
          }
        } else if (kMode == kCp) {
          if (ps <= INT32_MAX) {
            const uint32_t v_idx = (uint32_t)ps / (uint32_t)g.vbs;
            const uint32_t v_off = (uint32_t)ps - v_idx * (uint32_t)g.vbs;
            const uint32_t I = (uint32_t)g.interleave, Wd = (uint32_t)g.world;
            if (v_off % I + kTokPerThread <= I) {
              mine = (v_off / I) % Wd == (uint32_t)g.rank;
              const uint32_t local = (v_off / (Wd * I)) * I + v_off % I;
              page = (int64_t)v_idx * g.blocks_per_kv_block + local / (uint32_t)block_size;
              off = local % (uint32_t)block_size;
              one_page = off + kTokPerThread <= block_size;
            }
          }
        } else if (kMode == kPlainPow2) {
          page = ps >> g.shift;
          off = ps & (block_size - 1);
          one_page = off + kTokPerThread <= block_size;
        } else {
          page = ps / block_size;
          off = ps - page * block_size;
          one_page = off + kTokPerThread <= block_size;
        }
        if (!mine) {                                         // another rank's tokens
#pragma unroll
          for (int i = 0; i < kTokPerThread; ++i) res[i] = pad_id;
          done = true;
        } else if (one_page && page < stride) {
          const int32_t base = (int32_t)((int64_t)__ldg(bt + (int64_t)r * stride + page) * block_size + off);
#pragma unroll
          for (int i = 0; i < kTokPerThread; ++i) res[i] = base + i;
          done = true;
        }
      }
    }
    int64_t last = -1;                                       // (request, page) of the last lookup
    int32_t blk = 0;
#pragma unroll
    for (int i = 0; i < kTokPerThread && !done; ++i) {
      const int64_t t = t0 + i;
      res[i] = pad_id;
      if (t >= num_tokens) continue;
      while (r + 1 < num_reqs && t >= r_end) {
        ++r;
        r_start = r_end;
        r_end = __ldg(qsl + r + 1);
        if (kDerive) r_ctx = __ldg(ctx + r);
      }
      if (t < r_start || t >= r_end) continue;              // outside every request
      const int64_t ps = kDerive ? (int64_t)r_ctx + (t - r_start) : p[i];   // (p[] of the fast path is r's)
      if (ps < 0) { report(err, SWA_ERR_POSITION); continue; }
      int64_t page, off;
      if (kMode == kCpPow2) {
        const int64_t v_idx = ps >> g.vbs_shift;
        const int32_t v_off = (int32_t)(ps & (g.vbs - 1));
        if (((v_off >> g.inter_shift) & (g.world - 1)) != g.rank) continue;   // another rank's token
        const int32_t local = ((v_off >> g.wi_shift) << g.inter_shift) | (v_off & (g.interleave - 1));
        page = v_idx * g.blocks_per_kv_block + (local >> g.shift);
        off = local & (block_size - 1);
      } else if (kMode == kCp) {
        // 32-bit divisions whenever the position fits (the 64-bit ones are software routines)
        int64_t v_idx;
        uint32_t v_off;
        if (ps <= INT32_MAX) {
          v_idx = (uint32_t)ps / (uint32_t)g.vbs;
          v_off = (uint32_t)ps - (uint32_t)v_idx * (uint32_t)g.vbs;
        } else {
          v_idx = ps / g.vbs;
          v_off = (uint32_t)(ps - v_idx * g.vbs);
        }
        const uint32_t I = (uint32_t)g.interleave, Wd = (uint32_t)g.world;
        if ((v_off / I) % Wd != (uint32_t)g.rank) continue;          // another rank's token
        const uint32_t local = (v_off / (Wd * I)) * I + v_off % I;
        page = v_idx * g.blocks_per_kv_block + local / (uint32_t)block_size;
        off = local % (uint32_t)block_size;
      } else if (kMode == kPlainPow2) {
        page = ps >> g.shift;
        off = ps & (block_size - 1);
      } else {
        page = ps / block_size;
        off = ps - page * block_size;
      }
      if (page >= stride) { report(err, SWA_ERR_POSITION); continue; }
      const int64_t idx = (int64_t)r * stride + page;
      if (idx != last) {                                     // neighbouring tokens mostly share a page
        blk = __ldg(bt + idx);
        last = idx;
      }
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

cudaError_t launch_slot_mapping(const int32_t *qsl, const int64_t *pos, const int32_t *ctx, const int32_t *bt,
                                int64_t stride, int32_t block_size, int32_t num_reqs,
                                int64_t num_tokens, int64_t max_num_tokens, int32_t pad_id,
                                int32_t *out, int32_t *err, cudaStream_t st, const CpArgs *cp) {
  const int64_t work = max(ceil_div(max_num_tokens, kTokPerThread), (int64_t)num_reqs);
  if (work == 0) return cudaSuccess;
  const unsigned grid = (unsigned)ceil_div(work, kThreads);
  const bool vec = ((uintptr_t)pos % 16 == 0) && ((uintptr_t)out % 16 == 0);   // t0 is a multiple of 8 (a null pos is aligned)
  Geom g{};
  g.block_size = block_size;
  while (g.shift < 30 && (1 << g.shift) < block_size) ++g.shift;
  int mode = (1 << g.shift) == block_size ? kPlainPow2 : kPlain;
  if (cp != nullptr) {
    g.vbs = (int64_t)cp->kv_cache_block_size * cp->world;
    g.world = cp->world;
    g.rank = cp->rank;
    g.interleave = cp->interleave;
    g.blocks_per_kv_block = cp->kv_cache_block_size / block_size;
    auto log2_exact = [](int64_t x) -> int {       // -1 unless x is a power of two
      int k = 0;
      while (k < 62 && ((int64_t)1 << k) < x) ++k;
      return ((int64_t)1 << k) == x ? k : -1;
    };
    g.vbs_shift = log2_exact(g.vbs);
    g.inter_shift = log2_exact(g.interleave);
    g.wi_shift = log2_exact((int64_t)g.world * g.interleave);
    const bool pow2 = mode == kPlainPow2 && g.vbs_shift >= 0 && g.inter_shift >= 0 && g.wi_shift >= 0 &&
                      log2_exact(g.world) >= 0;
    mode = pow2 ? kCpPow2 : kCp;
  }
  using K = void (*)(const int32_t *, const int64_t *, const int32_t *, const int32_t *, int64_t, const Geom,
                     int32_t, int64_t, int64_t, int32_t, int32_t *, int32_t *);
  const K table[2][4] = {{slot_mapping_kernel<false, kPlainPow2, false>, slot_mapping_kernel<false, kPlain, false>,
                          slot_mapping_kernel<false, kCp, false>, slot_mapping_kernel<false, kCpPow2, false>},
                         {slot_mapping_kernel<true, kPlainPow2, false>, slot_mapping_kernel<true, kPlain, false>,
                          slot_mapping_kernel<true, kCp, false>, slot_mapping_kernel<true, kCpPow2, false>}};
  // derived positions (plain mapping only): no position reads; vector stores when out is aligned
  const K derived[2][2] = {{slot_mapping_kernel<false, kPlainPow2, true>, slot_mapping_kernel<false, kPlain, true>},
                           {slot_mapping_kernel<true, kPlainPow2, true>, slot_mapping_kernel<true, kPlain, true>}};
  const K fn = (pos == nullptr && cp == nullptr) ? derived[(uintptr_t)out % 16 == 0 ? 1 : 0][mode]
                                                 : table[vec ? 1 : 0][mode];
  fn<<<grid, kThreads, 0, st>>>(qsl, pos, ctx, bt, stride, g, num_reqs, num_tokens,
                                                       max_num_tokens, pad_id, out, err);
  return cudaGetLastError();
}

}  // namespace swa
