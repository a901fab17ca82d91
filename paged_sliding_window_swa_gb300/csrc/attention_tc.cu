// Tensor-core (tcgen05 / TMEM / TMA) prefill attention over the paged KV
// cache with the sliding window and the window-clamped image mask (vLLM PR
// #53147 summary, implementation items 1-2 and the compute_tile_loop_bounds
// excerpt).
//
// One CTA = one 128-row query tile: BQ = 128 / G query positions x the G query
// heads of one kv head (GQA packing -- every K/V tile is staged once for the
// whole group).  Eleven warps:
//   warps 0,10 TMA producers of K and V: K and V tiles of N keys, gathered
//              page by page through the block table into their own rings
//              (128-byte swizzled, one box per page and 64-column chunk; pages
//              past the sequence or with a bad block id are read from outside
//              the tensor, which the TMA fills with 0).  The Q tile is copied
//              once, as soon as the block's barriers exist.
//   warp 1     tcgen05 issuer and TMEM owner: S = Q K^T into one of two TMEM S
//              buffers, then O += P V with P read from TMEM (where the
//              softmax wrote it over S) and V from shared memory (MN-major).
//   warps 2-9  softmax, two warpgroups: thread i of each owns row i (TMEM
//              lane i) and one half of the tile's columns; masks only tiles
//              not fully inside its visible interval, keeps a running max in
//              the log2 domain and rescales O in TMEM only when the max grows
//              by more than 2^8, writes P as bf16 into TMEM, and finally
//              normalises its half of O and stores out / lse.
// The key loop covers only the union of the rows' visible intervals -- the
// pruned tile range [lo, hi) of the union formula.  Every mbarrier wait is
// bounded in time; on expiry the CTA sets SWA_ERR_TIMEOUT, drains its own
// TMA loads and MMAs, frees TMEM and exits.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr uint64_t kWaitLimitNs = 200000000ull;    // 200 ms per wait: far above any real stall

template <int D_, int N_, int KST_, int VST_>
struct Cfg {
  static constexpr int D = D_;          // head dim
  static constexpr int N = N_;          // keys per K/V tile
  static constexpr int KST = KST_;      // K ring depth
  static constexpr int VST = VST_;      // V ring depth
  static constexpr int M = 128;         // query rows per CTA
  static constexpr int CH = D / 64;     // 128-byte column chunks per row
  static constexpr int Q_CHUNK = M * 128;
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int KV_CHUNK = N * 128;
  static constexpr int KV_BYTES = N * D * 2;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
  static constexpr int OFF_CTRL = OFF_V + VST * KV_BYTES;         // control block (barriers, exchange)
  static constexpr int TM_O = 0;        // TMEM columns: O [0, D), S0 [D, D+N), S1 [D+N, D+2N)
  static constexpr int TM_S = D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, N, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
  static_assert(D + 2 * N <= 512, "TMEM budget");
  static_assert(KST <= 4 && VST <= 4 && VST <= KST, "ring depths");
  static_assert((N / 16) * CH <= 32, "one warp instruction must cover a tile's boxes");
};

constexpr int kMaxSmemRanges = 64;      // image ranges staged in shared memory (more: read from L1)

struct Ctrl {
  float red[2][2][128];                  // half-row max (and, at the end, sum) exchange buffers
  int32_t ranges[2 * kMaxSmemRanges];
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t o_full, drain;
  uint64_t xch[2], xl;                   // exchange barriers of the two softmax warpgroups
  uint32_t tmem_base;
  int abort;
  int kmin, kmax;
};

template <class C>
constexpr int smem_bytes() { return C::OFF_CTRL + (int)sizeof(Ctrl); }

template <class C>
__global__ void __launch_bounds__(352, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const AttnArgs a, const int G) {
  // Everything lives in dynamic shared memory, which starts 1024-byte aligned
  // when a kernel has no static shared data (checked below): the 128-byte
  // swizzled tiles need that alignment and there is no room for slack.
  extern __shared__ __align__(1024) uint8_t dsm_ptr[];
  const uint32_t dsm = smem_u32(dsm_ptr);
  Ctrl &ctl = *reinterpret_cast<Ctrl *>(dsm_ptr + C::OFF_CTRL);
  const uint32_t q_s = dsm;
  const uint32_t k_s = dsm + C::OFF_K;
  const uint32_t v_s = dsm + C::OFF_V;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bq = C::M / G;
  const int hk = blockIdx.y;

  // ---- which sequence / query block (uniform over the CTA) ----
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
  if (ctx < 0 || (a.ctx_lens != nullptr && __ldg(a.ctx_lens + s) != ctx)) {
    if (threadIdx.x == 0) report(a.err, SWA_ERR_LENS);
    return;
  }
  if ((dsm & 1023u) != 0) {
    if (threadIdx.x == 0) report(a.err, SWA_ERR_INTERNAL);
    return;
  }

  if (threadIdx.x == 0) {
    ctl.abort = 0;
    ctl.kmin = INT_MAX;
    ctl.kmax = -1;
    mbar_init(smem_u32(&ctl.q_full), 1);
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(smem_u32(&ctl.k_full[i]), 1);
      mbar_init(smem_u32(&ctl.k_empty[i]), 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(smem_u32(&ctl.v_full[i]), 1);
      mbar_init(smem_u32(&ctl.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl.s_full[i]), 1);
      mbar_init(smem_u32(&ctl.p_full[i]), 256);
      mbar_init(smem_u32(&ctl.xch[i]), 256);
    }
    mbar_init(smem_u32(&ctl.xl), 256);
    mbar_init(smem_u32(&ctl.o_full), 1);
    mbar_init(smem_u32(&ctl.drain), 1);
    mbar_fence_init();
    // the Q copy depends only on the block's first token: start it right away
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    mbar_expect_tx(smem_u32(&ctl.q_full), C::Q_BYTES);
    for (int c = 0; c < C::CH; ++c)
      tma_load_3d(q_s + c * C::Q_CHUNK, &tm_q, c * 64, hk * G, qstart + qpos_lo, smem_u32(&ctl.q_full));
  }
  // this sequence's image ranges, staged once for the 256 interval evaluations
  const int nr = a.mm_ranges ? a.max_mm_ranges : 0;
  const bool ranges_in_smem = nr <= kMaxSmemRanges;
  const int32_t *ranges_g = a.mm_ranges ? a.mm_ranges + (int64_t)s * a.max_mm_ranges * 2 : nullptr;
  if (warp == 1 && ranges_in_smem)
    for (int i = lane; i < 2 * nr; i += 32) ctl.ranges[i] = __ldg(ranges_g + i);
  __syncthreads();

  // ---- each softmax thread: its row's visible interval; the CTA's union ----
  const bool is_softmax = warp >= 2 && warp < 10;
  const int row = 32 * (warp & 3) + lane;            // TMEM lane of this thread
  int klo = 1, khi = 0;
  bool row_valid = false;
  int64_t out_row = 0;
  if (is_softmax) {
    const int qpos = qpos_lo + row / G;
    row_valid = qpos < qlen;
    int red_lo = INT_MAX, red_hi = -1;
    if (row_valid) {
      const Span sp = visible_span(ctx + qpos, seq_len, a.window, a.causal != 0,
                                   ranges_in_smem ? ctl.ranges : ranges_g, nr);
      klo = sp.lo;
      khi = sp.hi;
      out_row = (int64_t)(qstart + qpos) * a.hq + hk * G + row % G;
      if (klo <= khi) { red_lo = klo; red_hi = khi; }
    }
    red_lo = __reduce_min_sync(0xffffffffu, red_lo);
    red_hi = __reduce_max_sync(0xffffffffu, red_hi);
    if (lane == 0) {
      atomicMin(&ctl.kmin, red_lo);
      atomicMax(&ctl.kmax, red_hi);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const int kmin = ctl.kmin, kmax = ctl.kmax;
  const int tile_lo = kmax >= kmin ? kmin / C::N : 0;
  const int n_tiles = kmax >= kmin ? kmax / C::N - tile_lo + 1 : 0;
  volatile int *abort_flag = &ctl.abort;
  const volatile int32_t *gerr = a.err;

  if (warp == 0 || warp == 10) {
    // =============================== TMA producers ==============================
    // Warp 0 streams K tiles, warp 10 streams V tiles, each through its own
    // ring.  The whole warp runs the loop: each lane resolves the cache slot of
    // one box (one page, or part of one) through the block table, 32 boxes per
    // batch and one batch ahead, and one warp instruction then issues every
    // box of a tile (lane i*CH + c copies box i, 64-column chunk c).
    const bool is_v = warp == 10;
    const int ST = is_v ? C::VST : C::KST;
    int issued = 0;
    bool ok = true;
    if (n_tiles > 0) {
      const int R = min(a.block_size, C::N);             // rows per box
      const int boxes = C::N / R;                         // boxes per tile
      const int total_boxes = n_tiles * boxes;
      const int oob = (int)(a.num_blocks * a.block_size); // first slot outside the cache: zero fill
      const int32_t *bt = a.block_table + (int64_t)s * a.bt_stride;
      auto resolve = [&](int b) -> int {
        const int k = tile_lo * C::N + b * R;
        int slot = oob;
        if (b < total_boxes && k < seq_len) {
          const int page = k / a.block_size;
          const int32_t blk = page < a.bt_stride ? __ldg(bt + page) : -1;
          if (blk >= 0 && blk < a.num_blocks) slot = blk * a.block_size + (k - page * a.block_size);
          else if (!is_v) report(a.err, SWA_ERR_BLOCK_ID);
        }
        return slot;
      };
      int batch = 0;
      int prv = oob, cur = resolve(lane), nxt = resolve(32 + lane);
      auto advance = [&](int b_max) {                     // warp-uniform
        while (b_max >= (batch + 1) * 32) {
          prv = cur;
          cur = nxt;
          ++batch;
          nxt = resolve((batch + 1) * 32 + lane);
        }
      };
      auto slot_lane = [&](int b) -> int {                // per-lane b: current batch, or the one before
        const int from_cur = __shfl_sync(0xffffffffu, cur, (b - batch * 32) & 31);
        const int from_prv = __shfl_sync(0xffffffffu, prv, (b - (batch - 1) * 32) & 31);
        return b >= batch * 32 ? from_cur : from_prv;
      };
      const CUtensorMap *map = is_v ? &tm_v : &tm_k;
      auto issue = [&](int t) {
        const int st = t % ST;
        const uint32_t full = smem_u32(is_v ? &ctl.v_full[st] : &ctl.k_full[st]);
        const uint32_t dst = (is_v ? v_s : k_s) + st * C::KV_BYTES;
        if (lane == 0) mbar_expect_tx(full, C::KV_BYTES);
        __syncwarp();
        advance(t * boxes + boxes - 1);
        const int i = min(lane / C::CH, boxes - 1), c = lane % C::CH;
        const int slot = slot_lane(t * boxes + i);
        if (lane < boxes * C::CH) tma_load_3d(dst + c * C::KV_CHUNK + i * R * 128, map, c * 64, hk, slot, full);
      };
      // fill the ring, then refill each stage as soon as its consumer (QK_j
      // for K, PV_j for V) has released it
      issued = min(ST, n_tiles);
      for (int t = 0; t < issued; ++t) issue(t);
      for (int j = 0; j + ST < n_tiles; ++j) {
        const uint32_t empty = smem_u32(is_v ? &ctl.v_empty[j % ST] : &ctl.k_empty[j % ST]);
        ok = __all_sync(0xffffffffu, mbar_wait(empty, (j / ST) & 1, abort_flag, gerr, kWaitLimitNs));
        if (!ok) break;
        issue(j + ST);
        issued = j + ST + 1;
      }
      if (!ok && lane == 0) {
        *abort_flag = 1;
        report(a.err, SWA_ERR_TIMEOUT);
      }
    }
    // drain: every load issued by this warp must have landed before the CTA exits
    if (lane == 0) {
      for (int t = max(0, issued - ST); t < issued; ++t)
        mbar_wait(smem_u32(is_v ? &ctl.v_full[t % ST] : &ctl.k_full[t % ST]), (t / ST) & 1, nullptr, nullptr,
                  kWaitLimitNs);
      if (!is_v) mbar_wait(smem_u32(&ctl.q_full), 0, nullptr, nullptr, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // =============================== MMA issuer =================================
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait(smem_u32(&ctl.q_full), 0, abort_flag, gerr, kWaitLimitNs);
      tc_fence_after();
      auto issue_qk = [&](int j) -> bool {
        const int st = j % C::KST;
        if (!mbar_wait(smem_u32(&ctl.k_full[st]), (j / C::KST) & 1, abort_flag, gerr, kWaitLimitNs)) return false;
        tc_fence_after();
        const uint32_t d = tmem + C::TM_S + (j & 1) * C::N;
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;     // 16-column step inside the 128-byte swizzle row
          const uint64_t ad = smem_desc_sw128(q_s + (kk >> 2) * C::Q_CHUNK + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(k_s + st * C::KV_BYTES + (kk >> 2) * C::KV_CHUNK + off, 16, 1024);
          mma_ss(d, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&ctl.s_full[j & 1]));
        mma_commit(smem_u32(&ctl.k_empty[st]));
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles && !issue_qk(j + 1)) { ok = false; break; }
        const int st = j % C::VST;
        if (!mbar_wait(smem_u32(&ctl.p_full[j & 1]), (j >> 1) & 1, abort_flag, gerr, kWaitLimitNs) ||
            !mbar_wait(smem_u32(&ctl.v_full[st]), (j / C::VST) & 1, abort_flag, gerr, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t p_t = tmem + C::TM_S + (j & 1) * C::N;
#pragma unroll
        for (int kk = 0; kk < C::N / 16; ++kk) {
          const uint64_t bd = smem_desc_sw128(v_s + st * C::KV_BYTES + kk * 16 * 128, C::KV_CHUNK, 1024);
          mma_ts(tmem + C::TM_O, p_t + kk * 8, bd, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&ctl.v_empty[st]));
        mma_commit(smem_u32(&ctl.o_full));
      }
      if (!ok) {
        *abort_flag = 1;
        report(a.err, SWA_ERR_TIMEOUT);
      }
      // every MMA issued so far must finish before TMEM is released
      mma_commit(smem_u32(&ctl.drain));
      mbar_wait(smem_u32(&ctl.drain), 0, nullptr, nullptr, kWaitLimitNs);
    }
  } else if (is_softmax) {
    // =============================== softmax ====================================
    // Two warpgroups share every row: warpgroup h owns S columns
    // [h*N/2, (h+1)*N/2) and O columns [h*D/2, (h+1)*D/2).  Both keep the
    // same running max (half-row maxima are exchanged through shared memory
    // once per tile, ordered by a bounded mbarrier) and a partial row sum.
    constexpr int NH = C::N / 2;
    constexpr int DH = C::D / 2;
    const int h = (warp - 2) >> 2;
    const int sid = threadIdx.x - 64;                    // 0..255 over both warpgroups
    const uint32_t lane_t = (uint32_t)(32 * (warp & 3)) << 16;
    const float sl2 = a.scale * kLog2e;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int kc0 = (tile_lo + j) * C::N + h * NH;     // key of this warpgroup's first column
      ok = mbar_wait(smem_u32(&ctl.s_full[j & 1]), (j >> 1) & 1, abort_flag, gerr, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t raw[NH];
#pragma unroll
      for (int c = 0; c < NH / 32; ++c)
        tmem_ld32(tmem + lane_t + C::TM_S + (j & 1) * C::N + h * NH + 32 * c,
                  *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * c));
      tmem_wait_ld();
      float x[NH];
      const bool full = klo <= kc0 && khi >= kc0 + NH - 1;
      if (__all_sync(0xffffffffu, full)) {
#pragma unroll
        for (int c = 0; c < NH; ++c) x[c] = __uint_as_float(raw[c]) * sl2;
      } else {
#pragma unroll
        for (int c = 0; c < NH; ++c)
          x[c] = (kc0 + c >= klo && kc0 + c <= khi) ? __uint_as_float(raw[c]) * sl2 : -INFINITY;
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < NH; ++c) m4[c & 3] = fmaxf(m4[c & 3], x[c]);
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      ctl.red[j & 1][h][row] = mx;
      mbar_arrive(smem_u32(&ctl.xch[j & 1]));
      ok = mbar_wait(smem_u32(&ctl.xch[j & 1]), (j >> 1) & 1, abort_flag, gerr, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      mx = fmaxf(mx, ctl.red[j & 1][h ^ 1][row]);
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + 8.f;             // also true on the first visible tile
      // PV_{j-1} is confirmed exactly once per tile (here if O must be
      // rescaled, else before P_j is published), so this thread is never more
      // than one o_full phase behind and every parity wait is unambiguous.
      bool pv_prev_done = (j == 0);
      if (__any_sync(0xffffffffu, need)) {               // same decision in both warpgroups
        const float m_next = need ? m_new : m_used;
        const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_next);
        if (j > 0) {
          ok = mbar_wait(smem_u32(&ctl.o_full), (j - 1) & 1, abort_flag, gerr, kWaitLimitNs);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          pv_prev_done = true;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DH / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_t + C::TM_O + h * DH + 32 * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(tmem + lane_t + C::TM_O + h * DH + 32 * c, r);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_used = m_next;
      }
      const float ms = (m_used == -INFINITY) ? 0.f : m_used;
      uint32_t pk[NH / 2];
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < NH / 2; ++c) {
        const float p0 = ex2(x[2 * c] - ms), p1 = ex2(x[2 * c + 1] - ms);
        s4[c & 3] += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
      l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
      const int kt0 = (tile_lo + j) * C::N;
      if (kt0 + C::N > seq_len) {
        // keys past the sequence end: their V rows may hold anything; zero them
        const int st = j % C::VST;
        ok = mbar_wait(smem_u32(&ctl.v_full[st]), (j / C::VST) & 1, abort_flag, gerr, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const int r0 = max(0, seq_len - kt0);
        const int n16 = (C::N - r0) * 8 * C::CH;
        for (int i = sid; i < n16; i += 256) {
          const int c = i / ((C::N - r0) * 8), rem = i % ((C::N - r0) * 8);
          uint4 *dst = reinterpret_cast<uint4 *>(dsm_ptr + C::OFF_V + st * C::KV_BYTES + c * C::KV_CHUNK +
                                                 (r0 + rem / 8) * 128 + (rem % 8) * 16);
          *dst = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      if (!pv_prev_done) {
        ok = mbar_wait(smem_u32(&ctl.o_full), (j - 1) & 1, abort_flag, gerr, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
#pragma unroll
      for (int c = 0; c < NH / 2; c += 16)
        tmem_st16(tmem + lane_t + C::TM_S + (j & 1) * C::N + h * (NH / 2) + c, pk + c);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&ctl.p_full[j & 1]));
    }
    if (ok && n_tiles > 0) {
      ok = mbar_wait(smem_u32(&ctl.o_full), (n_tiles - 1) & 1, abort_flag, gerr, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      // full row sum = both halves; buffer n_tiles & 1 was last read at tile
      // n_tiles - 2, before every thread passed the exchange of tile n_tiles - 1
      ctl.red[n_tiles & 1][h][row] = l;
      mbar_arrive(smem_u32(&ctl.xl));
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.xl), 0, abort_flag, gerr, kWaitLimitNs));
      l += ctl.red[n_tiles & 1][h ^ 1][row];
    }
    if (!ok) {
      *abort_flag = 1;
      report(a.err, SWA_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + out_row * C::D + h * DH;
#pragma unroll 1
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_t + C::TM_O + h * DH + 32 * c, r);
        tmem_wait_ld();
        if (row_valid) {
          uint4 v[4];
          uint32_t *w = reinterpret_cast<uint32_t *>(v);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
          uint4 *dst = reinterpret_cast<uint4 *>(o + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = v[e];
        }
      }
      if (row_valid && h == 0 && a.lse != nullptr)
        a.lse[out_row] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
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

template <class C>
cudaError_t run(const AttnArgs &a, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  const int bq = C::M / G;
  const int R = a.block_size < C::N ? a.block_size : C::N;
  CUtensorMap mq, mk, mv;
  const uint64_t esz = 2;
  if (!make_map(&mq, a.q, C::D, a.hq, a.num_tokens, C::D * esz, (uint64_t)a.hq * C::D * esz, 64, G, bq) ||
      !make_map(&mk, a.k_cache, C::D, a.hkv, (uint64_t)a.num_blocks * a.block_size, C::D * esz,
                (uint64_t)a.hkv * C::D * esz, 64, 1, R) ||
      !make_map(&mv, a.v_cache, C::D, a.hkv, (uint64_t)a.num_blocks * a.block_size, C::D * esz,
                (uint64_t)a.hkv * C::D * esz, 64, 1, R))
    return cudaErrorInvalidValue;
  constexpr int smem = smem_bytes<C>();
  static_assert(smem <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = a.num_tokens / bq + a.num_seqs;
  dim3 grid((unsigned)blocks, (unsigned)a.hkv);
  attn_tc_kernel<C><<<grid, 352, smem, st>>>(mq, mk, mv, a, G);
  return cudaGetLastError();
}

using Cfg256 = Cfg<256, 64, 3, 2>;     // 64 KB Q + 3 x 32 KB K + 2 x 32 KB V
using Cfg128 = Cfg<128, 128, 3, 3>;    // 32 KB Q + 3 x 32 KB K + 3 x 32 KB V

}  // namespace

bool tc_supported(const AttnArgs &a) {
  const int G = a.hq / a.hkv;
  return a.dtype == SWA_DTYPE_BF16 && (a.head_dim == 128 || a.head_dim == 256) && a.num_splits == 1 &&
         (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) && a.max_query_len > 1 &&
         a.num_blocks * a.block_size < (int64_t)INT32_MAX && a.num_tokens < (int64_t)INT32_MAX &&
         encoder() != nullptr;
}

cudaError_t launch_attention_tc(const AttnArgs &a, cudaStream_t st) {
  return a.head_dim == 256 ? run<Cfg256>(a, st) : run<Cfg128>(a, st);
}

}  // namespace swa
