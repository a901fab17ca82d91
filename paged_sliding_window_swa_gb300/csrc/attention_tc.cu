// Tensor-core (tcgen05 / TMEM / TMA) prefill attention over the paged KV
// cache with the sliding window and the window-clamped image mask (vLLM PR
// #53147 summary, implementation items 1-2 and the compute_tile_loop_bounds
// excerpt).
//
// One CTA = one 128-row query tile: BQ = 128 / G query positions x the G query
// heads of one kv head (GQA packing -- every K/V tile is staged once for the
// whole group).  The key loop walks 128-key tiles over the union of the rows'
// visible intervals (the pruned tile range of the union formula).
//
// Shared memory: the Q tile (TMA, 128-byte swizzled, K-major) and two rings of
// 32 KB units (for head_dim 256; 16 KB for 128): a K unit holds one half of
// head_dim for all 128 keys of a tile, a V unit holds all of head_dim for one
// 64-key half of a tile.  So QK_j consumes two K units and PV_j two V units,
// and each unit is recycled as soon as its half of the MMA work is done.
// TMEM (512 columns): O [0, D), S buffers [D, D+128) and [D+128, D+256) in
// fp32; the softmax overwrites the front half of S_j with P_j as bf16 pairs,
// which the PV MMA reads as its A operand.
//
// Eleven warps:
//   warp 0     K producer, warp 10 V producer: every lane resolves the cache
//              slot of one page box through the block table (32 boxes per
//              batch, one batch ahead) and one warp instruction issues a whole
//              unit's boxes (one per page and 64-column chunk); pages past the
//              sequence or with a bad block id are read from outside the
//              tensor, which the TMA fills with 0.  Thread 0 copies Q as soon
//              as the barriers exist.
//   warp 1     tcgen05 issuer and TMEM owner: QK_0, QK_1, then per tile
//              PV_j (once P_j is written) and QK_{j+2}.
//   warps 2-9  softmax, two warpgroups: thread i of each owns row i (TMEM lane
//              i) and one half of the tile's columns; the half-row maxima are
//              exchanged through shared memory once per tile.  Masks only tiles
//              not fully inside the row's visible interval, keeps the running
//              max in the log2 domain and rescales O in TMEM only when the max
//              grows by more than 2^8, and at the end normalises its half of O.
// Every mbarrier wait is bounded in time; on expiry the CTA sets
// SWA_ERR_TIMEOUT, drains its own TMA loads and MMAs, frees TMEM and exits.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

constexpr uint64_t kWaitLimitNs = 200000000ull;    // 200 ms per wait: far above any real stall
constexpr int kMaxSmemRanges = 64;                 // image ranges staged in shared memory
constexpr int kMaxUnits = 8;                       // ring slots per operand

template <int D_, int KSU_, int VSU_>
struct Cfg {
  static constexpr int D = D_;          // head dim
  static constexpr int N = 128;         // keys per tile
  static constexpr int M = 128;         // query rows per CTA
  static constexpr int CH = D / 64;     // 128-byte column chunks per row
  static constexpr int KSU = KSU_;      // K ring slots (units)
  static constexpr int VSU = VSU_;      // V ring slots (units)
  static constexpr int Q_CHUNK = M * 128;
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int UNIT = N * D;                 // bytes of a K or V unit (= 64 keys x D x 2)
  static constexpr int KU_CH = CH / 2;               // chunks per K unit (half of head_dim)
  static constexpr int KU_CHUNK = N * 128;           // bytes per chunk in a K unit (128 keys)
  static constexpr int VU_KEYS = N / 2;              // keys per V unit
  static constexpr int VU_CHUNK = VU_KEYS * 128;     // bytes per chunk in a V unit
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + KSU * UNIT;
  static constexpr int OFF_CTRL = OFF_V + VSU * UNIT;
  static constexpr int TM_O = 0;        // TMEM columns: O [0, D), S buffer b at [D + b*N, D + (b+1)*N)
  static constexpr int TM_S = D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, N, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
  static_assert(D + 2 * N <= 512, "TMEM budget");
  static_assert(KSU <= kMaxUnits && VSU <= kMaxUnits && KSU >= 2 && VSU >= 2, "ring sizes");
  static_assert((N / 16) * KU_CH <= 32 && (VU_KEYS / 16) * CH <= 32, "one warp instruction per unit");
};

struct Ctrl {
  float red[2][2][128];                  // half-row max (and, at the end, sum) exchange buffers
  int32_t ranges[2 * kMaxSmemRanges];
  uint64_t q_full;
  uint64_t k_full[kMaxUnits], k_empty[kMaxUnits], v_full[kMaxUnits], v_empty[kMaxUnits];
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
  const uint32_t q_s = dsm + C::OFF_Q;
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
    for (int i = 0; i < C::KSU; ++i) {
      mbar_init(smem_u32(&ctl.k_full[i]), 1);
      mbar_init(smem_u32(&ctl.k_empty[i]), 1);
    }
    for (int i = 0; i < C::VSU; ++i) {
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
    const bool is_v = warp == 10;
    const int SU = is_v ? C::VSU : C::KSU;
    const int n_units = 2 * n_tiles;               // unit u = 2*tile + half
    int issued = 0;
    bool ok = true;
    if (n_tiles > 0) {
      // K units cover 128 keys, V units 64 keys; a box is one page (or a
      // 128-key part of a bigger page)
      const int unit_keys = is_v ? C::VU_KEYS : C::N;
      const int R = min(a.block_size, unit_keys);    // rows per box
      const int boxes = unit_keys / R;               // boxes per unit (per chunk)
      const int uch = is_v ? C::CH : C::KU_CH;       // chunks per unit
      const int total_boxes = (n_tiles * C::N) / R;
      const int oob = (int)(a.num_blocks * a.block_size);
      const int32_t *bt = a.block_table + (int64_t)s * a.bt_stride;
      auto resolve = [&](int b) -> int {           // slot of the first key of box b
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
      auto advance = [&](int b_max) {               // warp-uniform
        while (b_max >= (batch + 1) * 32) {
          prv = cur;
          cur = nxt;
          ++batch;
          nxt = resolve((batch + 1) * 32 + lane);
        }
      };
      auto slot_lane = [&](int b) -> int {          // per-lane b: current batch, or the one before
        const int from_cur = __shfl_sync(0xffffffffu, cur, (b - batch * 32) & 31);
        const int from_prv = __shfl_sync(0xffffffffu, prv, (b - (batch - 1) * 32) & 31);
        return b >= batch * 32 ? from_cur : from_prv;
      };
      const CUtensorMap *map = is_v ? &tm_v : &tm_k;
      auto issue = [&](int u) {
        const int t = u >> 1, half = u & 1, slot_i = u % SU;
        const uint32_t full = smem_u32(is_v ? &ctl.v_full[slot_i] : &ctl.k_full[slot_i]);
        const uint32_t dst = (is_v ? v_s : k_s) + slot_i * C::UNIT;
        if (lane == 0) mbar_expect_tx(full, C::UNIT);
        __syncwarp();
        // K: unit = head_dim half `half` of tile t's 128 keys; V: key half `half`
        const int b0 = is_v ? (2 * t + half) * boxes : t * boxes;
        advance(b0 + boxes - 1);
        const int i = min(lane / uch, boxes - 1), c = lane % uch;
        const int slot = slot_lane(b0 + i);
        const int x = (is_v ? c : half * C::KU_CH + c) * 64;
        const uint32_t d = dst + c * (is_v ? C::VU_CHUNK : C::KU_CHUNK) + i * R * 128;
        if (lane < boxes * uch) tma_load_3d(d, map, x, hk, slot, full);
      };
      // fill the ring, then refill a slot as soon as its half of QK (for K) or
      // of PV (for V) has finished with it
      issued = min(SU, n_units);
      for (int u = 0; u < issued; ++u) issue(u);
      for (int u = SU; u < n_units; ++u) {
        const uint32_t empty = smem_u32(is_v ? &ctl.v_empty[u % SU] : &ctl.k_empty[u % SU]);
        ok = __all_sync(0xffffffffu, mbar_wait(empty, ((u / SU) - 1) & 1, abort_flag, gerr, kWaitLimitNs));
        if (!ok) break;
        issue(u);
        issued = u + 1;
      }
      if (!ok && lane == 0) {
        *abort_flag = 1;
        report(a.err, SWA_ERR_TIMEOUT);
      }
    }
    // drain: every load issued by this warp must have landed before the CTA exits
    if (lane == 0) {
      for (int u = max(0, issued - SU); u < issued; ++u)
        mbar_wait(smem_u32(is_v ? &ctl.v_full[u % SU] : &ctl.k_full[u % SU]), (u / SU) & 1, nullptr, nullptr,
                  kWaitLimitNs);
      if (!is_v) mbar_wait(smem_u32(&ctl.q_full), 0, nullptr, nullptr, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // =============================== MMA issuer =================================
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait(smem_u32(&ctl.q_full), 0, abort_flag, gerr, kWaitLimitNs);
      tc_fence_after();
      auto issue_qk = [&](int j) -> bool {
        const uint32_t d = tmem + C::TM_S + (j & 1) * C::N;
        for (int half = 0; half < 2; ++half) {
          const int u = 2 * j + half, slot = u % C::KSU;
          if (!mbar_wait(smem_u32(&ctl.k_full[slot]), (u / C::KSU) & 1, abort_flag, gerr, kWaitLimitNs))
            return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::D / 32; ++kk) {     // 16-column steps over this half of head_dim
            const uint32_t off = (kk & 3) * 32;         // inside the 128-byte swizzle row
            const int cl = kk >> 2;                     // chunk within the unit
            const uint64_t ad = smem_desc_sw128(q_s + (half * C::KU_CH + cl) * C::Q_CHUNK + off, 16, 1024);
            const uint64_t bd = smem_desc_sw128(k_s + slot * C::UNIT + cl * C::KU_CHUNK + off, 16, 1024);
            mma_ss(d, ad, bd, C::IDESC_QK, (half > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&ctl.k_empty[slot]));
        }
        mma_commit(smem_u32(&ctl.s_full[j & 1]));
        return true;
      };
      // S buffer j & 1 last held P_{j-2}, whose PV was issued before QK_j;
      // tcgen05 ops from one thread run in issue order
      if (ok) ok = issue_qk(0);
      if (ok && n_tiles > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (!mbar_wait(smem_u32(&ctl.p_full[j & 1]), (j >> 1) & 1, abort_flag, gerr, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const uint32_t p_t = tmem + C::TM_S + (j & 1) * C::N;
        for (int half = 0; half < 2 && ok; ++half) {
          const int u = 2 * j + half, slot = u % C::VSU;
          if (!mbar_wait(smem_u32(&ctl.v_full[slot]), (u / C::VSU) & 1, abort_flag, gerr, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::VU_KEYS / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(v_s + slot * C::UNIT + kk * 16 * 128, C::VU_CHUNK, 1024);
            mma_ts(tmem + C::TM_O, p_t + (half * (C::VU_KEYS / 16) + kk) * 8, bd, C::IDESC_PV,
                   (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&ctl.v_empty[slot]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&ctl.o_full));
        if (j + 2 < n_tiles && !issue_qk(j + 2)) { ok = false; break; }
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
      const int kt0 = (tile_lo + j) * C::N;
      const int kc0 = kt0 + h * NH;                      // key of this warpgroup's first column
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
      if (!pv_prev_done) {
        ok = mbar_wait(smem_u32(&ctl.o_full), (j - 1) & 1, abort_flag, gerr, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      if (kt0 + C::N > seq_len) {
        // keys past the sequence end: their V rows may hold anything; zero
        // them.  PV_{j-1} is done, so every earlier unit of each V slot has
        // been consumed and the v_full parity below is unambiguous.
        for (int half = 0; half < 2 && ok; ++half) {
          const int k0 = kt0 + half * C::VU_KEYS;
          if (k0 + C::VU_KEYS <= seq_len) continue;
          const int u = 2 * j + half, slot = u % C::VSU;
          ok = mbar_wait(smem_u32(&ctl.v_full[slot]), (u / C::VSU) & 1, abort_flag, gerr, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const int r0 = max(0, seq_len - k0);
          const int n16 = (C::VU_KEYS - r0) * 8 * C::CH;
          for (int i = sid; i < n16; i += 256) {
            const int c = i / ((C::VU_KEYS - r0) * 8), rem = i % ((C::VU_KEYS - r0) * 8);
            uint4 *dst = reinterpret_cast<uint4 *>(dsm_ptr + C::OFF_V + slot * C::UNIT + c * C::VU_CHUNK +
                                                   (r0 + rem / 8) * 128 + (rem % 8) * 16);
            *dst = make_uint4(0, 0, 0, 0);
          }
        }
        if (!ok) break;
        fence_proxy_async_smem();
      }
#pragma unroll
      for (int c = 0; c < NH / 2; c += 32)
        tmem_st32(tmem + lane_t + C::TM_S + (j & 1) * C::N + h * (NH / 2) + c,
                  *reinterpret_cast<const uint32_t(*)[32]>(pk + c));
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
  CUtensorMap mq, mk, mv;
  const uint64_t esz = 2;
  const uint64_t slots = (uint64_t)a.num_blocks * a.block_size;
  if (!make_map(&mq, a.q, C::D, a.hq, a.num_tokens, C::D * esz, (uint64_t)a.hq * C::D * esz, 64, G, bq) ||
      !make_map(&mk, a.k_cache, C::D, a.hkv, slots, C::D * esz, (uint64_t)a.hkv * C::D * esz, 64, 1,
                (uint32_t)min(a.block_size, C::N)) ||
      !make_map(&mv, a.v_cache, C::D, a.hkv, slots, C::D * esz, (uint64_t)a.hkv * C::D * esz, 64, 1,
                (uint32_t)min(a.block_size, C::VU_KEYS)))
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

using Cfg256 = Cfg<256, 2, 3>;    // 64 KB Q + 2 K + 3 V units of 32 KB
using Cfg128 = Cfg<128, 6, 6>;    // 32 KB Q + 6 K + 6 V units of 16 KB

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
