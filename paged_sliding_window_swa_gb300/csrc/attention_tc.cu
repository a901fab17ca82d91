// Tensor-core (tcgen05 / TMEM / TMA) prefill attention over the paged KV
// cache with the sliding window and the window-clamped image mask (vLLM PR
// #53147 summary, implementation items 1-2 and the compute_tile_loop_bounds
// excerpt).
//
// Persistent: one CTA per SM walks its share of the work items.  An item is
// one 128-row query tile -- 128 / G query positions x the G query heads of one
// kv head (GQA packing: every K/V tile is staged once for the whole group) --
// and its key loop covers the 128-key tiles of the union of its rows' visible
// intervals (the pruned tile range of the union formula).  A scheduler warp
// decodes the items and publishes them as records in a small ring (the item,
// its tile range and the image ranges meeting its rows); every role reads
// them and counts tiles, K/V units and exchanges globally, so the rings, the
// S buffers and every barrier phase simply continue from one item to the
// next: the next item's Q copy and first two QK MMAs overlap the current
// item's tail.
//
// Built for head_dim 256 (head_dim 128 runs on attention_tc_pair.cu).
// Shared memory: the Q tile (TMA, 128-byte swizzled, K-major) and two rings
// of 32 KB units: a K unit holds one half of
// head_dim for all 128 keys of a tile, a V unit all of head_dim for one
// 64-key half of a tile, so QK consumes two K units and PV two V units and
// each is recycled as soon as its half of the MMA work is done.  At the end
// of an item, once its PVs are done, the V ring holds its normalised O (bf16,
// in the output map's swizzled boxes) until the TMA stores have read it.
// TMEM (512 columns): O [0, D) and two S buffers of 128 fp32 columns; the
// softmax overwrites the front of S with P as bf16 pairs, the A operand of PV.
//
// Sixteen warps; setmaxnreg moves registers from the first two warpgroups
// (64 each) to the softmax warpgroups (192 each):
//   warps 0, 2  K producers, warps 4-6 V producers:
//              every lane resolves the cache slot of one page box through the
//              block table (32 boxes per batch, one batch ahead); a unit's
//              boxes (one per page and 64-column chunk) are dealt round-robin
//              over the operand's producer warps, since one warp issues TMA
//              boxes one after another; pages past the sequence or with a bad
//              block id are read from outside the tensor, which the TMA fills
//              with 0.  Warp 4 also writes each item's staged O out.
//   warp 1     QK issuer, Q loads and TMEM owner (the Q copy of an item can
//              only start once the previous item's last QK is done, when
//              this thread would wait for it anyway; the K producers never
//              wait for it), warp 3 PV issuer: two tcgen05
//              streams, so a ready PV never waits behind a QK issue that the
//              tensor pipe holds up; QK runs two tiles ahead of PV along the
//              CTA's flat tile stream (QK_t waits until PV_{t-2} is issued).
//   warp 7     scheduler: decodes the items (dependent global loads) ahead
//              of the other roles and publishes their records.
//   warps 8-15 softmax, two warpgroups: thread i of each owns row i (TMEM lane
//              i) and one half of the tile's columns; half-row maxima meet in
//              shared memory once per tile.  Masks only tiles not fully inside
//              the row's interval, keeps the running max in the log2 domain,
//              rescales O in TMEM only when the max grows by more than 2^8, and
//              at the end of an item normalises its half of O into the V ring.
// Every mbarrier wait is bounded in time; on expiry the CTA sets
// SWA_ERR_TIMEOUT, drains its own TMA loads and MMAs, frees TMEM and exits.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "attn_tc_common.cuh"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;


// Warpgroups 0-1 hold the TMA producers and the MMA issuers and give registers
// away (setmaxnreg); the NSW warpgroups from warp 8 on are the softmax.
constexpr int kFirstSoftmaxWarp = 8;

template <int D_, int KSU_, int VSU_, int KW_, int VW_, int NSW_, int NS_>
struct Cfg {
  static constexpr int D = D_;          // head dim
  static constexpr int N = 128;         // keys per tile
  static constexpr int M = 128;         // query rows per item
  static constexpr int CH = D / 64;     // 128-byte column chunks per row
  static constexpr int KSU = KSU_;      // K ring slots (units)
  static constexpr int VSU = VSU_;      // V ring slots (units)
  // TMA issue from one warp is serial (about one 2 KB page box per 90 cycles),
  // so each K and V unit's boxes are shared between KW and VW producer warps:
  // K warps 0 and 2; V warps 4 .. 4 + VW - 1.
  static constexpr int KW = KW_;
  static constexpr int VW = VW_;
  // NSW softmax warpgroups share every row (each owns N / NSW columns of S and
  // D / NSW of O); NS S buffers in TMEM let QK run NS tiles ahead of PV.
  static constexpr int NSW = NSW_;
  static constexpr int NS = NS_;
  static constexpr int THREADS = 32 * (kFirstSoftmaxWarp + 4 * NSW);
  static constexpr int REC_READERS = KW + VW + 2 + 4 * NSW;   // warps that read every item record
  static constexpr int LAUNCH_REGS = (65536 / THREADS) & ~7;   // what the launch allocates per thread
  static constexpr int LOW_REGS = 64;                           // producers and MMA issuers
  static constexpr int HIGH_REGS =                             // softmax: all that the others free
      ((LAUNCH_REGS * THREADS - 32 * kFirstSoftmaxWarp * LOW_REGS) / (128 * NSW)) & ~7;
  static constexpr int Q_CHUNK = M * 128;
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int UNIT = N * D;                 // bytes of a K or V unit
  static constexpr int KU_CH = CH / 2;               // chunks per K unit (half of head_dim)
  static constexpr int KU_CHUNK = N * 128;           // bytes per chunk of a K unit (128 keys)
  static constexpr int VU_KEYS = N / 2;              // keys per V unit
  static constexpr int VU_CHUNK = VU_KEYS * 128;     // bytes per chunk of a V unit
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + KSU * UNIT;
  static constexpr int OFF_CTRL = OFF_V + VSU * UNIT;
  static constexpr int O_CHUNK = M * 128;            // bytes of one staged 64-column chunk of O (bf16)
  static constexpr int TM_O = 0;        // TMEM columns: O [0, D), S buffer b at [D + b*N, D + (b+1)*N)
  static constexpr int TM_S = D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, N, false);
  static constexpr uint32_t IDESC_QK_HALF = idesc_bf16(128, N / 2, false);   // an item's last tile, first half
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
  static_assert(D + NS * N <= 512, "TMEM budget");
  static_assert((NSW == 2 || NSW == 4) && NS >= 2 && NS <= 3, "softmax warpgroups, S buffers");
  static_assert(32 * kFirstSoftmaxWarp * LOW_REGS + 128 * NSW * HIGH_REGS <= LAUNCH_REGS * THREADS,
                "the register split can only hand over what the launch allocated");
  static_assert(KSU <= kMaxUnits && VSU <= kMaxUnits && KSU >= 2 && VSU >= 2, "ring sizes");
  static_assert(KW >= 1 && KW <= 2 && VW >= 1 && VW <= 4, "producer warps");
  static_assert((N / 16) * KU_CH <= 32 && (VU_KEYS / 16) * CH <= 32, "one warp instruction per unit");
  static_assert(CH * O_CHUNK <= VSU * UNIT, "the item's O (bf16) is staged in the V ring");
};

template <int NSW, int NS>
struct Ctrl {
  float red[2][NSW][128];                // partial row max / row-sum exchange buffers
  uint64_t q_full, q_empty;
  uint64_t k_full[kMaxUnits], k_empty[kMaxUnits], v_full[kMaxUnits], v_empty[kMaxUnits];
  uint64_t s_full[NS], p_full[NS];
  uint64_t pv_iss[NS];                   // PV of the tile issued (its S buffer may be overwritten)
  uint64_t o_full[2];                    // PV of tile t complete, alternating by t & 1
  uint64_t o_item, drain, drain2;
  uint64_t stall;                        // never signalled: the watchdog test's stalled wait
  uint64_t xch[2];                       // exchanges between the softmax warpgroups
  uint64_t rec_full[kRecSlots];          // item record ord published at [ord % kRecSlots]
  uint64_t rec_empty[kRecSlots];         // ... and read by every consumer warp
  uint64_t ostage_full;                  // the item's O staged in the V ring (or stored directly)
  uint64_t ostage_free;                  // the staged O has been read: the V ring may be refilled
  ItemRec rec[kRecSlots];
  uint32_t tmem_base;
  int abort;
};

// V warp 4: an item's O, staged in the V ring by the softmax (bf16, boxes of
// 64 columns x 128 rows, 128-byte swizzle), to the output; the V ring is
// released (`free_bar`) once the staged O has been read, unless this is the
// CTA's last item.  A tile whose rows all lie inside the sequence goes out as
// TMA stores issued by lane 0; any other tile is copied by the warp, one
// 512-byte row per instruction, for the rows of the sequence only.  `tok`:
// the tile's first token, `ntok`: its tokens inside the sequence.  (Freeing
// the two V slots one at a time, as each half is read, measured slower.)
template <class C>
__device__ inline void store_staged_o(const CUtensorMap *tm_o, int o_tma, const AttnArgs &a, uint32_t v_s, int G,
                                      int bq, int hk, int tok, int ntok, int lane, bool last, uint32_t free_bar) {
  static_assert(C::CH * 8 == 32, "one lane per 16-byte piece of a row");
  if (o_tma && ntok == bq) {
    if (lane == 0) {
      for (int c = 0; c < C::CH; ++c) tma_store_3d(tm_o, v_s + c * C::O_CHUNK, c * 64, hk * G, tok);
      bulk_commit();
      if (!last) {
        bulk_wait_read<0>();
        mbar_arrive(free_bar);
      }
    }
    return;
  }
  const int lg = 31 - __clz(G);                         // G is a power of two
  const int chunk = lane >> 3, j = lane & 7;
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
  for (int r = 0; r < (ntok << lg); ++r) {
    const uint4 v = ld_shared_v4(v_s + (uint32_t)(chunk * C::O_CHUNK + r * 128 + ((j ^ (r & 7)) << 4)));
    const int64_t orow = (int64_t)(tok + (r >> lg)) * a.hq + hk * G + (r & (G - 1));
    *reinterpret_cast<uint4 *>(out + orow * C::D + lane * 8) = v;
  }
  __syncwarp();
  if (lane == 0 && !last) mbar_arrive(free_bar);
}

template <class C>
constexpr int smem_bytes() { return C::OFF_CTRL + (int)sizeof(Ctrl<C::NSW, C::NS>); }

template <class C, bool NEG>
__global__ void __launch_bounds__(C::THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const AttnArgs a, const int G, const int n_items, const int o_tma) {
  // Everything lives in dynamic shared memory, which starts 1024-byte aligned
  // when a kernel has no static shared data (checked below): the 128-byte
  // swizzled tiles need that alignment and there is no room for slack.
  extern __shared__ __align__(1024) uint8_t dsm_ptr[];
  const uint32_t dsm = smem_u32(dsm_ptr);
  Ctrl<C::NSW, C::NS> &ctl = *reinterpret_cast<Ctrl<C::NSW, C::NS> *>(dsm_ptr + C::OFF_CTRL);
  const uint32_t q_s = dsm + C::OFF_Q;
  const uint32_t k_s = dsm + C::OFF_K;
  const uint32_t v_s = dsm + C::OFF_V;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bq = C::M / G;
  if ((dsm & 1023u) != 0) {
    if (threadIdx.x == 0) report(a.err, SWA_ERR_INTERNAL);
    return;
  }
  if (threadIdx.x == 0) {
    ctl.abort = 0;
    mbar_init(smem_u32(&ctl.q_full), 1);
    mbar_init(smem_u32(&ctl.q_empty), 1);
    for (int i = 0; i < C::KSU; ++i) {
      mbar_init(smem_u32(&ctl.k_full[i]), 1);
      mbar_init(smem_u32(&ctl.k_empty[i]), 1);
    }
    for (int i = 0; i < C::VSU; ++i) {
      mbar_init(smem_u32(&ctl.v_full[i]), 1);
      mbar_init(smem_u32(&ctl.v_empty[i]), 1);
    }
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(smem_u32(&ctl.s_full[i]), 1);
      mbar_init(smem_u32(&ctl.p_full[i]), 128 * C::NSW);
      mbar_init(smem_u32(&ctl.pv_iss[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl.xch[i]), 128 * C::NSW);
      mbar_init(smem_u32(&ctl.o_full[i]), 1);
    }
    mbar_init(smem_u32(&ctl.o_item), 1);
    for (int i = 0; i < kRecSlots; ++i) {
      mbar_init(smem_u32(&ctl.rec_full[i]), 1);
      mbar_init(smem_u32(&ctl.rec_empty[i]), C::REC_READERS);
    }
    mbar_init(smem_u32(&ctl.ostage_full), 128 * C::NSW);
    mbar_init(smem_u32(&ctl.ostage_free), 1);
    mbar_init(smem_u32(&ctl.drain), 1);
    mbar_init(smem_u32(&ctl.stall), 1);                 // nothing ever arrives here
    mbar_init(smem_u32(&ctl.drain2), 1);
    mbar_fence_init();
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    if (o_tma) tma_prefetch_map(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int *abort_flag = &ctl.abort;
  const uint64_t wl = a.wait_ns;                      // bound of every pipeline wait (drains: kWaitLimitNs)
  const int stride = gridDim.x;

  // Register split (warpgroup-wide, at the top of each side so every warp of a
  // warpgroup executes it converged; the freed registers are handed over at
  // once, so the increase never waits on work of the other side).
  if (warp < kFirstSoftmaxWarp) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::LOW_REGS));
  const bool k_warp = warp == 0 || (warp >= 2 && warp < 1 + C::KW);
  const bool v_warp = warp >= 4 && warp < 4 + C::VW;
  if (k_warp || v_warp) {
    // =============================== TMA producers ==============================
    // Every producer warp of an operand walks all units; the unit's boxes are
    // dealt round-robin over the warps (share), and share 0 posts the expected
    // bytes (a box of another share may land first: the transaction count may
    // go below zero, but the phase cannot complete before that arrival).
    const bool is_v = v_warp;
    const int nsh = is_v ? C::VW : C::KW;
    const int share = is_v ? warp - 4 : (warp == 0 ? 0 : warp - 1);
    const int SU = is_v ? C::VSU : C::KSU;
    const CUtensorMap *map = is_v ? &tm_v : &tm_k;
    const int unit_keys = is_v ? C::VU_KEYS : C::N;     // K units: 128 keys, V units: 64 keys
    const int R = min(a.block_size, unit_keys);         // rows per box
    const int boxes = unit_keys / R;                    // boxes per unit (per chunk)
    const int uch = is_v ? C::CH : C::KU_CH;            // chunks per unit
    const int oob = (int)(a.num_blocks * a.block_size);
    const int lg_bs = 31 - __clz(a.block_size);         // block sizes are powers of two
    int64_t u_base = 0;                                 // units issued by this warp before this item
    int ord = 0;                                        // items so far
    bool ok = true;
    // V warps: the previous item's output tile (kv head, first token, tokens inside the sequence)
    int prev_hk = 0, prev_tok = 0, prev_ntok = 0;
    for (;; ++ord) {
      // the item's record (n_tiles 0: the end of the stream)
      const int rs = ord % kRecSlots;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.rec_full[rs]), (uint32_t)((ord / kRecSlots) & 1),
                                             abort_flag, wl));
      if (!ok) break;
      const Item it = ctl.rec[rs].it;
      const int key_lo = ctl.rec[rs].key_lo, n_tiles = ctl.rec[rs].n_tiles;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.rec_empty[rs]));
      if (n_tiles == 0) break;
      if (is_v && share == 0 && ord > 0) {
        // The previous item's O is staged in the V ring once its last PV is
        // done (so are its V units): V warp 4 stores it and frees the slots.
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.ostage_full), (uint32_t)((ord - 1) & 1), abort_flag, wl));
        if (!ok) break;
        store_staged_o<C>(&tm_o, o_tma, a, v_s, G, bq, prev_hk, prev_tok, prev_ntok, lane, false,
                          smem_u32(&ctl.ostage_free));
      }
      if (is_v && ord > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.ostage_free), (uint32_t)((ord - 1) & 1), abort_flag, wl));
        if (!ok) break;
      }
      const int total_boxes = (n_tiles * C::N) / R;
      const int32_t *bt = a.block_table + (int64_t)it.s * a.bt_stride;
      auto resolve = [&](int b) -> int {                // slot of the first key of box b
        const int k = key_lo + b * R;
        int slot = oob;
        if (b < total_boxes && k < it.seq_len) {
          const int page = k >> lg_bs;
          const int32_t blk = page < a.bt_stride ? __ldg(bt + page) : -1;
          if (blk >= 0 && blk < a.num_blocks) slot = (blk << lg_bs) + (k & (a.block_size - 1));
          else if (warp == 0) report(a.err, SWA_ERR_BLOCK_ID);
        }
        return slot;
      };
      int batch = 0;
      int prv = oob, cur = resolve(lane), nxt = resolve(32 + lane);
      int ul = 0;
      for (; ul < 2 * n_tiles; ++ul) {                 // unit ul of this item: tile ul/2, half ul%2
        const int64_t u = u_base + ul;
        const int slot_i = (int)(u % SU);
        if (u >= SU) {
          const uint32_t empty = smem_u32(is_v ? &ctl.v_empty[slot_i] : &ctl.k_empty[slot_i]);
          ok = __all_sync(0xffffffffu,
                          mbar_wait(empty, (uint32_t)(((u / SU) - 1) & 1), abort_flag, wl));
          if (!ok) break;
        }
        const int t = ul >> 1, half = ul & 1;
        const uint32_t full = smem_u32(is_v ? &ctl.v_full[slot_i] : &ctl.k_full[slot_i]);
        const uint32_t dst = (is_v ? v_s : k_s) + slot_i * C::UNIT;
        if (share == 0 && lane == 0) mbar_expect_tx(full, C::UNIT);
        __syncwarp();
        // K: unit = head_dim half `half` of tile t's 128 keys; V: key half `half`
        const int b0 = is_v ? (2 * t + half) * boxes : t * boxes;
        while (b0 + boxes - 1 >= (batch + 1) * 32) {    // warp-uniform batch advance
          prv = cur;
          cur = nxt;
          ++batch;
          nxt = resolve((batch + 1) * 32 + lane);
        }
        const int i = min(lane / uch, boxes - 1), c = lane % uch;
        const int b = b0 + i;
        const int from_cur = __shfl_sync(0xffffffffu, cur, (b - batch * 32) & 31);
        const int from_prv = __shfl_sync(0xffffffffu, prv, (b - (batch - 1) * 32) & 31);
        const int slot = b >= batch * 32 ? from_cur : from_prv;
        const int x = (is_v ? c : half * C::KU_CH + c) * 64;
        const uint32_t d = dst + c * (is_v ? C::VU_CHUNK : C::KU_CHUNK) + i * R * 128;
        if (lane < boxes * uch && lane % nsh == share) tma_load_3d(d, map, x, it.hk, slot, full);
      }
      u_base += ul;                                     // units issued (all of them unless aborted)
      if (!ok) break;
      prev_hk = it.hk;
      prev_tok = it.qstart + it.qpos_lo;
      prev_ntok = min(bq, it.qlen - it.qpos_lo);
    }
    if (is_v && share == 0) {
      // the last item's O
      if (ok && ord > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.ostage_full), (uint32_t)((ord - 1) & 1), abort_flag, wl));
        if (ok)
          store_staged_o<C>(&tm_o, o_tma, a, v_s, G, bq, prev_hk, prev_tok, prev_ntok, lane, true, 0u);
      }
      if (lane == 0) bulk_wait_all();                   // every store has landed before the CTA exits
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report(a.err, SWA_ERR_TIMEOUT);
    }
    // drain: every load issued by this warp must have landed before the CTA exits
    if (lane == 0) {
      for (int64_t u = max((int64_t)0, u_base - SU); u < u_base; ++u)
        mbar_wait(smem_u32(is_v ? &ctl.v_full[u % SU] : &ctl.k_full[u % SU]), (uint32_t)((u / SU) & 1), nullptr, kWaitLimitNs);
    }
  } else if (warp == 1 || warp == 3) {
    // =============================== MMA issuers ================================
    // Warp 1 issues the QK MMAs, warp 3 the PV MMAs, each from its own stream,
    // so a PV never waits behind a QK issue that is blocked on the tensor pipe.
    // QK_t writes S buffer t & 1, which holds P_{t-2}: it is issued only after
    // PV_{t-2} (warp 3 fences and arrives on pv_iss after issuing it; tcgen05
    // work ordered through a fence pair runs in that order).
    if (lane == 0 && warp == 1) {
      bool ok = true;
      int ord = 0;
      int n_q = 0;                                       // Q copies issued
      int t = 0;                                         // tiles of this CTA's stream
      while (ok) {
        // the item's record (n_tiles 0: the end of the stream), then its Q
        const int rs = ord % kRecSlots;
        ok = mbar_wait(smem_u32(&ctl.rec_full[rs]), (uint32_t)((ord / kRecSlots) & 1), abort_flag, wl);
        if (!ok) break;
        const int n = ctl.rec[rs].n_tiles, hl = ctl.rec[rs].half_last;
        const int q_hk = ctl.rec[rs].it.hk, q_tok = ctl.rec[rs].it.qstart + ctl.rec[rs].it.qpos_lo;
        mbar_arrive(smem_u32(&ctl.rec_empty[rs]));
        if (n == 0) break;
        // Q: once the previous item's last QK is done with the buffer (this
        // thread would wait for the copy before its next MMA anyway)
        if (ord > 0) ok = mbar_wait(smem_u32(&ctl.q_empty), (uint32_t)((ord - 1) & 1), abort_flag, wl);
        if (!ok) break;
        mbar_expect_tx(smem_u32(&ctl.q_full), C::Q_BYTES);
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d(q_s + c * C::Q_CHUNK, &tm_q, c * 64, q_hk * G, q_tok, smem_u32(&ctl.q_full));
        ++n_q;
        ok = mbar_wait(smem_u32(&ctl.q_full), (uint32_t)(ord & 1), abort_flag, wl);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; ok && j < n; ++j, ++t) {
          const int sb = (int)(t % C::NS);               // S buffer of tile t
          if (t >= C::NS) {
            ok = mbar_wait(smem_u32(&ctl.pv_iss[sb]), (uint32_t)(((t / C::NS) - 1) & 1), abort_flag, wl);
            if (!ok) break;
            tc_fence_after();
          }
          const uint32_t d = tmem + C::TM_S + (uint32_t)sb * C::N;
          // the item's last tile: only its first N / 2 keys when no row sees the rest
          const uint32_t idesc = (j == n - 1 && hl) ? C::IDESC_QK_HALF : C::IDESC_QK;
          for (int half = 0; ok && half < 2; ++half) {
            const uint32_t u = 2u * (uint32_t)t + half;
            const int slot = (int)(u % C::KSU);
            ok = mbar_wait(smem_u32(&ctl.k_full[slot]), (uint32_t)((u / C::KSU) & 1), abort_flag, wl);
            if (!ok) break;
            tc_fence_after();
            const uint32_t qa = q_s + half * C::KU_CH * C::Q_CHUNK;
            const uint32_t kb = k_s + slot * C::UNIT;
#pragma unroll
            for (int kk = 0; kk < C::D / 32; ++kk) {    // 16-column steps over this half of head_dim
              const uint32_t off = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;   // chunk, then 32 B in the swizzle row
              const uint32_t offk = (kk >> 2) * C::KU_CHUNK + (kk & 3) * 32;
              mma_ss(d, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(kb + offk, 16, 1024), idesc,
                     (half > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&ctl.k_empty[slot]));
          }
          if (!ok) break;
          mma_commit(smem_u32(&ctl.s_full[sb]));
          if (j == n - 1) mma_commit(smem_u32(&ctl.q_empty));   // the item's Q is no longer read
        }
        ++ord;
      }
      if (!ok) {
        *abort_flag = 1;
        report(a.err, SWA_ERR_TIMEOUT);
      }
      // every MMA issued by this thread must finish before TMEM is released,
      // and every Q copy must have landed
      mma_commit(smem_u32(&ctl.drain));
      mbar_wait(smem_u32(&ctl.drain), 0, nullptr, kWaitLimitNs);
      if (n_q > 0) mbar_wait(smem_u32(&ctl.q_full), (uint32_t)((n_q - 1) & 1), nullptr, kWaitLimitNs);
    } else if (lane == 0 && warp == 3) {
      bool ok = true;
      // watchdog test: a wait that can only run out (a.stall, set by swa_set_watchdog)
      if (a.stall) ok = mbar_wait(smem_u32(&ctl.stall), 0, abort_flag, wl);
      int t = 0;
      for (int ord = 0; ok; ++ord) {
        // the item's record (n_tiles 0: the end of the stream)
        ok = mbar_wait(smem_u32(&ctl.rec_full[ord % kRecSlots]), (uint32_t)((ord / kRecSlots) & 1), abort_flag, wl);
        if (!ok) break;
        const int n_tiles = ctl.rec[ord % kRecSlots].n_tiles, hl = ctl.rec[ord % kRecSlots].half_last;
        mbar_arrive(smem_u32(&ctl.rec_empty[ord % kRecSlots]));
        if (n_tiles == 0) break;
        for (int j = 0; ok && j < n_tiles; ++j, ++t) {
          const int sb = (int)(t % C::NS);
          ok = mbar_wait(smem_u32(&ctl.p_full[sb]), (uint32_t)((t / C::NS) & 1), abort_flag, wl);
          // keys of the tile that take part: the first N / 2 of an item's last tile when half_last
          const int lim = (j == n_tiles - 1 && hl) ? C::N / 2 : C::N;
          for (int half = 0; ok && half < 2; ++half) {
            const uint32_t u = 2u * (uint32_t)t + half;
            const int slot = (int)(u % C::VSU);
            ok = mbar_wait(smem_u32(&ctl.v_full[slot]), (uint32_t)((u / C::VSU) & 1), abort_flag, wl);
            if (!ok) break;
            tc_fence_after();
            const uint32_t p_t = tmem + C::TM_S + (uint32_t)sb * C::N + half * (C::VU_KEYS / 16) * 8;
            const uint32_t vb = v_s + slot * C::UNIT;
#pragma unroll
            for (int kk = 0; kk < C::VU_KEYS / 16; ++kk)
              if (half * C::VU_KEYS + kk * 16 < lim)
                mma_ts(tmem + C::TM_O, p_t + kk * 8, smem_desc_sw128(vb + kk * 16 * 128, C::VU_CHUNK, 1024), C::IDESC_PV,
                       (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(&ctl.v_empty[slot]));
          }
          if (!ok) break;
          mma_commit(smem_u32(&ctl.o_full[t & 1]));
          if (j == n_tiles - 1) mma_commit(smem_u32(&ctl.o_item));   // the item's O is final
          tc_fence_before();
          mbar_arrive(smem_u32(&ctl.pv_iss[sb]));
        }
      }
      if (!ok) {
        *abort_flag = 1;
        report(a.err, SWA_ERR_TIMEOUT);
      }
      mma_commit(smem_u32(&ctl.drain2));
      mbar_wait(smem_u32(&ctl.drain2), 0, nullptr, kWaitLimitNs);
    }
  } else if (warp == 7) {
    // =============================== scheduler ==================================
    // Decodes the CTA's items (a chain of dependent global loads) ahead of
    // every other role and publishes them as records, up to kRecSlots ahead
    // of the slowest reader.
    bool ok = true;
    int ord = 0;
    auto publish = [&](const Item &it, int key_lo, int n_tiles, int hl, int nr, int rrs, int rre) -> bool {
      const int rs = ord % kRecSlots;
      if (ord >= kRecSlots &&
          !__all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&ctl.rec_empty[rs]), (uint32_t)(((ord / kRecSlots) - 1) & 1),
                                             abort_flag, wl)))
        return false;
      write_rec(ctl.rec[rs], it, key_lo, n_tiles, hl, nr, rrs, rre, lane);
      if (lane == 0) mbar_arrive(smem_u32(&ctl.rec_full[rs]));
      ++ord;
      return true;
    };
    for (int item = blockIdx.x; ok && item < n_items; item += stride) {
      Item it;
      int32_t eb;
      if (!decode_item(a, item, bq, it, eb)) {
        if (eb != 0 && lane == 0) report(a.err, eb);
        continue;
      }
      int key_lo, n_tiles, hl, nr, rrs, rre;
      block_keys_rec<C::N>(a, it, lane, key_lo, n_tiles, hl, nr, rrs, rre);
      ok = publish(it, key_lo, n_tiles, hl, nr, rrs, rre);
    }
    if (ok) ok = publish(Item{}, 0, 0, 0, 0, 0, -1);         // the end of the stream
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report(a.err, SWA_ERR_TIMEOUT);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::HIGH_REGS));
    // =============================== softmax ====================================
    // Two warpgroups share every row: warpgroup h owns S columns
    // [h*N/2, (h+1)*N/2) and O columns [h*D/2, (h+1)*D/2).  Both keep the
    // same running max (half-row maxima are exchanged through shared memory
    // once per tile, ordered by a bounded mbarrier) and a partial row sum.
    constexpr int NSW = C::NSW;
    constexpr int NH = C::N / NSW;                       // S columns of one warpgroup
    constexpr int DH = C::D / NSW;                       // O columns of one warpgroup
    const int h = (warp - kFirstSoftmaxWarp) >> 2;
    const int sid = threadIdx.x - 32 * kFirstSoftmaxWarp;   // 0 .. 128 * NSW - 1
    const int row = 32 * (warp & 3) + lane;              // TMEM lane of this thread
    const uint32_t lane_t = (uint32_t)(32 * (warp & 3)) << 16;
    // the scale is folded into the exponent's FFMA: maxima are taken on the raw
    // scores (of -S for a negative scale, NEG) and scaled once
    const float asl2 = fmaxf(fabsf(a.scale * kLog2e), 1.17549435e-38f);
    int t = 0;                                           // this CTA's tiles so far
    int64_t xc = 0;                                      // exchanges so far (buffer xc & 1)
    int n_done = 0;                                      // items finished
    // Items come from the records the Q producer publishes; the next one is
    // set up while the current item's last PV runs.
    RowSetup cur;
    bool have = false;
    auto next_rec = [&]() -> bool {                      // false: the wait ran out
      const int slot = n_done % kRecSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.rec_full[slot]),
                                             (uint32_t)((n_done / kRecSlots) & 1), abort_flag, wl)))
        return false;
      have = ctl.rec[slot].n_tiles > 0;
      if (have) row_setup_rec(a, ctl.rec[slot], row, G, lane, cur);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.rec_empty[slot]));
      return true;
    };
    bool ok = next_rec();
    while (ok && have) {
      const Item &it = cur.it;
      const int key_lo = cur.key_lo, n_tiles = cur.n_tiles;
      const int klo = cur.klo, khi = cur.khi;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < n_tiles; ++j, ++t) {
        const int kt0 = key_lo + j * C::N;
        const int kc0 = kt0 + h * NH;                    // key of this warpgroup's first column
        const int sb = (int)(t % C::NS);                 // S buffer of tile t
        ok = mbar_wait(smem_u32(&ctl.s_full[sb]), (uint32_t)((t / C::NS) & 1), abort_flag, wl);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t raw[NH];
        float lred[NH / 32];                              // per 32 columns: max of S (min for NEG)
#pragma unroll
        for (int c = 0; c < NH / 32; ++c)
          tmem_ld32_red<NEG>(tmem + lane_t + C::TM_S + (uint32_t)sb * C::N + h * NH + 32 * c,
                             *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * c), lred[c]);
        tmem_wait_ld();
        float x[NH];
        float mx;
        const bool full = klo <= kc0 && khi >= kc0 + NH - 1;
        if (__all_sync(0xffffffffu, full)) {
#pragma unroll
          for (int c = 0; c < NH; ++c) x[c] = NEG ? -__uint_as_float(raw[c]) : __uint_as_float(raw[c]);
          float r = lred[0];
#pragma unroll
          for (int c = 1; c < NH / 32; ++c) r = NEG ? fminf(r, lred[c]) : fmaxf(r, lred[c]);
          mx = NEG ? -r : r;
        } else {
          // column c is visible when c_lo <= c <= c_lo + span: one unsigned compare
          // (an empty interval puts c_lo past the tile, so c - c_lo wraps above span)
          const bool empty = khi < klo;
          const int c_lo = empty ? 2 * NH : klo - kc0;
          const uint32_t c_span = empty ? 0u : (uint32_t)(khi - klo);
#pragma unroll
          for (int c = 0; c < NH; ++c)
            x[c] = (uint32_t)(c - c_lo) <= c_span ? (NEG ? -__uint_as_float(raw[c]) : __uint_as_float(raw[c]))
                                                  : -INFINITY;
          float m4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = x[i];
#pragma unroll
          for (int c = 4; c + 8 <= NH; c += 8)
#pragma unroll
            for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], x[c + 2 * i], x[c + 2 * i + 1]);
#pragma unroll
          for (int c = 4 + ((NH - 4) / 8) * 8; c < NH; ++c) m4[c & 3] = fmaxf(m4[c & 3], x[c]);
          mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        }
        mx = mx == -INFINITY ? -INFINITY : mx * asl2;
        ctl.red[xc & 1][h][row] = mx;
        mbar_arrive(smem_u32(&ctl.xch[xc & 1]));
        ok = mbar_wait_spin(smem_u32(&ctl.xch[xc & 1]), (uint32_t)((xc >> 1) & 1), abort_flag, wl);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
        for (int g = 0; g < NSW; ++g)
          if (g != h) mx = fmaxf(mx, ctl.red[xc & 1][g][row]);
        ++xc;
        const float m_new = fmaxf(m_used, mx);
        const bool need = m_new > m_used + 8.f;           // also true on the first visible tile
        // P_t does not wait for PV_{t-1}; only a rescale of O (and the V tail
        // below) does.  PV_{t-2} has completed here (QK_t, seen complete, was
        // issued after it and tcgen05 work completes in issue order), so the
        // o_full phase of PV_{t-1} is the only one that can still be open and
        // its parity is unambiguous.  An item's first tile needs no wait: the
        // previous item's epilogue saw all of its PVs complete.
        if (__any_sync(0xffffffffu, need)) {             // same decision in both warpgroups
          const float m_next = need ? m_new : m_used;
          const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_next);
          if (j > 0) {
            ok = mbar_wait(smem_u32(&ctl.o_full[(t - 1) & 1]), (uint32_t)(((t - 1) >> 1) & 1), abort_flag, wl);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
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
        uint64_t sl2x2, nms;
        asm volatile("mov.b64 %0, {%1, %1};" : "=l"(sl2x2) : "f"(asl2));
        asm volatile("mov.b64 %0, {%1, %1};" : "=l"(nms) : "f"(-ms));
        uint32_t pk[NH / 2];
        uint64_t s2[2] = {0, 0};
#pragma unroll
        for (int c = 0; c < NH / 2; ++c) {
          float e0, e1;
          f2_unpack(f2_fma(f2_pack(x[2 * c], x[2 * c + 1]), sl2x2, nms), e0, e1);
          const float p0 = ex2(e0), p1 = ex2(e1);
          s2[c & 1] = f2_add(s2[c & 1], f2_pack(p0, p1));
          pk[c] = pack_bf16(p0, p1);
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(s2[0], a0, a1);
          f2_unpack(s2[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        if (kt0 + C::N > it.seq_len) {
          // keys past the sequence end: their V rows may hold anything; zero
          // them.  Once PV_{t-1} is done every earlier unit of each V slot has
          // been consumed, so the v_full parity below is unambiguous.
          if (j > 0) {
            ok = mbar_wait(smem_u32(&ctl.o_full[(t - 1) & 1]), (uint32_t)(((t - 1) >> 1) & 1), abort_flag, wl);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          }
          for (int half = 0; half < 2 && ok; ++half) {
            const int k0 = kt0 + half * C::VU_KEYS;
            if (k0 + C::VU_KEYS <= it.seq_len) continue;
            const uint32_t u = 2u * (uint32_t)t + half;
            const int slot = (int)(u % C::VSU);
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.v_full[slot]), (uint32_t)((u / C::VSU) & 1),
                                                   abort_flag, wl));
            if (!ok) break;
            const int r0 = max(0, it.seq_len - k0);       // first row to clear
            uint8_t *unit = dsm_ptr + C::OFF_V + slot * C::UNIT;
#pragma unroll 1
            for (int i = sid; i < C::CH * C::VU_KEYS * 8; i += 128 * NSW) {   // 16-byte pieces: chunk, row, piece
              const int r = (i >> 3) & (C::VU_KEYS - 1);
              if (r >= r0)
                *reinterpret_cast<uint4 *>(unit + (i / (C::VU_KEYS * 8)) * C::VU_CHUNK + r * 128 + (i & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
          }
          if (!ok) break;
          fence_proxy_async_smem();
        }
        if constexpr (NH / 2 >= 32) {
#pragma unroll
          for (int c = 0; c < NH / 2; c += 32)
            tmem_st32(tmem + lane_t + C::TM_S + (uint32_t)sb * C::N + h * (NH / 2) + c,
                      *reinterpret_cast<const uint32_t(*)[32]>(pk + c));
        } else {
          tmem_st16(tmem + lane_t + C::TM_S + (uint32_t)sb * C::N + h * (NH / 2), pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl.p_full[sb]));
      }
      if (!ok) break;
      const bool row_valid = cur.row_valid;
      const int64_t out_row = cur.out_row;
      ++n_done;
      if (!next_rec()) { ok = false; break; }
      // the item's last PV (one o_item phase per item), then the full row sum
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.o_item), (uint32_t)((n_done - 1) & 1), abort_flag, wl));
      if (!ok) break;
      ctl.red[xc & 1][h][row] = l;
      mbar_arrive(smem_u32(&ctl.xch[xc & 1]));
      ok = __all_sync(0xffffffffu, mbar_wait_spin(smem_u32(&ctl.xch[xc & 1]), (uint32_t)((xc >> 1) & 1), abort_flag, wl));
      if (!ok) break;
#pragma unroll
      for (int g = 0; g < NSW; ++g)
        if (g != h) l += ctl.red[xc & 1][g][row];
      ++xc;
      // epilogue: O / l -> bf16 rows in the V ring (free: the item's PVs are
      // done and the V producers wait for ostage_free), laid out as the output
      // map's boxes of 64 columns x 128 rows with the 128-byte swizzle, so that
      // the 16-byte pieces of 8 rows hit all banks; V warp 4 stores them.  The
      // next item's first PV overwrites O only after this thread's P for it
      // (published after these loads completed).
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < DH / 64; ++c) {                  // one staged 64-column chunk per pass
        uint32_t r[64];
        tmem_ld32(tmem + lane_t + C::TM_O + h * DH + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld32(tmem + lane_t + C::TM_O + h * DH + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        const uint32_t rb = v_s + (uint32_t)((h * (DH / 64) + c) * C::O_CHUNK + row * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)                        // 16-byte piece j of the 128-byte row
          st_shared_v4(rb + ((uint32_t)(j ^ (row & 7)) << 4),
                       pack_bf16(__uint_as_float(r[8 * j]) * inv, __uint_as_float(r[8 * j + 1]) * inv),
                       pack_bf16(__uint_as_float(r[8 * j + 2]) * inv, __uint_as_float(r[8 * j + 3]) * inv),
                       pack_bf16(__uint_as_float(r[8 * j + 4]) * inv, __uint_as_float(r[8 * j + 5]) * inv),
                       pack_bf16(__uint_as_float(r[8 * j + 6]) * inv, __uint_as_float(r[8 * j + 7]) * inv));
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&ctl.ostage_full));
      if (row_valid && h == 0 && a.lse != nullptr)
        a.lse[out_row] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before();
    }
    if (!ok) {
      *abort_flag = 1;
      report(a.err, SWA_ERR_TIMEOUT);
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
template <class C, bool NEG>
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
  // the output through the same box shape as Q (TMA stores of whole tiles);
  // an output the map cannot describe is written with plain stores
  CUtensorMap mo;
  memset(&mo, 0, sizeof(mo));
  const int o_tma = make_map(&mo, a.out, C::D, a.hq, a.num_tokens, C::D * esz, (uint64_t)a.hq * C::D * esz, 64, G, bq)
                        ? 1 : 0;
  constexpr int smem = smem_bytes<C>();
  static_assert(smem <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<C, NEG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (a.num_tokens / bq + a.num_seqs) * (int64_t)a.hkv;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = (int)(items < sms ? items : (int64_t)sms);
  // The register split hands over exactly the launch allocation: a kernel built
  // with another per-thread count would wait forever in setmaxnreg.inc.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, attn_tc_kernel<C, NEG>) != cudaSuccess || fa.numRegs != C::LAUNCH_REGS)
    return cudaErrorInvalidConfiguration;
  attn_tc_kernel<C, NEG><<<grid, C::THREADS, smem, st>>>(mq, mk, mv, mo, a, G, (int)items, o_tma);
  return cudaGetLastError();
}

using Cfg256 = Cfg<256, 3, 2, 2, 3, 2, 2>;    // 64 KB Q + 3 K + 2 V units of 32 KB; 2 softmax WGs, 2 S

}  // namespace

bool tc_supported(const AttnArgs &a) { return a.head_dim == 256 && tc_prefill_ok(a); }

cudaError_t launch_attention_tc(const AttnArgs &a, cudaStream_t st) {
  // the sign of the scale is a template argument: a negative scale takes the
  // maximum of -S, without a per-score select
  return a.scale < 0.f ? run<Cfg256, true>(a, st) : run<Cfg256, false>(a, st);
}

}  // namespace swa
