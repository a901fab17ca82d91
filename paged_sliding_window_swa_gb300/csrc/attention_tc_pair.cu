// Tensor-core prefill attention for head_dim 128 and 64 with two query tiles
// per work item (same mask and pruning as attention_tc.cu: vLLM PR #53147
// summary, implementation items 1-2 and the compute_tile_loop_bounds excerpt).
//
// At head_dim 128 the tensor memory holds the two O accumulators, one S
// buffer and the two tiles' P (at head_dim 64, one S buffer per tile), so an
// item is a PAIR of consecutive 128-row query tiles A and B of one sequence
// and kv head (2 x 128/G positions x G heads).  Every K/V tile is staged once
// for both, and each query tile has its own softmax warpgroup that owns whole
// rows: no max exchange between warpgroups.  The key loop covers the 128-key
// tiles of the union of the pair's rows.
//
// At head_dim 128 the S buffer is shared: QK_A(t) and QK_B(t) take turns in
// it, and each QK waits only until the other tile's softmax has LOADED the
// previous scores (s_free).  P goes to a region of its own, so a tile's next
// QK never waits for its softmax to finish or for its PV: while one softmax
// warpgroup works on its scores the tensor pipe runs the other tile's QK and
// the PVs.
//
// Shared memory: Q_A and Q_B (D x 256 B each, TMA, 128-byte swizzle, K-major)
// and two rings of 16 KB units.  At head_dim 128 a K unit holds one 64-column
// half of head_dim for the 128 keys of a tile and a V unit all 128 columns for
// one 64-key half (rings of 5 + 5 units); at head_dim 64 one K unit and one V
// unit cover a tile (rings of 6 + 6).  TMEM (512 columns): O_A [0,D),
// O_B [D,2D), S [2D,2D+128), P_A and P_B 64 columns each after S (P as bf16
// pairs).  At head_dim 64 there is room for one S buffer per tile (S_A, S_B),
// so each QK waits only for its own tile's previous score load.
//
// Sixteen warps; setmaxnreg moves registers from warps 0-7 (64 each) to the
// softmax warpgroups (192 each):
//   warp 0      K producer; warps 4-6 V producers (a unit's page boxes are
//               dealt over them, one TMA box per page and chunk); warp 4 also
//               writes each item's O out (below)
//   warp 1      QK issuer, Q loads and TMEM owner: QK_A(t), QK_B(t) per key
//               tile, each after the previous scores were loaded from S; an
//               item's Q copy once the previous item's last QK is done
//   warp 3      PV issuer: PV_A(t) once P_A(t) is published, then PV_B(t)
//   warp 7      scheduler: decodes the items ahead of the other roles and
//               publishes them as records (as in attention_tc.cu)
//   warp 2      no role
//   warps 8-11  softmax of tile A, warps 12-15 softmax of tile B: thread i of
//               a warpgroup owns row i (TMEM lane i) of its tile.
// At the end of an item, once both tiles' last PVs are done, the V ring is
// idle (its producers wait for the hand-off below before the next item's
// units), so the softmax warpgroups normalise O_A and O_B into it as bf16 in
// the output map's swizzled boxes, and V warp 4 writes them out with TMA
// stores (rows of a tile that runs past its sequence: plain 16-byte copies).
// The code is kept small on purpose (32-bit counters, shifts for the
// power-of-two page size, no runtime division in the loops): at this size the
// SM's instruction cache decides how fast the rarely taken paths (item
// boundaries, masked tiles) run.  Every mbarrier wait is bounded in time; on
// expiry the CTA sets SWA_ERR_TIMEOUT, drains its own TMA loads and MMAs,
// frees TMEM and exits.
#include "attn_tc_common.cuh"
#include "tc_ptx.cuh"

namespace swa {
namespace {

using namespace tc;

template <int D_, int RING_>
struct PairCfg {
  static constexpr int D = D_;
  static constexpr int N = 128;                      // keys per tile
  static constexpr int M = 128;                      // rows per query tile
  static constexpr int CH = D / 64;                  // 128-byte column chunks per row
  static constexpr int KSU = RING_, VSU = RING_;     // ring slots (16 KB units)
  static constexpr int UPT = CH;                     // K units and V units per key tile
  static constexpr int VW = 3;                       // V producer warps 4 .. 4 + VW - 1
  static constexpr int THREADS = 512;
  static constexpr int LAUNCH_REGS = 128;
  static constexpr int LOW_REGS = 64;
  static constexpr int HIGH_REGS = 192;
  static constexpr int REC_READERS = 1 + VW + 2 + 8;   // warps that read every item record
  static constexpr int Q_CHUNK = M * 128;            // bytes of one 64-column chunk of a Q tile
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int UNIT = 16384;                 // bytes of a K or V unit
  static constexpr int KU_CHUNK = N * 128;           // a K unit is one chunk of 128 keys
  static constexpr int VU_KEYS = N / UPT;            // keys per V unit
  static constexpr int VU_CHUNK = VU_KEYS * 128;     // bytes per chunk of a V unit
  static constexpr int OFF_Q = 0;                    // Q_A, then Q_B
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KSU * UNIT;
  static constexpr int OFF_CTRL = OFF_V + VSU * UNIT;
  static constexpr int O_CHUNK = M * 128;            // bytes of one staged 64-column chunk of a tile's O
  static constexpr int TM_O = 0;                     // O_X at X * D
  // one S buffer per query tile where TMEM has room (head_dim 64), else one
  // shared by the two tiles
  static constexpr bool SEP_S = 2 * D + 3 * N <= 512;
  static constexpr int TM_S = 2 * D;                 // S_X at TM_S + X * N (SEP_S), else the shared S
  static constexpr int TM_P = 2 * D + (SEP_S ? 2 : 1) * N;   // P_X at TM_P + X * N / 2
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, N, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
  static_assert(2 * D + (SEP_S ? 2 : 1) * N + 2 * (N / 2) <= 512, "TMEM budget");
  static_assert(LAUNCH_REGS * THREADS <= 65536 && (65536 / THREADS) >= LAUNCH_REGS, "launch registers");
  static_assert(256 * LOW_REGS + 256 * HIGH_REGS <= LAUNCH_REGS * THREADS,
                "the register split can only hand over what the launch allocated");
  static_assert(KSU <= kMaxUnits && VSU <= kMaxUnits && KSU >= 2 && VSU >= 4, "ring sizes");
  static_assert(KSU == VSU, "the producers share one ring walk");
  static_assert(2 * CH * O_CHUNK <= VSU * UNIT, "both tiles' O (bf16) are staged in the V ring");
  static_assert((D == 64 || D == 128) && UPT <= 2 && VU_KEYS * D * 2 == UNIT && N * 128 == UNIT, "16 KB units");
};

struct PairCtrl {
  uint64_t q_full, q_empty;
  uint64_t k_full[kMaxUnits], k_empty[kMaxUnits], v_full[kMaxUnits], v_empty[kMaxUnits];
  uint64_t s_full[2], p_full[2];         // per query tile X: S holds QK_X(t), P_X(t) published
  uint64_t s_free[2];                    // scores loaded: S (S_X with one buffer per tile) may be overwritten
  uint64_t o_full[2], o_item[2];         // PV_X(t) complete; the item's last PV_X complete
  uint64_t drain, drain2;
  uint64_t stall;                        // never signalled: the watchdog test's stalled wait
  uint64_t rec_full[kRecSlots];          // item record ord published at [ord % kRecSlots]
  uint64_t rec_empty[kRecSlots];         // ... and read by every consumer warp
  uint64_t ostage_full;                  // both tiles' O staged in the V ring
  uint64_t ostage_free;                  // the staged O has been read: the V ring may be refilled
  ItemRec rec[kRecSlots];
  uint32_t tmem_base;
  int abort;
};

template <class C>
constexpr int pair_smem_bytes() { return C::OFF_CTRL + (int)sizeof(PairCtrl); }


// V warp 4: an item's O (both tiles), staged in the V ring by the softmax
// (bf16, tile X at CH X O_CHUNK, 64-column chunks of 128 rows, 128-byte
// swizzle), to the output; the ring is released (`free_bar`) once read, unless
// this is the CTA's last item.  A tile whose rows all lie inside the sequence
// goes out as TMA stores by lane 0; any other is copied by the warp, for the
// rows of the sequence only.  `tok`: tile A's first token, `ntok[X]`: tile X's
// tokens inside the sequence.
template <class C>
__device__ inline void store_staged_pair(const CUtensorMap *tm_o, int o_tma, const AttnArgs &a, uint32_t v_s,
                                         int G, int bq, int hk, int tok, int ntok0, int ntok1, int lane, bool last,
                                         uint32_t free_bar) {
  bool tma = false;
  for (int x = 0; x < 2; ++x) {
    const int ntok = x ? ntok1 : ntok0;
    if (ntok <= 0) continue;
    const uint32_t base = v_s + (uint32_t)(x * C::CH * C::O_CHUNK);
    if (o_tma && ntok == bq) {
      if (lane == 0)
        for (int c = 0; c < C::CH; ++c) tma_store_3d(tm_o, base + c * C::O_CHUNK, c * 64, hk * G, tok + x * bq);
      tma = true;
      continue;
    }
    const int lg = 31 - __clz(G);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
    for (int i = lane; i < (ntok << lg) * C::CH * 8; i += 32) {   // (row, 16-byte piece)
      const int r = i / (C::CH * 8), p = i % (C::CH * 8);
      const int c = p >> 3, j = p & 7;
      const uint4 v = ld_shared_v4(base + (uint32_t)(c * C::O_CHUNK + r * 128 + ((j ^ (r & 7)) << 4)));
      const int64_t orow = (int64_t)(tok + x * bq + (r >> lg)) * a.hq + hk * G + (r & (G - 1));
      *reinterpret_cast<uint4 *>(out + orow * C::D + p * 8) = v;
    }
  }
  if (lane == 0 && tma) bulk_commit();
  __syncwarp();
  if (lane == 0 && !last) {
    if (tma) bulk_wait_read<0>();
    mbar_arrive(free_bar);
  }
}

// A ring position: slot and the parity of its current fill.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ void next(int size) {
    if (++slot == size) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

template <class C, bool NEG>
__global__ void __launch_bounds__(C::THREADS, 1)
attn_tc_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const AttnArgs a, const int G, const int n_items, const int o_tma) {
  extern __shared__ __align__(1024) uint8_t dsm_ptr[];
  const uint32_t dsm = smem_u32(dsm_ptr);
  PairCtrl &ctl = *reinterpret_cast<PairCtrl *>(dsm_ptr + C::OFF_CTRL);
  const uint32_t q_s = dsm + C::OFF_Q;
  const uint32_t k_s = dsm + C::OFF_K;
  const uint32_t v_s = dsm + C::OFF_V;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bq = C::M / G;                    // positions per query tile
  const int bq2 = 2 * bq;                     // positions per item (the pair)
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
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&ctl.s_full[x]), 1);
      mbar_init(smem_u32(&ctl.p_full[x]), 128);
      mbar_init(smem_u32(&ctl.o_full[x]), 1);
      mbar_init(smem_u32(&ctl.o_item[x]), 1);
    }
    mbar_init(smem_u32(&ctl.s_free[0]), 128);
    mbar_init(smem_u32(&ctl.s_free[1]), 128);
    mbar_init(smem_u32(&ctl.ostage_full), 256);
    mbar_init(smem_u32(&ctl.ostage_free), 1);
    for (int i = 0; i < kRecSlots; ++i) {
      mbar_init(smem_u32(&ctl.rec_full[i]), 1);
      mbar_init(smem_u32(&ctl.rec_empty[i]), C::REC_READERS);
    }
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

  if (warp < 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::LOW_REGS));
  const bool k_warp = warp == 0;
  const bool v_warp = warp >= 4 && warp < 4 + C::VW;
  if (k_warp || v_warp) {
    // =============================== TMA producers ==============================
    // As in attention_tc.cu: every producer warp of an operand walks all units,
    // a unit's boxes are dealt round-robin over the warps, share 0 posts the
    // expected bytes.
    const bool is_v = v_warp;
    const int nsh = is_v ? C::VW : 1;
    const int share = is_v ? warp - 4 : 0;
    const int SU = is_v ? C::VSU : C::KSU;
    const CUtensorMap *map = is_v ? &tm_v : &tm_k;
    const int unit_keys = is_v ? C::VU_KEYS : C::N;     // K units: 128 keys, V units: 128 / UPT keys
    const int R = min(a.block_size, unit_keys);         // rows per box
    const int boxes = unit_keys / R;                    // boxes per unit (per chunk)
    const int uch = is_v ? C::CH : 1;                   // chunks per unit
    const int oob = (int)(a.num_blocks * a.block_size);
    const int lg_bs = 31 - __clz(a.block_size);
    int u_base = 0;                                     // units issued by this warp before this item
    bool ok = true;
    // V warps: the previous item's output tiles (kv head, tile A's first token, tokens of A and B in the sequence)
    int prev_hk = 0, prev_tok = 0, prev_n0 = 0, prev_n1 = 0;
    int ord = 0;
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
      if (is_v && ord > 0) {
        // The previous item's O is staged in the V ring once both of its
        // tiles' last PVs are done: V warp 4 stores it and frees the ring
        if (share == 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.ostage_full), (uint32_t)((ord - 1) & 1), abort_flag, wl));
          if (!ok) break;
          store_staged_pair<C>(&tm_o, o_tma, a, v_s, G, bq, prev_hk, prev_tok, prev_n0, prev_n1, lane, false,
                            smem_u32(&ctl.ostage_free));
        }
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
      for (; ul < C::UPT * n_tiles; ++ul) {            // unit ul of this item: tile ul / UPT, part ul % UPT
        const int u = u_base + ul;
        const int slot_i = (int)(u % SU);
        if (u >= SU) {
          const uint32_t empty = smem_u32(is_v ? &ctl.v_empty[slot_i] : &ctl.k_empty[slot_i]);
          ok = __all_sync(0xffffffffu,
                          mbar_wait(empty, (uint32_t)(((u / SU) - 1) & 1), abort_flag, wl));
          if (!ok) break;
        }
        const int t = ul / C::UPT, half = ul % C::UPT;
        const uint32_t full = smem_u32(is_v ? &ctl.v_full[slot_i] : &ctl.k_full[slot_i]);
        const uint32_t dst = (is_v ? v_s : k_s) + slot_i * C::UNIT;
        if (share == 0 && lane == 0) mbar_expect_tx(full, C::UNIT);
        __syncwarp();
        // K: unit = 64-column chunk `half` of tile t's 128 keys; V: key part `half`
        const int b0 = is_v ? (C::UPT * t + half) * boxes : t * boxes;
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
        const int x = (is_v ? c : half) * 64;
        const uint32_t d = dst + c * (is_v ? C::VU_CHUNK : C::KU_CHUNK) + i * R * 128;
        if (lane < boxes * uch && lane % nsh == share) tma_load_3d(d, map, x, it.hk, slot, full);
      }
      u_base += ul;
      if (!ok) break;
      prev_hk = it.hk;
      prev_tok = it.qstart + it.qpos_lo;
      prev_n0 = max(0, min(bq, it.qlen - it.qpos_lo));
      prev_n1 = max(0, min(bq, it.qlen - it.qpos_lo - bq));
    }
    if (is_v && share == 0) {
      // the last item's O
      if (ok && ord > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.ostage_full), (uint32_t)((ord - 1) & 1), abort_flag, wl));
        if (ok) store_staged_pair<C>(&tm_o, o_tma, a, v_s, G, bq, prev_hk, prev_tok, prev_n0, prev_n1, lane, true, 0u);
      }
      if (lane == 0) bulk_wait_all();                   // every store has landed before the CTA exits
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report(a.err, SWA_ERR_TIMEOUT);
    }
    // drain: every load issued by this warp must have landed before the CTA exits
    if (lane == 0) {
      for (int u = max(0, u_base - SU); u < u_base; ++u)
        mbar_wait(smem_u32(is_v ? &ctl.v_full[u % SU] : &ctl.k_full[u % SU]), (uint32_t)((u / SU) & 1), nullptr, kWaitLimitNs);
    }
  } else if (warp == 1 || warp == 3) {
    // =============================== MMA issuers ================================
    // Warp 1 issues QK_A(t), QK_B(t) into the shared S buffer, each once the
    // previous QK's scores have been loaded by their softmax (s_free); warp 3
    // issues PV_A(t), PV_B(t) from P_A, P_B.
    if (lane == 0 && warp == 1) {
      bool ok = true;
      int ord = 0;
      int n_q = 0;                                      // Q copies issued
      int n_qk = 0;                                     // QKs issued (both tiles)
      RingPos kp;
      while (ok) {
        // the item's record (n_tiles 0: the end of the stream), then Q_A and
        // Q_B, once the previous item's last QK_B is done with them (this
        // thread would wait for the copy before its next MMA anyway)
        const int rs = ord % kRecSlots;
        ok = mbar_wait(smem_u32(&ctl.rec_full[rs]), (uint32_t)((ord / kRecSlots) & 1), abort_flag, wl);
        if (!ok) break;
        const int n = ctl.rec[rs].n_tiles;
        const int q_hk = ctl.rec[rs].it.hk, q_tok = ctl.rec[rs].it.qstart + ctl.rec[rs].it.qpos_lo;
        mbar_arrive(smem_u32(&ctl.rec_empty[rs]));
        if (n == 0) break;
        if (ord > 0) ok = mbar_wait(smem_u32(&ctl.q_empty), (uint32_t)((ord - 1) & 1), abort_flag, wl);
        if (!ok) break;
        mbar_expect_tx(smem_u32(&ctl.q_full), 2 * C::Q_BYTES);
        for (int x = 0; x < 2; ++x)
          for (int c = 0; c < C::CH; ++c)
            tma_load_3d(q_s + x * C::Q_BYTES + c * C::Q_CHUNK, &tm_q, c * 64, q_hk * G, q_tok + x * bq,
                        smem_u32(&ctl.q_full));
        ++n_q;
        ok = mbar_wait(smem_u32(&ctl.q_full), (uint32_t)(ord & 1), abort_flag, wl);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; ok && j < n; ++j) {
          const RingPos k0 = kp;                        // the tile's K units (one per 64 columns)
          RingPos k1 = kp;
          if (C::UPT > 1) k1.next(C::KSU);
          for (int x = 0; ok && x < 2; ++x) {
            if (C::SEP_S ? n_qk > 1 : n_qk > 0) {
              // shared S: the previous QK's scores (the other tile's) were loaded;
              // S_X: this tile's previous scores were loaded
              ok = C::SEP_S ? mbar_wait(smem_u32(&ctl.s_free[x]), (uint32_t)(((n_qk >> 1) - 1) & 1), abort_flag, wl)
                            : mbar_wait(smem_u32(&ctl.s_free[0]), (uint32_t)((n_qk - 1) & 1), abort_flag, wl);
              if (!ok) break;
              tc_fence_after();
            }
            for (int half = 0; ok && half < C::UPT; ++half) {  // K unit = one 64-column chunk of head_dim
              const RingPos &kh = half ? k1 : k0;
              if (x == 0) {
                ok = mbar_wait(smem_u32(&ctl.k_full[kh.slot]), kh.phase, abort_flag, wl);
                if (!ok) break;
                tc_fence_after();
              }
              const uint32_t qa = q_s + x * C::Q_BYTES + half * C::Q_CHUNK;
              const uint32_t kb = k_s + kh.slot * C::UNIT;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)              // 16-column steps over the 64 columns
                mma_ss(tmem + C::TM_S + (C::SEP_S ? (uint32_t)x * C::N : 0u), smem_desc_sw128(qa + kk * 32, 16, 1024),
                       smem_desc_sw128(kb + kk * 32, 16, 1024), C::IDESC_QK, (half > 0 || kk > 0) ? 1u : 0u);
              if (x == 1) mma_commit(smem_u32(&ctl.k_empty[kh.slot]));
            }
            if (!ok) break;
            mma_commit(smem_u32(&ctl.s_full[x]));
            ++n_qk;
          }
          kp = k1;
          kp.next(C::KSU);
          if (ok && j == n - 1) mma_commit(smem_u32(&ctl.q_empty));   // the item's Q is no longer read
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
      uint32_t tpar = 0;                                // parity of this CTA's tile count
      RingPos vp;
      for (int ord = 0; ok; ++ord) {
        // the item's record (n_tiles 0: the end of the stream)
        const int rs = ord % kRecSlots;
        ok = mbar_wait(smem_u32(&ctl.rec_full[rs]), (uint32_t)((ord / kRecSlots) & 1), abort_flag, wl);
        if (!ok) break;
        const int n_tiles = ctl.rec[rs].n_tiles;
        mbar_arrive(smem_u32(&ctl.rec_empty[rs]));
        if (n_tiles == 0) break;
        for (int j = 0; ok && j < n_tiles; ++j, tpar ^= 1u) {
          const RingPos v0 = vp;
          RingPos v1 = vp;
          if (C::UPT > 1) v1.next(C::VSU);
          for (int x = 0; ok && x < 2; ++x) {
            ok = mbar_wait(smem_u32(&ctl.p_full[x]), tpar, abort_flag, wl);
            if (!ok) break;
            tc_fence_after();
            for (int half = 0; ok && half < C::UPT; ++half) {  // V unit = N / UPT keys of the tile
              const RingPos &vh = half ? v1 : v0;
              if (x == 0) {
                ok = mbar_wait(smem_u32(&ctl.v_full[vh.slot]), vh.phase, abort_flag, wl);
                if (!ok) break;
                tc_fence_after();
              }
              const uint32_t p_t = tmem + C::TM_P + (uint32_t)x * (C::N / 2) + half * (C::VU_KEYS / 16) * 8;
              const uint32_t vb = v_s + vh.slot * C::UNIT;
#pragma unroll
              for (int kk = 0; kk < C::VU_KEYS / 16; ++kk)
                mma_ts(tmem + C::TM_O + (uint32_t)x * C::D, p_t + kk * 8,
                       smem_desc_sw128(vb + kk * 16 * 128, C::VU_CHUNK, 1024), C::IDESC_PV,
                       (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
              if (x == 1) mma_commit(smem_u32(&ctl.v_empty[vh.slot]));
            }
            if (!ok) break;
            mma_commit(smem_u32(&ctl.o_full[x]));
            if (j == n_tiles - 1) mma_commit(smem_u32(&ctl.o_item[x]));   // the item's O_X is final
          }
          vp = v1;
          vp.next(C::VSU);
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
          !__all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&ctl.rec_empty[rs]),
                                                   (uint32_t)(((ord / kRecSlots) - 1) & 1), abort_flag, wl)))
        return false;
      write_rec(ctl.rec[rs], it, key_lo, n_tiles, hl, nr, rrs, rre, lane);
      if (lane == 0) mbar_arrive(smem_u32(&ctl.rec_full[rs]));
      ++ord;
      return true;
    };
    for (int item = blockIdx.x; ok && item < n_items; item += stride) {
      Item it;
      int32_t eb;
      if (!decode_item(a, item, bq2, it, eb)) {
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
  // warp 2 has no role: it only gives its registers to the softmax
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::HIGH_REGS));
    // =============================== softmax ====================================
    // Warpgroup x (0: tile A, 1: tile B); thread i owns row i of its tile: all
    // N columns of S_x and all D columns of O_x.  The running max is kept in
    // the log2 domain on raw scores (the scale is folded into the exponent's
    // FFMA), O_x is rescaled in TMEM only when the max grows by more than 2^8.
    constexpr int N = C::N;
    const int x = (warp - 8) >> 2;
    const int sid = threadIdx.x - 256 - 128 * x;         // 0 .. 127 within the warpgroup
    const int row = 32 * (warp & 3) + lane;              // TMEM lane of this thread
    const uint32_t lane_t = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t s_col = tmem + lane_t + C::TM_S + (C::SEP_S ? (uint32_t)x * N : 0u);
    const uint32_t p_col = tmem + lane_t + C::TM_P + (uint32_t)x * (N / 2);
    const uint32_t o_col = tmem + lane_t + C::TM_O + (uint32_t)x * C::D;
    const float asl2 = fmaxf(fabsf(a.scale * kLog2e), 1.17549435e-38f);
    int t = 0;                                           // this CTA's tiles so far
    int n_done = 0;                                      // items finished
    // Items come from the scheduler's records; the next one is set up while
    // the current item's last PV runs.
    RowSetup cur;
    bool have = false;
    auto next_rec = [&]() -> bool {                      // false: the wait ran out
      const int slot = n_done % kRecSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.rec_full[slot]),
                                             (uint32_t)((n_done / kRecSlots) & 1), abort_flag, wl)))
        return false;
      have = ctl.rec[slot].n_tiles > 0;
      if (have) row_setup_rec(a, ctl.rec[slot], row, G, lane, cur, x * bq);   // this warpgroup's tile of the pair
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
        const int kt0 = key_lo + j * N;
        ok = mbar_wait(smem_u32(&ctl.s_full[x]), (uint32_t)(t & 1), abort_flag, wl);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t raw[N];
        float lred[N / 32];                               // per 32 columns: max of S (min for NEG)
#pragma unroll
        for (int c = 0; c < N / 32; ++c)
          tmem_ld32_red<NEG>(s_col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * c), lred[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl.s_free[C::SEP_S ? x : 0]));   // S may take the next QK
        float xv[N];
        float mx;
        if (__all_sync(0xffffffffu, klo <= kt0 && khi >= kt0 + N - 1)) {
#pragma unroll
          for (int c = 0; c < N; ++c) xv[c] = NEG ? -__uint_as_float(raw[c]) : __uint_as_float(raw[c]);
          float r = lred[0];
#pragma unroll
          for (int c = 1; c < N / 32; ++c) r = NEG ? fminf(r, lred[c]) : fmaxf(r, lred[c]);
          mx = NEG ? -r : r;
        } else {
          // column c is visible when c_lo <= c <= c_lo + span: one unsigned compare
          // (an empty interval puts c_lo past the tile, so c - c_lo wraps above span)
          const bool empty = khi < klo;
          const int c_lo = empty ? 2 * N : klo - kt0;
          const uint32_t c_span = empty ? 0u : (uint32_t)(khi - klo);
#pragma unroll
          for (int c = 0; c < N; ++c)
            xv[c] = (uint32_t)(c - c_lo) <= c_span ? (NEG ? -__uint_as_float(raw[c]) : __uint_as_float(raw[c]))
                                                   : -INFINITY;
          float m4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = xv[i];
#pragma unroll
          for (int c = 4; c + 8 <= N; c += 8)
#pragma unroll
            for (int i = 0; i < 4; ++i) m4[i] = fmax3(m4[i], xv[c + 2 * i], xv[c + 2 * i + 1]);
#pragma unroll
          for (int c = 4 + ((N - 4) / 8) * 8; c < N; ++c) m4[c & 3] = fmaxf(m4[c & 3], xv[c]);
          mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        }
        mx = mx == -INFINITY ? -INFINITY : mx * asl2;
        const float m_new = fmaxf(m_used, mx);
        const bool need = m_new > m_used + 8.f;           // also true on the first visible tile
        if (__any_sync(0xffffffffu, need)) {
          const float m_next = need ? m_new : m_used;
          const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_next);
          if (j > 0) {
            // PV_x(t-1) must be complete before O_x is rescaled.  The P store
            // of tile t-1 waited for PV_x(t-2), so the o_full phase of
            // PV_x(t-1) is the only one that can still be open.
            ok = mbar_wait(smem_u32(&ctl.o_full[x]), (uint32_t)((t - 1) & 1), abort_flag, wl);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < C::D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(o_col + 32 * c, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(o_col + 32 * c, r);
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
        uint64_t s2[2] = {0, 0};                         // two paired partial sums (0.0f bits)
        if (x == 0 && kt0 + N > it.seq_len) {
          // keys past the sequence end: their V rows may hold anything; zero
          // them before P_A(t) is published (PV_B(t) follows PV_A(t)).  V unit
          // UPT t + half is the latest fill of its slot (tile t-1's units sit in
          // other slots, which PV_B(t-1) may still read), so its v_full parity
          // is unambiguous.
          for (int half = 0; half < C::UPT && ok; ++half) {
            const int k0 = kt0 + half * C::VU_KEYS;
            if (k0 + C::VU_KEYS <= it.seq_len) continue;
            const uint32_t u = (uint32_t)C::UPT * (uint32_t)t + half;
            const int slot = (int)(u % C::VSU);
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.v_full[slot]), (u / C::VSU) & 1u, abort_flag,
                                                   wl));
            if (!ok) break;
            const int r0 = max(0, it.seq_len - k0);       // first row to clear
            uint8_t *unit = dsm_ptr + C::OFF_V + slot * C::UNIT;
#pragma unroll 1
            for (int i = sid; i < C::CH * C::VU_KEYS * 8; i += 128) {   // 16-byte pieces: chunk, row, piece
              const int r = (i >> 3) & (C::VU_KEYS - 1);
              if (r >= r0)
                *reinterpret_cast<uint4 *>(unit + (i / (C::VU_KEYS * 8)) * C::VU_CHUNK + r * 128 + (i & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
            }
          }
          if (!ok) break;
          fence_proxy_async_smem();
        }
        if (t > 0) {
          // P_x(t) overwrites P_x(t-1): PV_x(t-1) must have read it
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.o_full[x]), (uint32_t)((t - 1) & 1), abort_flag, wl));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {                 // P in two stores of 32 columns (64 keys each)
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float e0, e1;
            f2_unpack(f2_fma(f2_pack(xv[64 * hh + 2 * c], xv[64 * hh + 2 * c + 1]), sl2x2, nms), e0, e1);
            const float p0 = ex2(e0), p1 = ex2(e1);
            s2[c & 1] = f2_add(s2[c & 1], f2_pack(p0, p1));
            pk[c] = pack_bf16(p0, p1);
          }
          tmem_st32(p_col + 32 * hh, pk);
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(s2[0], a0, a1);
          f2_unpack(s2[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl.p_full[x]));
      }
      if (!ok) break;
      const bool row_valid = cur.row_valid;
      const int64_t out_row = cur.out_row;
      ++n_done;
      if (!next_rec()) { ok = false; break; }
      // the item's last PVs of both tiles (one o_item phase per tile and item):
      // the V ring, where O is staged, is then free of both tiles' V units
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl.o_item[x]), (uint32_t)((n_done - 1) & 1), abort_flag, wl) &&
                                   mbar_wait(smem_u32(&ctl.o_item[x ^ 1]), (uint32_t)((n_done - 1) & 1), abort_flag, wl));
      if (!ok) break;
      // epilogue: O / l -> bf16 rows in the V ring (the V producers wait for
      // ostage_free), tile X's 64-column chunks at CH X O_CHUNK, laid out as
      // the output map's boxes with the 128-byte swizzle; V warp 4 stores them.
      // The next item's first PV_x overwrites O_x only after this thread's P
      // for it (published after these loads completed).
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < C::D / 64; ++c) {
        uint32_t r[64];
        tmem_ld32(o_col + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld32(o_col + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        const uint32_t rb = v_s + (uint32_t)((x * C::CH + c) * C::O_CHUNK + row * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_shared_v4(rb + ((uint32_t)(j ^ (row & 7)) << 4),
                       pack_bf16(__uint_as_float(r[8 * j]) * inv, __uint_as_float(r[8 * j + 1]) * inv),
                       pack_bf16(__uint_as_float(r[8 * j + 2]) * inv, __uint_as_float(r[8 * j + 3]) * inv),
                       pack_bf16(__uint_as_float(r[8 * j + 4]) * inv, __uint_as_float(r[8 * j + 5]) * inv),
                       pack_bf16(__uint_as_float(r[8 * j + 6]) * inv, __uint_as_float(r[8 * j + 7]) * inv));
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&ctl.ostage_full));
      if (row_valid && a.lse != nullptr) a.lse[out_row] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
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
cudaError_t run_pair(const AttnArgs &a, cudaStream_t st) {
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
  constexpr int smem = pair_smem_bytes<C>();
  static_assert(smem <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_tc_pair_kernel<C, NEG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (a.num_tokens / (2 * bq) + a.num_seqs) * (int64_t)a.hkv;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = (int)(items < sms ? items : (int64_t)sms);
  // The register split hands over exactly the launch allocation: a kernel built
  // with another per-thread count would wait forever in setmaxnreg.inc.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, attn_tc_pair_kernel<C, NEG>) != cudaSuccess || fa.numRegs != C::LAUNCH_REGS)
    return cudaErrorInvalidConfiguration;
  attn_tc_pair_kernel<C, NEG><<<grid, C::THREADS, smem, st>>>(mq, mk, mv, mo, a, G, (int)items, o_tma);
  return cudaGetLastError();
}

using Pair128 = PairCfg<128, 5>;   // K and V rings of 5 units
using Pair64 = PairCfg<64, 6>;     // Q tiles of 16 KB leave room for 6 + 6

}  // namespace

bool tc_pair_supported(const AttnArgs &a) { return (a.head_dim == 128 || a.head_dim == 64) && tc_prefill_ok(a); }

cudaError_t launch_attention_tc_pair(const AttnArgs &a, cudaStream_t st) {
  // the sign of the scale is a template argument, as in attention_tc.cu
  if (a.head_dim == 64) return a.scale < 0.f ? run_pair<Pair64, true>(a, st) : run_pair<Pair64, false>(a, st);
  return a.scale < 0.f ? run_pair<Pair128, true>(a, st) : run_pair<Pair128, false>(a, st);
}

}  // namespace swa
