"""Pins for the oracle's KV-cache write and context-parallel slot mapping.

Sources: the vllm-ascend slot-mapping article -- section 2 (non-CP formula),
section 3.1 steps 1-5 (interleaved CP slot formula) and section 3.3 (worked
example: W=2, interleave 128, block 128); the DCP decode study notes,
section 1.1 (partials merged by LSE equal one softmax over the sequence).
"""
import numpy as np
import pytest

from oracle import swa_oracle as O


def _random_requests(rng, n_req, max_len, block_size, spare=8):
    lens = rng.integers(1, max_len + 1, size=n_req)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    positions = np.concatenate([np.arange(int(n)) for n in lens]).astype(np.int64)
    pages = -(-int(lens.max()) // block_size) + spare
    bt = rng.permutation(n_req * pages).reshape(n_req, pages).astype(np.int64)
    return qsl, positions, bt


@pytest.mark.parametrize("seed", range(12))
def test_cp_with_one_rank_is_the_plain_mapping(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([1, 4, 16, 64]))
    qsl, pos, bt = _random_requests(rng, 3, 300, bs)
    T = int(qsl[-1])
    plain, bad_p = O.slot_mapping(qsl, pos, bt, bs, T, T + 5)
    for kvb in (bs, 2 * bs, 4 * bs):
        cp, bad_c = O.slot_mapping_cp(qsl, pos, bt, bs, T + 5, kvb, 1, 0, 1)
        assert np.array_equal(cp, plain) and bad_c == bad_p


def test_cp_worked_example_section_3_3():
    # W=2, interleave 128, block 128: positions 0..127 and 256..383 on rank 0,
    # 128..255 and 384..511 on rank 1; a rank's segments are concatenated.
    bt = np.array([[7, 3, 11, 5]])
    pos = np.arange(512)
    qsl = [0, 512]
    r0, _ = O.slot_mapping_cp(qsl, pos, bt, 128, 512, 128, 2, 0, 128)
    r1, _ = O.slot_mapping_cp(qsl, pos, bt, 128, 512, 128, 2, 1, 128)
    exp0 = np.full(512, -1)
    exp0[0:128] = 7 * 128 + np.arange(128)          # local offsets 0..127 -> block index 0
    exp0[256:384] = 3 * 128 + np.arange(128)        # local offsets 128..255 -> block index 1
    exp1 = np.full(512, -1)
    exp1[128:256] = 7 * 128 + np.arange(128)
    exp1[384:512] = 3 * 128 + np.arange(128)
    assert np.array_equal(r0, exp0) and np.array_equal(r1, exp1)


@pytest.mark.parametrize("seed", range(10))
def test_cp_each_token_on_exactly_one_rank_and_ranks_are_contiguous(seed):
    rng = np.random.default_rng(100 + seed)
    bs = int(rng.choice([4, 16]))
    W = int(rng.choice([2, 3, 4]))
    bpk = int(rng.choice([1, 2, 4]))
    kvb = bs * bpk
    divisors = [d for d in range(1, kvb + 1) if kvb % d == 0]
    I = int(rng.choice(divisors))
    qsl, pos, bt = _random_requests(rng, 2, 400, bs, spare=400 // bs + 8)
    T = int(qsl[-1])
    maps = [O.slot_mapping_cp(qsl, pos, bt, bs, T, kvb, W, r, I)[0] for r in range(W)]
    owners = np.stack([m >= 0 for m in maps]).sum(axis=0)
    assert np.all(owners == 1)
    for r in range(W):
        for q in range(len(qsl) - 1):
            toks = [t for t in range(int(qsl[q]), int(qsl[q + 1])) if maps[r][t] >= 0]
            # the j-th token this rank owns sits at local offset j: the plain
            # formula applied to j with this rank's block-table row
            got = np.array([maps[r][t] for t in sorted(toks, key=lambda t: pos[t])])
            j = np.arange(len(toks))
            exp = bt[q, j // bs] * bs + j % bs
            assert np.array_equal(got, exp)


def test_cp_rejects_inconsistent_geometry():
    with pytest.raises(ValueError):
        O.slot_mapping_cp([0, 4], np.arange(4), np.zeros((1, 4), int), 16, 4, 24, 2, 0, 8)  # 16 does not divide 24
    with pytest.raises(ValueError):
        O.slot_mapping_cp([0, 4], np.arange(4), np.zeros((1, 4), int), 16, 4, 32, 2, 2, 8)  # rank >= W


def test_kv_cache_write_pads_bad_slots_and_round_trip():
    rng = np.random.default_rng(5)
    bs, hkv, d = 16, 2, 8
    qsl, pos, bt = _random_requests(rng, 3, 50, bs)
    T = int(qsl[-1])
    slots, _ = O.slot_mapping(qsl, pos, bt, bs, T, T + 3)
    nblocks = int(bt.max()) + 1
    kc = rng.standard_normal((nblocks, bs, hkv, d))
    vc = rng.standard_normal((nblocks, bs, hkv, d))
    kn = rng.standard_normal((T + 3, hkv, d))
    vn = rng.standard_normal((T + 3, hkv, d))
    slots = slots.astype(np.int64)
    slots[T + 1] = nblocks * bs + 4                  # out of range: reported, not written
    k2, v2, bad = O.kv_cache_write(kn, vn, slots, kc, vc)
    assert bad == [T + 1]
    flat_k, flat_v = k2.reshape(-1, hkv, d), v2.reshape(-1, hkv, d)
    written = set()
    for t in range(T):
        s = int(slots[t])
        assert np.array_equal(flat_k[s], kn[t]) and np.array_equal(flat_v[s], vn[t])
        written.add(s)
    untouched = [s for s in range(nblocks * bs) if s not in written]
    assert np.array_equal(flat_k[untouched], kc.reshape(-1, hkv, d)[untouched])
    # the attention gather through the block table sees exactly the new rows
    for r in range(len(qsl) - 1):
        L = int(qsl[r + 1] - qsl[r])
        g = O._gather(k2, bt[r], L, bs, 1)
        assert np.array_equal(g, kn[int(qsl[r]):int(qsl[r + 1]), 1])


@pytest.mark.parametrize("W,I", [(2, 16), (4, 16), (3, 32), (2, 64)])
def test_rank_split_decode_merges_to_full_attention(W, I):
    """Context-parallel decode on simulated ranks: every rank attends over the
    keys it owns, the partials are merged by LSE, and the result is one
    softmax over the whole sequence (DCP notes, section 1.1)."""
    rng = np.random.default_rng(W * 100 + I)
    bs, hq, hkv, d = 16, 4, 2, 16
    lens = np.array([300, 129, 517])
    S = len(lens)
    kv_seq = [(rng.standard_normal((int(n), hkv, d)), rng.standard_normal((int(n), hkv, d))) for n in lens]
    q = rng.standard_normal((S, hq, d))
    scale = d ** -0.5
    # the full attention: one query per sequence at its last position, causal, no window
    pages = -(-int(lens.max()) // bs) + 2
    bt_full = rng.permutation(S * pages).reshape(S, pages)
    kc = np.zeros((S * pages, bs, hkv, d))
    vc = np.zeros_like(kc)
    for s in range(S):
        for p in range(int(lens[s])):
            blk, off = bt_full[s, p // bs], p % bs
            kc[blk, off], vc[blk, off] = kv_seq[s][0][p], kv_seq[s][1][p]
    qsl = np.arange(S + 1)
    full_out, full_lse = O.attention(q, kc, vc, bt_full, qsl, lens, None, 0, True, scale)
    # per rank: its own block table and cache, filled through the CP slot mapping
    part_out = np.zeros((W, S, hq, d))
    part_lse = np.full((W, S, hq), -np.inf)
    for r in range(W):
        bt_r = rng.permutation(S * pages).reshape(S, pages)
        ctx_qsl = np.concatenate([[0], np.cumsum(lens)])
        positions = np.concatenate([np.arange(int(n)) for n in lens])
        kvb = int(np.lcm(bs, I))                         # the interleave must divide the kv-cache block
        slots, bad = O.slot_mapping_cp(ctx_qsl, positions, bt_r, bs, int(ctx_qsl[-1]), kvb, W, r, I)
        assert not bad
        kn = np.concatenate([kv_seq[s][0] for s in range(S)])
        vn = np.concatenate([kv_seq[s][1] for s in range(S)])
        kc_r, vc_r, bad = O.kv_cache_write(kn, vn, slots, np.zeros_like(kc), np.zeros_like(vc))
        assert not bad
        n_local = np.array([int(np.sum(slots[int(ctx_qsl[s]):int(ctx_qsl[s + 1])] >= 0)) for s in range(S)])
        # every local key is visible to the query (it is the sequence's last position)
        o, l = O.attention(q, kc_r, vc_r, bt_r, qsl, n_local, None, 0, False, scale)
        for s in range(S):
            for h in range(hq):
                part_out[r, s, h] = o[(s, h)]
                part_lse[r, s, h] = l[(s, h)]
    mo, ml = O.lse_combine(part_out, part_lse)
    for s in range(S):
        for h in range(hq):
            assert np.allclose(mo[s, h], full_out[(s, h)], atol=1e-12)
            assert abs(ml[s, h] - full_lse[(s, h)]) < 1e-12


def test_slot_mapping_positions_derived_from_context_lengths():
    """Without positions, request r's i-th token sits after its cached context:
    the same slots as explicit positions ctx[r] + i; a worked case by hand."""
    bt = np.array([[5, 2, 9], [7, 1, 0]])
    qsl = [0, 3, 5]
    ctx = [14, 0]                                   # request 0: positions 14, 15, 16; request 1: 0, 1
    got, bad = O.slot_mapping(qsl, None, bt, 8, 5, 8, context_lens=ctx)
    # 14 -> page 1 (block 2) offset 6 = 22; 15 -> 23; 16 -> page 2 (block 9) offset 0 = 72; 0 -> 56; 1 -> 57
    assert got.tolist() == [22, 23, 72, 56, 57, -1, -1, -1] and bad == []
    rng = np.random.default_rng(9)
    for _ in range(5):
        qsl, pos, bt = _random_requests(rng, 3, 200, 16)
        ctxs = rng.integers(0, 300, size=3)
        explicit = np.concatenate([ctxs[r] + np.arange(int(qsl[r + 1] - qsl[r])) for r in range(3)])
        bt = np.tile(np.arange(64), (3, 1))
        a, ba = O.slot_mapping(qsl, None, bt, 16, int(qsl[-1]), int(qsl[-1]) + 4, context_lens=ctxs)
        b, bb = O.slot_mapping(qsl, explicit, bt, 16, int(qsl[-1]), int(qsl[-1]) + 4)
        assert np.array_equal(a, b) and ba == bb
