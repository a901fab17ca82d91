"""Pins the CPU oracle to facts fixed outside itself.

Each test checks the oracle against something it does not compute itself:
values printed on the pages (tests/golden), closed forms derived by hand,
library routines the method reduces to (torch's fp64 scaled-dot-product
attention), invariants (paging, GQA head sharing, the log-sum-exp identity),
and brute force over tiny inputs.  The last tests plant plausible mistakes in
copies of oracle functions and check that a pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import swa_oracle as O


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# tile bounds: the pages' printed geometry
# ---------------------------------------------------------------------------
def _geometry_bounds(causal, ranges, g):
    qsl = np.array([0, g["query_len"]])
    seq = np.array([g["seq_len"]])
    mm = np.array([ranges], dtype=np.int32)
    tb = O.tile_bounds(qsl, seq, mm, g["window"], causal, g["tile_size"], g["block_q"],
                       max_qblocks=g["q_block_local_idx"] + 1)
    return tb[0, g["q_block_local_idx"]].tolist()


def test_tile_bounds_printed_causal(golden_dir):
    gd = _load(golden_dir, "tile_bounds_pages.json")
    c = gd["cases"][0]
    assert _geometry_bounds(c["causal"], c["mm_ranges"], gd["geometry"]) == c["expect"]


def test_tile_bounds_printed_noncausal_right_window(golden_dir):
    gd = _load(golden_dir, "tile_bounds_pages.json")
    c = gd["cases"][1]
    lo, hi, _ = _geometry_bounds(c["causal"], c["mm_ranges"], gd["geometry"])
    assert [lo, hi] == c["expect_lo_hi"]
    # the first-version bug (right edge = last query row) would stop at tile 40
    assert hi > 1127 // 32 + 1


def test_tile_bounds_pruning_happens(golden_dir):
    gd = _load(golden_dir, "tile_bounds_pages.json")
    lo, hi, _ = _geometry_bounds(True, gd["cases"][0]["mm_ranges"], gd["geometry"])
    full = gd["full_scan_without_pruning"]
    assert (hi - lo) < (full[1] - full[0])


# ---------------------------------------------------------------------------
# the visibility rule: closed form, hand-derived cases, the tiny config count
# ---------------------------------------------------------------------------
def _interval(q, seq_len, window, causal, ranges):
    """Hand-derived closed form: the visible keys of q are one interval."""
    lo = max(0, q - window + 1) if window > 0 else 0
    if window > 0:
        hi = q if causal else q + window - 1
    else:
        hi = q if causal else seq_len - 1
    if ranges is not None:
        for s, e in ranges:
            if s < e and s <= q <= e:
                hi = max(hi, e)
    return lo, min(hi, seq_len - 1)


@pytest.mark.parametrize("seed", range(40))
def test_mask_is_one_interval_per_query(seed):
    rng = np.random.default_rng(seed)
    seq_len = int(rng.integers(1, 120))
    window = int(rng.choice([0, -3, 1, 2, 5, 17, 200]))
    causal = bool(rng.integers(0, 2))
    ranges = []
    for _ in range(int(rng.integers(0, 5))):
        a = int(rng.integers(0, seq_len))
        b = int(rng.integers(a, seq_len))
        ranges.append((a, b))
    ranges.append((0, 0))
    for q in range(seq_len):
        vis = O.visible_keys(q, seq_len, window, causal, np.array(ranges))
        lo, hi = _interval(q, seq_len, window, causal, ranges)
        expect = np.zeros(seq_len, bool)
        expect[lo:hi + 1] = True
        assert np.array_equal(vis, expect), (q, lo, hi, np.nonzero(vis)[0])


@pytest.mark.parametrize("q,causal,expect", [
    (8, True, [7, 8, 9, 10, 11]),     # image [4, 11] re-opens keys up to its end
    (4, True, list(range(3, 12))),    # first image row: window edge 3 .. image end 11
    (12, True, [11, 12]),             # outside the image: plain window
    (3, True, [2, 3]),
    (3, False, [2, 3, 4]),            # non-causal right window
    (8, False, [7, 8, 9, 10, 11]),    # image end beats the right window (9)
    (11, False, [10, 11, 12]),
])
def test_mask_hand_cases(q, causal, expect):
    vis = O.visible_keys(q, 16, 2, causal, np.array([[4, 11], [0, 0]]))
    assert np.nonzero(vis)[0].tolist() == expect


def test_mask_tiny_config_pair_count():
    # hand count for 256 tokens, W=64, causal, image [40,120]:
    # q<40: q+1 -> 820; 40..63: keys 0..120 -> 24*121 = 2904;
    # 64..120: keys q-63..120 -> sum_{j=64}^{120} j = 5244; 121..255: 64 each -> 8640.
    lay = W.tiny()
    n = O.allowed_pair_count(lay.query_start_loc, lay.seq_lens, lay.mm_ranges, lay.window, lay.causal)
    assert n == 820 + 2904 + 5244 + 8640 == 17608


def test_one_token_image_adds_nothing():
    for q in range(10):
        a = O.visible_keys(q, 10, 3, True, np.array([[5, 5]]))
        b = O.visible_keys(q, 10, 3, True, None)
        assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# tile bounds: brute force against the mask
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(60))
def test_tile_bounds_cover_every_visible_key(seed):
    rng = np.random.default_rng(500 + seed)
    S = int(rng.integers(1, 4))
    qlen = rng.integers(0, 90, size=S)
    ctx = rng.integers(0, 90, size=S)
    seq = ctx + qlen
    window = int(rng.choice([0, 1, 3, 9, 33, 500]))
    causal = bool(rng.integers(0, 2))
    tile = int(rng.choice([1, 4, 8, 16, 32]))
    bq = int(rng.choice([1, 2, 3, 8, 16]))
    R = int(rng.integers(1, 4))
    mm = np.zeros((S, R, 2), dtype=np.int32)
    for s in range(S):
        for i in range(R):
            if seq[s] > 1 and rng.integers(0, 3):
                a = int(rng.integers(0, seq[s] - 1))
                mm[s, i] = (a, int(rng.integers(a, seq[s])))
    qsl = np.concatenate([[0], np.cumsum(qlen)])
    maxb = int(max(1, -(-qlen.max() // bq)))
    tb = O.tile_bounds(qsl, seq, mm, window, causal, tile, bq, maxb)
    for s in range(S):
        for b in range(maxb):
            rows = range(b * bq, min((b + 1) * bq, int(qlen[s])))
            if not rows:
                assert tb[s, b].tolist() == [0, 0, 0]
                continue
            keys = set()
            for i in rows:
                keys |= set(np.nonzero(O.visible_keys(ctx[s] + i, seq[s], window, causal, mm[s]))[0].tolist())
            lo, hi, _ = tb[s, b]
            tiles = {k // tile for k in keys}
            assert tiles <= set(range(lo, hi)), (s, b, lo, hi, sorted(tiles))
            if window > 0:
                # with a window the union formula is exact: no tile outside the key span
                assert lo == min(tiles) and hi == max(tiles) + 1


def test_tile_bounds_padding_ranges_equal_no_ranges():
    rng = np.random.default_rng(3)
    for _ in range(20):
        qlen = int(rng.integers(1, 200))
        ctx = int(rng.integers(0, 200))
        qsl, seq = np.array([0, qlen]), np.array([ctx + qlen])
        pad = np.zeros((1, 3, 2), dtype=np.int32)
        a = O.tile_bounds(qsl, seq, pad, 40, True, 16, 8, 30)
        b = O.tile_bounds(qsl, seq, None, 40, True, 16, 8, 30)
        assert np.array_equal(a[..., :2], b[..., :2])


# ---------------------------------------------------------------------------
# tile bounds: the third field, max_seq_prefix_len
# ---------------------------------------------------------------------------
def _random_blocks(seed, with_ranges):
    """Small random (sequence, query block) layouts with context and a ragged tail."""
    rng = np.random.default_rng(900 + seed)
    S = int(rng.integers(1, 4))
    qlen = rng.integers(1, 70, size=S)
    ctx = rng.integers(0, 70, size=S)
    seq = ctx + qlen
    mm = None
    if with_ranges:
        mm = np.zeros((S, 2, 2), dtype=np.int32)
        for s in range(S):
            a = int(rng.integers(0, seq[s]))
            mm[s, 0] = (a, int(rng.integers(a, seq[s])))
    qsl = np.concatenate([[0], np.cumsum(qlen)])
    return rng, qsl, ctx, seq, mm


def _max_visible_key_plus_one(ctx, seq_len, rows, window, causal, mm_row, **kw):
    top = -1
    for i in rows:
        vis = np.nonzero(O.visible_keys(ctx + i, seq_len, window, causal, mm_row, **kw))[0]
        if vis.size:
            top = max(top, int(vis[-1]))
    return top + 1


@pytest.mark.parametrize("seed", range(30))
def test_max_prefix_is_the_block_key_bound_when_causal_without_images(seed):
    """Causal, no image ranges: the field is the exact bound on the keys the
    block's rows can see, 1 + the largest visible key (brute force over the
    per-pair rule), with and without chunked lookback, for every window."""
    rng, qsl, ctx, seq, _ = _random_blocks(seed, with_ranges=False)
    window = int(rng.choice([0, 1, 4, 9, 33, 500]))
    bq = int(rng.choice([1, 3, 8, 16]))
    tile = int(rng.choice([1, 4, 16]))
    kw = {}
    if window > 0 and rng.integers(0, 2):
        kw = dict(chunk_size=int(rng.choice([4, 8, 32])), chunk_lookback=int(rng.integers(0, 3)))
    maxb = int(-(-max(np.diff(qsl)) // bq))
    tb = O.tile_bounds(qsl, seq, None, window, True, tile, bq, maxb, **kw)
    for s in range(len(seq)):
        for b in range(maxb):
            rows = range(b * bq, min((b + 1) * bq, int(qsl[s + 1] - qsl[s])))
            if not rows:
                continue
            bound = _max_visible_key_plus_one(int(ctx[s]), int(seq[s]), rows, window, True, None, **kw)
            assert tb[s, b, 2] == bound, (s, b, tb[s, b].tolist(), bound)
            # the tile range lies inside the prefix the field announces
            assert tb[s, b, 1] <= -(-int(tb[s, b, 2]) // tile)


@pytest.mark.parametrize("seed", range(20))
def test_max_prefix_is_the_sequence_length_with_images_or_noncausal(seed):
    """With image ranges enabled, non-causal attention, or the per-sequence
    causal mode, the field is seq_len: the printed [3, 72, 4096] case of the
    PR #53147 geometry test generalised.  It still bounds every visible key."""
    for with_ranges, causal, per_seq in ((True, True, False), (False, False, False),
                                         (True, False, False), (False, True, True)):
        rng, qsl, ctx, seq, mm = _random_blocks(seed, with_ranges)
        window = int(rng.choice([0, 2, 9, 33]))
        bq = int(rng.choice([1, 4, 8]))
        maxb = int(-(-max(np.diff(qsl)) // bq))
        tb = O.tile_bounds(qsl, seq, mm, window, causal, 4, bq, maxb, per_seq_causal=per_seq)
        for s in range(len(seq)):
            for b in range(maxb):
                rows = range(b * bq, min((b + 1) * bq, int(qsl[s + 1] - qsl[s])))
                if not rows:
                    continue
                assert tb[s, b, 2] == seq[s]
                mm_row = None if mm is None else mm[s]
                assert tb[s, b, 2] >= _max_visible_key_plus_one(int(ctx[s]), int(seq[s]), rows,
                                                                window, causal, mm_row)


def test_max_prefix_pages_geometry_without_images():
    """The PR #53147 geometry (4096 tokens, W=1024, tile 32, block 8) without an
    image: rows 1120..1127 see keys 97..1127, so the prefix is 1128 keys and the
    tiles run [3, 36)."""
    qsl, seq = np.array([0, 4096]), np.array([4096])
    tb = O.tile_bounds(qsl, seq, None, 1024, True, 32, 8, 141)
    assert tb[0, 140].tolist() == [3, 36, 1128]


# ---------------------------------------------------------------------------
# attention: reduction to torch's fp64 scaled-dot-product attention
# ---------------------------------------------------------------------------
def _dense(lay, q, k, v):
    """Contiguous K/V of every sequence by reading the block table (test-side)."""
    out = []
    for s in range(lay.num_seqs):
        n = int(lay.seq_lens[s])
        pages = lay.block_table[s, :(n + lay.block_size - 1) // lay.block_size]
        kk = k[torch.from_numpy(pages.astype(np.int64))].reshape(-1, lay.num_heads_kv, lay.head_dim)[:n]
        vv = v[torch.from_numpy(pages.astype(np.int64))].reshape(-1, lay.num_heads_kv, lay.head_dim)[:n]
        out.append((kk.double(), vv.double()))
    return out


def _sdpa_case(lay, q, k, v, mask_fn):
    ref_out = torch.zeros(q.shape, dtype=torch.float64)
    qsl = lay.query_start_loc
    for s, (kk, vv) in enumerate(_dense(lay, q, k, v)):
        qs = q[qsl[s]:qsl[s + 1]].double()                   # [n_q, Hq, D]
        G = lay.group
        kk = kk.repeat_interleave(G, dim=1)
        vv = vv.repeat_interleave(G, dim=1)
        mask = mask_fn(qs.shape[0], kk.shape[0], int(lay.context_lens[s]))
        o = torch.nn.functional.scaled_dot_product_attention(
            qs.transpose(0, 1), kk.transpose(0, 1), vv.transpose(0, 1), attn_mask=mask,
            scale=lay.scale)
        ref_out[qsl[s]:qsl[s + 1]] = o.transpose(0, 1)
    return ref_out


def _oracle_all(lay, q, k, v):
    out, lse = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens,
                           lay.mm_ranges, lay.window, lay.causal, lay.scale)
    T, H, D = q.shape
    o = torch.zeros((T, H, D), dtype=torch.float64)
    for (t, h), val in out.items():
        o[t, h] = torch.from_numpy(val)
    return o, lse


def _small(seed, **kw):
    lay = W.random_small(seed, max_seqs=2, max_ctx=40, max_q=40, head_dim=kw.pop("head_dim", 16), **kw)
    q, k, v = W.make_tensors(lay, data_seed=seed)
    return lay, q, k, v


@pytest.mark.parametrize("seed", range(4))
def test_attention_full_causal_is_sdpa(seed):
    lay, q, k, v = _small(seed, window=100000, causal=True, with_ranges=False, dtype="fp32")
    ref = _sdpa_case(lay, q, k, v, lambda nq, nk, c: torch.ones(nq, nk, dtype=torch.bool).tril(c))
    got, _ = _oracle_all(lay, q, k, v)
    assert torch.allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("seed", range(4))
def test_attention_full_noncausal_is_sdpa(seed):
    lay, q, k, v = _small(seed, window=0, causal=False, with_ranges=False, dtype="fp32")
    ref = _sdpa_case(lay, q, k, v, lambda nq, nk, c: None)
    got, _ = _oracle_all(lay, q, k, v)
    assert torch.allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("seed,window,causal", [(0, 3, True), (1, 7, True), (2, 4, False), (3, 1, False)])
def test_attention_band_is_sdpa(seed, window, causal):
    lay, q, k, v = _small(seed, window=window, causal=causal, with_ranges=False, dtype="fp32")

    def band(nq, nk, c):
        ones = torch.ones(nq, nk, dtype=torch.bool)
        upper = ones.tril(c) if causal else ones.tril(c + window - 1)
        return upper & ones.triu(c - window + 1)
    ref = _sdpa_case(lay, q, k, v, band)
    got, _ = _oracle_all(lay, q, k, v)
    assert torch.allclose(got, ref, atol=1e-12, rtol=0)


def test_attention_single_visible_key_copies_v():
    lay, q, k, v = _small(5, window=1, causal=True, with_ranges=False, dtype="fp32")
    got, lse = _oracle_all(lay, q, k, v)
    dense = _dense(lay, q, k, v)
    qsl, ctx = lay.query_start_loc, lay.context_lens
    for s, (kk, vv) in enumerate(dense):
        for i in range(qsl[s + 1] - qsl[s]):
            t = qsl[s] + i
            for h in range(lay.num_heads_q):
                hk = h // lay.group
                assert torch.allclose(got[t, h], vv[ctx[s] + i, hk], atol=1e-12)
                s_qq = lay.scale * float(q[t, h].double() @ kk[ctx[s] + i, hk])
                assert abs(lse[(t, h)] - s_qq) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_attention_uniform_keys_average_the_visible_interval(causal):
    """K rows all equal -> uniform weights: out = mean of V over the visible keys."""
    seq_len, window, rngs = 40, 4, [(10, 25), (30, 31), (0, 0)]
    lay = W.Layout("hand", query_lens=np.array([seq_len], np.int32), seq_lens=np.array([seq_len], np.int32),
                   mm_ranges=np.array([rngs], np.int32), block_table=np.arange(5, dtype=np.int32)[None, ::-1].copy(),
                   num_blocks=5, num_heads_q=1, num_heads_kv=1, head_dim=2, block_size=8,
                   window=window, causal=causal, dtype="fp32")
    q = torch.ones(seq_len, 1, 2)
    k = torch.ones(5, 8, 1, 2)
    v = torch.zeros(5, 8, 1, 2)
    for j in range(seq_len):                # key j sits in page 4 - j // 8 (reversed table)
        v[4 - j // 8, j % 8, 0, 0] = j
        v[4 - j // 8, j % 8, 0, 1] = j * j
    out, lse = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                           window, causal, scale=0.5)
    for qq in range(seq_len):
        lo, hi = _interval(qq, seq_len, window, causal, rngs)
        js = np.arange(lo, hi + 1)
        assert np.allclose(out[(qq, 0)], [js.mean(), (js * js).mean()], atol=1e-12)
        assert abs(lse[(qq, 0)] - (0.5 * 2.0 + math.log(len(js)))) < 1e-12


def test_removing_image_ranges_changes_output():
    lay = W.tiny()
    q, k, v = W.make_tensors(lay)
    rows = [(t, h) for t in range(40, 121, 5) for h in range(2)]
    a, _ = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                       lay.window, lay.causal, lay.scale, rows=rows)
    b, _ = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, None,
                       lay.window, lay.causal, lay.scale, rows=rows)
    diff = max(np.abs(a[r] - b[r]).max() for r in rows)
    assert diff > 1e-3


def test_paging_is_invisible():
    lay, q, k, v = _small(7, window=9, causal=True, with_ranges=True, dtype="fp32", block_size=16)
    perm = np.random.default_rng(0).permutation(lay.num_blocks)
    inv = np.argsort(perm)
    k2, v2 = k[torch.from_numpy(inv)], v[torch.from_numpy(inv)]    # page p moves to perm[p]
    bt2 = np.where(lay.block_table >= 0, perm[np.maximum(lay.block_table, 0)], -1).astype(np.int32)
    a, la = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                        lay.window, lay.causal, lay.scale)
    b, lb = O.attention(q, k2, v2, bt2, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                        lay.window, lay.causal, lay.scale)
    for r in a:
        assert np.array_equal(a[r], b[r]) and la[r] == lb[r]


def test_gqa_heads_share_their_kv_head():
    lay, q, k, v = _small(8, window=5, causal=False, with_ranges=True, dtype="fp32", group=2)
    from dataclasses import replace
    Hkv = lay.num_heads_kv
    lay_full = replace(lay, num_heads_kv=lay.num_heads_q)
    k_full = k.repeat_interleave(lay.group, dim=2)
    v_full = v.repeat_interleave(lay.group, dim=2)
    a, _ = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                       lay.window, lay.causal, lay.scale)
    b, _ = O.attention(q, k_full, v_full, lay_full.block_table, lay.query_start_loc, lay.seq_lens,
                       lay.mm_ranges, lay.window, lay.causal, lay.scale)
    assert Hkv < lay.num_heads_q
    for r in a:
        assert np.allclose(a[r], b[r], atol=1e-13)


# ---------------------------------------------------------------------------
# LSE merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_split_then_merge_equals_unsplit(seed):
    lay, q, k, v = _small(seed, window=int([0, 5, 30, 0][seed]), causal=bool(seed % 2),
                          with_ranges=True, dtype="fp32")
    lay.seq_lens = lay.seq_lens  # unchanged
    P = 4
    sps = np.random.default_rng(seed).integers(1, P + 1, size=lay.num_seqs)
    po, pl = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                         lay.window, lay.causal, lay.scale, num_splits=P, splits_per_seq=sps)
    T, H, D = q.shape
    part_o = np.full((P, T, H, D), np.nan)           # -inf partitions stay NaN: must not be read
    part_l = np.full((P, T, H), -np.inf)
    for (p, t, h), val in po.items():
        if pl[(p, t, h)] != -np.inf:
            part_o[p, t, h] = val
        part_l[p, t, h] = pl[(p, t, h)]
    mo, ml = O.lse_combine(part_o, part_l)
    ref, rl = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                          lay.window, lay.causal, lay.scale)
    for (t, h), val in ref.items():
        assert np.allclose(mo[t, h], val, atol=1e-12)
        assert abs(ml[t, h] - rl[(t, h)]) < 1e-12


def test_merge_special_cases():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((3, 2, 2, 4))
    # one partition: identity
    mo, ml = O.lse_combine(o[:1], np.array([[[0.3, -1.0], [2.0, 5.0]]]))
    assert np.allclose(mo, o[0]) and np.allclose(ml, [[0.3, -1.0], [2.0, 5.0]])
    # equal LSE: plain average, lse + ln 3
    mo, ml = O.lse_combine(o, np.full((3, 2, 2), 1.5))
    assert np.allclose(mo, o.mean(0)) and np.allclose(ml, 1.5 + math.log(3))
    # a single live partition is copied; all -inf gives 0 and -inf
    lse = np.full((3, 2, 2), -np.inf)
    lse[1, 0, 0] = 0.7
    o2 = o.copy()
    o2[0] = np.nan
    o2[2] = np.nan
    mo, ml = O.lse_combine(o2, lse)
    assert np.allclose(mo[0, 0], o[1, 0, 0]) and ml[0, 0] == 0.7
    assert np.all(mo[1] == 0) and np.all(mo[0, 1] == 0) and ml[1, 1] == -np.inf
    # two partitions with lse a, b: weights e^a : e^b
    mo, ml = O.lse_combine(o[:2], np.stack([np.zeros((2, 2)), np.full((2, 2), math.log(3.0))]))
    assert np.allclose(mo, 0.25 * o[0] + 0.75 * o[1]) and np.allclose(ml, math.log(4.0))


def test_split_key_ranges_partition_the_sequence():
    for n in [1, 5, 127, 128, 129, 4097, 65537]:
        for P in [1, 2, 3, 8, 32]:
            r = O.split_key_ranges(n, P)
            assert len(r) == P and r[0][0] == 0 and r[-1][1] == n
            for (a, b), (c, d) in zip(r, r[1:]):
                assert b == c and a <= b
            assert all(a % 128 == 0 for a, b in r if a < b)


# ---------------------------------------------------------------------------
# slot mapping
# ---------------------------------------------------------------------------
def test_slot_mapping_pages_worked_example(golden_dir):
    g = _load(golden_dir, "slot_mapping_pages_example.json")
    slots, bad = O.slot_mapping(g["query_start_loc"], g["positions"], np.array(g["block_table"]),
                                g["block_size"], g["num_tokens"], g["max_num_tokens"], g["pad_id"])
    assert slots[:10].tolist() == g["expect_first"]
    assert np.all(slots[10:] == g["expect_tail_value"]) and len(slots) == g["max_num_tokens"]
    assert bad == []


@pytest.mark.parametrize("seed", range(5))
def test_slot_mapping_invariants(seed):
    lay = W.random_small(seed)
    pos = lay.positions
    pos_bad = pos.copy()
    if len(pos_bad) > 2:
        pos_bad[1] = -3
        pos_bad[2] = lay.block_table.shape[1] * lay.block_size + 5
    slots, bad = O.slot_mapping(lay.query_start_loc, pos_bad, lay.block_table, lay.block_size,
                                lay.num_tokens, lay.max_num_tokens)
    qsl = lay.query_start_loc
    B = lay.block_size
    for s in range(lay.num_seqs):
        for t in range(qsl[s], qsl[s + 1]):
            if t in bad:
                assert slots[t] == -1
                continue
            # the page holding the token is the table entry for its block; offset kept
            assert slots[t] // B == lay.block_table[s, pos_bad[t] // B]
            assert slots[t] % B == pos_bad[t] % B
    assert np.all(slots[lay.num_tokens:] == -1)
    if len(pos_bad) > 2:
        assert set(bad) == {1, 2}
    # distinct positions of one request map to distinct slots
    for s in range(lay.num_seqs):
        seg = [slots[t] for t in range(qsl[s], qsl[s + 1]) if t not in bad]
        assert len(seg) == len(set(seg))


# ---------------------------------------------------------------------------
# planted mistakes: each one must be caught by a pin above
# ---------------------------------------------------------------------------
def test_planted_left_edge_from_last_row_is_caught():
    """Using the block's last row for the window's left edge drops keys."""
    def wrong(qsl, seq, mm, window, causal, tile, bq, maxb):
        tb = O.tile_bounds(qsl, seq, mm, window, causal, tile, bq, maxb)
        for b in range(maxb):
            q_hi = min(b * bq + bq - 1, int(qsl[1]) - 1)
            tb[0, b, 0] = max(0, (q_hi - window + 1) // tile)
        return tb
    qsl, seq = np.array([0, 64]), np.array([64])
    tb = wrong(qsl, seq, None, 5, True, 4, 8, 8)
    keys = set()
    for i in range(8, 16):
        keys |= set(np.nonzero(O.visible_keys(i, 64, 5, True, None))[0].tolist())
    assert not {k // 4 for k in keys} <= set(range(tb[0, 1, 0], tb[0, 1, 1]))


def test_planted_unclamped_image_mask_is_caught():
    """An image mask without the window clamp breaks the closed-form interval."""
    q, seq_len, window = 30, 40, 4
    rngs = [(10, 35)]
    k = np.arange(seq_len)
    wrong = ((k >= q - window + 1) & (k <= q)) | ((k >= 10) & (k <= 35))
    lo, hi = _interval(q, seq_len, window, True, rngs)
    right = np.zeros(seq_len, bool)
    right[lo:hi + 1] = True
    assert not np.array_equal(wrong, right)
    assert np.array_equal(O.visible_keys(q, seq_len, window, True, np.array(rngs)), right)


def test_planted_max_prefix_seq_len_when_causal_is_caught():
    """Reporting seq_len as the prefix of a causal block without images
    overstates the keys the block can see; the brute-force pin catches it."""
    qsl, seq = np.array([0, 40]), np.array([60])
    tb = O.tile_bounds(qsl, seq, None, 8, True, 4, 8, 5)
    wrong = tb.copy()
    wrong[0, :, 2] = 60
    rows = range(0, 8)
    bound = _max_visible_key_plus_one(20, 60, rows, 8, True, None)
    assert tb[0, 0, 2] == bound
    assert wrong[0, 0, 2] != bound
