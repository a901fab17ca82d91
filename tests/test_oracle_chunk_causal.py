"""Pins for the oracle's chunked lookback and per-sequence causal modes.

Sources: "vLLM PR #53147 summary" -- the compute_tile_loop_bounds excerpt
(the chunk branch: the base window's left edge becomes the start of the chunk
CHUNK_LOOKBACK chunks before the query's chunk; the right edge under
USE_PER_SEQ_CAUSAL is the non-causal one), the reviewer's notes in the same
summary (the image mask is OR-ed after the chunk restriction and keeps the
ordinary window clamp, so it can re-enable keys before the chunk boundary; the
tile lower bound is the minimum of the chunk edge and every intersecting
range's clamped start), and the geometry test with the non-causal right
window ([3, 68)).

Each test checks the oracle against something it does not compute itself:
the chunk rule restated through chunk indices, masks built from torch's
block-diagonal and triangular constructors fed to fp64 scaled-dot-product
attention, hand-derived cases, closed-form pair counts, brute-force tile
covers and the printed bounds.  The last tests plant mistakes in copies of
oracle functions and check that a pin catches each.
"""
import json
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
# the chunked mask
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(30))
def test_chunk_mask_by_chunk_index(seed):
    """Without images: key k is visible iff its chunk is at most L chunks
    before the query's chunk and k is inside the right edge."""
    rng = np.random.default_rng(seed)
    seq_len = int(rng.integers(1, 150))
    C = int(rng.choice([1, 2, 3, 8, 16, 40]))
    L = int(rng.choice([0, 1, 2, 5]))
    window = int(rng.choice([1, 4, 16, 100, 1000]))
    causal = bool(rng.integers(0, 2))
    for q in range(seq_len):
        got = O.visible_keys(q, seq_len, window, causal, None, C, L)
        right = q if causal else q + window - 1
        exp = [k for k in range(seq_len) if q // C - k // C <= L and k <= right]
        assert np.nonzero(got)[0].tolist() == exp, (q, C, L, window, causal)


def _chunk_lay(seed, causal, seq_causal=None):
    lay = W.random_small(seed, max_seqs=3, max_ctx=30, max_q=50, head_dim=16, window=64, causal=causal,
                         with_ranges=False, dtype="fp32")
    q, k, v = W.make_tensors(lay, data_seed=seed)
    return lay, q, k, v


def _dense_kv(lay, k, v, s):
    n = int(lay.seq_lens[s])
    pages = torch.from_numpy(lay.block_table[s, :(n + lay.block_size - 1) // lay.block_size].astype(np.int64))
    kk = k[pages].reshape(-1, lay.num_heads_kv, lay.head_dim)[:n].double()
    vv = v[pages].reshape(-1, lay.num_heads_kv, lay.head_dim)[:n].double()
    return kk.repeat_interleave(lay.group, dim=1), vv.repeat_interleave(lay.group, dim=1)


def _sdpa_rows(lay, q, k, v, s, mask):
    """fp64 SDPA of sequence s's query rows against its whole key sequence."""
    qsl = lay.query_start_loc
    kk, vv = _dense_kv(lay, k, v, s)
    qs = q[int(qsl[s]):int(qsl[s + 1])].double()
    o = torch.nn.functional.scaled_dot_product_attention(
        qs.transpose(0, 1), kk.transpose(0, 1), vv.transpose(0, 1), attn_mask=mask, scale=lay.scale)
    return o.transpose(0, 1)


def _oracle_seq(lay, q, k, v, s, **kw):
    out, _ = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, None, lay.window,
                         lay.causal, lay.scale, **kw)
    qsl = lay.query_start_loc
    rows = range(int(qsl[s]), int(qsl[s + 1]))
    return torch.stack([torch.stack([torch.from_numpy(out[(t, h)]) for h in range(lay.num_heads_q)])
                        for t in rows]) if len(rows) else torch.zeros((0, lay.num_heads_q, lay.head_dim))


@pytest.mark.parametrize("seed,C", [(0, 4), (1, 7), (2, 16), (3, 1)])
def test_chunk_lookback_zero_is_block_diagonal_causal_sdpa(seed, C):
    """L = 0, causal, window wider than a chunk: every query attends causally
    inside its own chunk -- a block-diagonal lower-triangular mask."""
    lay, q, k, v = _chunk_lay(seed, True)
    for s in range(lay.num_seqs):
        n, c = int(lay.seq_lens[s]), int(lay.context_lens[s])
        if n == c:
            continue
        sizes = [min(C, n - i) for i in range(0, n, C)]
        full = torch.block_diag(*[torch.ones(m, m).tril() for m in sizes]).bool()
        ref = _sdpa_rows(lay, q, k, v, s, full[c:])
        got = _oracle_seq(lay, q, k, v, s, chunk_size=C, chunk_lookback=0)
        assert torch.allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("seed", range(3))
def test_chunk_lookback_covering_the_sequence_is_full_causal_sdpa(seed):
    lay, q, k, v = _chunk_lay(10 + seed, True)
    for s in range(lay.num_seqs):
        n, c = int(lay.seq_lens[s]), int(lay.context_lens[s])
        if n == c:
            continue
        ref = _sdpa_rows(lay, q, k, v, s, torch.ones(n - c, n, dtype=torch.bool).tril(c))
        got = _oracle_seq(lay, q, k, v, s, chunk_size=8, chunk_lookback=n // 8 + 1)
        assert torch.allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("window,ranges,causal,expect", [
    # q = 10, chunk 4, lookback 0: the chunk starts at 8
    (8, None, True, [8, 9, 10]),
    (8, None, False, [8, 9, 10, 11, 12, 13, 14, 15]),       # right window 10 + 7 = 17, seq end 15
    # image [5, 12] holds q: clamped start max(5, 10 - 8 + 1) = 5, before the chunk start
    (8, [[5, 12]], True, [5, 6, 7, 8, 9, 10, 11, 12]),
    # a narrow window clamps the image to max(5, 10 - 3 + 1) = 8: nothing before the chunk
    (3, [[5, 12]], True, [8, 9, 10, 11, 12]),
    # an image that does not hold q changes nothing
    (8, [[0, 6], [12, 15]], True, [8, 9, 10]),
])
def test_chunk_hand_cases_image_reaches_before_the_chunk(window, ranges, causal, expect):
    rng = None if ranges is None else np.array(ranges)
    got = O.visible_keys(10, 16, window, causal, rng, 4, 0)
    assert np.nonzero(got)[0].tolist() == expect


def test_chunk_pair_count_closed_form():
    """One sequence of n tokens, causal, L = 0: sum over chunks of m(m+1)/2;
    L = 1: each query also sees the whole previous chunk."""
    n, C = 103, 10
    qsl, seq = [0, n], [n]
    sizes = [min(C, n - i) for i in range(0, n, C)]
    assert O.allowed_pair_count(qsl, seq, None, 10 ** 6, True, chunk_size=C, chunk_lookback=0) == \
        sum(m * (m + 1) // 2 for m in sizes)
    assert O.allowed_pair_count(qsl, seq, None, 10 ** 6, True, chunk_size=C, chunk_lookback=1) == \
        sum(m * (m + 1) // 2 for m in sizes) + sum(C * m for m in sizes[1:])


def test_chunk_needs_a_window_and_a_chunk_size():
    with pytest.raises(ValueError):
        O.visible_keys(3, 10, 0, True, None, 4, 0)
    with pytest.raises(ValueError):
        O.visible_keys(3, 10, 5, True, None, 0, 1)
    # lookback -1 is off whatever the chunk size
    assert np.array_equal(O.visible_keys(7, 10, 3, True, None, 0, -1), O.visible_keys(7, 10, 3, True, None))


# ---------------------------------------------------------------------------
# per-sequence causal
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(3))
def test_per_seq_causal_each_sequence_is_its_own_sdpa(seed):
    """W <= 0 with flags: causal sequences get the lower-triangular mask,
    the others attend to every key."""
    lay, q, k, v = _chunk_lay(20 + seed, True)
    lay.window = 0
    flags = np.array([(s + seed) % 2 for s in range(lay.num_seqs)], dtype=np.int32)
    for s in range(lay.num_seqs):
        n, c = int(lay.seq_lens[s]), int(lay.context_lens[s])
        if n == c:
            continue
        mask = torch.ones(n - c, n, dtype=torch.bool)
        if flags[s]:
            mask = mask.tril(c)
        ref = _sdpa_rows(lay, q, k, v, s, mask)
        got = _oracle_seq(lay, q, k, v, s, seq_causal=flags)
        assert torch.allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("seed", range(4))
def test_per_seq_causal_all_equal_flags_reduce_to_the_scalar(seed):
    lay = W.random_small(40 + seed, max_seqs=3, max_ctx=40, max_q=30, head_dim=16, dtype="fp32")
    q, k, v = W.make_tensors(lay, data_seed=seed)
    for c in (True, False):
        flags = np.full(lay.num_seqs, int(c), dtype=np.int32)
        a, la = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                            lay.window, not c, lay.scale, seq_causal=flags)
        b, lb = O.attention(q, k, v, lay.block_table, lay.query_start_loc, lay.seq_lens, lay.mm_ranges,
                            lay.window, c, lay.scale)
        assert all(np.array_equal(a[r], b[r]) and la[r] == lb[r] for r in b)


# ---------------------------------------------------------------------------
# tile bounds
# ---------------------------------------------------------------------------
def test_per_seq_causal_bounds_are_the_printed_noncausal_ones(golden_dir):
    """The excerpt bounds the per-sequence causal mode with the non-causal
    right edge: with causal set and the mode on, the printed [3, 68)."""
    gd = _load(golden_dir, "tile_bounds_pages.json")
    g, c = gd["geometry"], gd["cases"][1]
    qsl, seq = np.array([0, g["query_len"]]), np.array([g["seq_len"]])
    tb = O.tile_bounds(qsl, seq, np.array([c["mm_ranges"]], np.int32), g["window"], True, g["tile_size"],
                       g["block_q"], g["q_block_local_idx"] + 1, per_seq_causal=True)
    assert tb[0, g["q_block_local_idx"], :2].tolist() == c["expect_lo_hi"]


def _random_bounds_case(rng):
    S = int(rng.integers(1, 4))
    qlen = rng.integers(0, 90, size=S)
    ctx = rng.integers(0, 90, size=S)
    seq = ctx + qlen
    window = int(rng.choice([1, 3, 9, 33, 500]))
    tile = int(rng.choice([1, 4, 8, 16, 32]))
    bq = int(rng.choice([1, 2, 3, 8, 16]))
    R = int(rng.integers(1, 4))
    mm = np.zeros((S, R, 2), dtype=np.int32)
    for s in range(S):
        for i in range(R):
            if seq[s] > 1 and rng.integers(0, 3):
                a = int(rng.integers(0, seq[s] - 1))
                mm[s, i] = (a, int(rng.integers(a, seq[s])))
    C = int(rng.choice([1, 5, 16, 64]))
    L = int(rng.choice([0, 1, 3]))
    return S, qlen, ctx, seq, window, tile, bq, mm, C, L


@pytest.mark.parametrize("seed", range(60))
def test_chunk_tile_bounds_cover_every_visible_key(seed):
    rng = np.random.default_rng(900 + seed)
    S, qlen, ctx, seq, window, tile, bq, mm, C, L = _random_bounds_case(rng)
    causal = bool(rng.integers(0, 2))
    per_seq = bool(rng.integers(0, 2))
    flags = rng.integers(0, 2, size=S)
    qsl = np.concatenate([[0], np.cumsum(qlen)])
    maxb = int(max(1, -(-qlen.max() // bq)))
    tb = O.tile_bounds(qsl, seq, mm, window, causal, tile, bq, maxb, per_seq_causal=per_seq,
                       chunk_size=C, chunk_lookback=L)
    for s in range(S):
        c_s = bool(flags[s]) if per_seq else causal
        for b in range(maxb):
            rows = range(b * bq, min((b + 1) * bq, int(qlen[s])))
            if not rows:
                assert tb[s, b].tolist() == [0, 0, 0]
                continue
            keys = set()
            for i in rows:
                keys |= set(np.nonzero(O.visible_keys(ctx[s] + i, seq[s], window, c_s, mm[s], C, L))[0].tolist())
            lo, hi, _ = tb[s, b]
            tiles = {k // tile for k in keys}
            assert tiles <= set(range(lo, hi)), (s, b, lo, hi, sorted(tiles))
            # the left edge is exact: the chunk start of the first row or a range's clamped start
            assert lo == min(tiles)
            if not per_seq:
                assert hi == max(tiles) + 1


# ---------------------------------------------------------------------------
# planted mistakes: each one must be caught by a pin above
# ---------------------------------------------------------------------------
def test_planted_chunk_edge_from_last_row_is_caught():
    """Taking the chunk start of the block's last row (the excerpt's q_abs)
    drops the earlier rows' chunk when the block straddles a chunk boundary:
    context 4, block 0 holds positions 4..11, chunks of 8."""
    qsl, seq = np.array([0, 60]), np.array([64])
    C, L, tile, bq, window = 8, 0, 4, 8, 100
    tb = O.tile_bounds(qsl, seq, None, window, True, tile, bq, 8, chunk_size=C, chunk_lookback=L)
    keys = set()
    for pos in range(4, 12):
        keys |= set(np.nonzero(O.visible_keys(pos, 64, window, True, None, C, L))[0].tolist())
    tiles = {k // tile for k in keys}
    wrong_lo = ((11 // C) - L) * C // tile           # the last row's chunk start: tile 2
    assert not tiles <= set(range(wrong_lo, tb[0, 0, 1]))
    assert tiles <= set(range(tb[0, 0, 0], tb[0, 0, 1])) and tb[0, 0, 0] == 0


def test_planted_image_clamped_by_the_chunk_is_caught():
    """Clamping the image mask at the chunk edge instead of the window edge
    loses keys 5..7 of the hand case above."""
    k = np.arange(16)
    q, C, L, window = 10, 4, 0, 8
    chunk_lo = (q // C - L) * C
    wrong = ((k >= chunk_lo) & (k <= q)) | ((k >= 5) & (k <= 12) & (k >= chunk_lo))
    right = O.visible_keys(q, 16, window, True, np.array([[5, 12]]), C, L)
    assert not np.array_equal(wrong, right)
    assert np.nonzero(right)[0].tolist() == [5, 6, 7, 8, 9, 10, 11, 12]


def test_planted_ignored_flags_are_caught():
    """A mask that ignores the per-sequence flags fails the SDPA pin."""
    lay, q, k, v = _chunk_lay(20, True)
    lay.window = 0
    flags = np.array([s % 2 for s in range(lay.num_seqs)], dtype=np.int32)
    caught = False
    for s in range(lay.num_seqs):
        n, c = int(lay.seq_lens[s]), int(lay.context_lens[s])
        if n - c < 2 or flags[s]:
            continue
        ref = _sdpa_rows(lay, q, k, v, s, torch.ones(n - c, n, dtype=torch.bool))
        wrong = _oracle_seq(lay, q, k, v, s)             # the scalar causal flag only
        caught |= not torch.allclose(wrong, ref, atol=1e-12, rtol=0)
    assert caught
