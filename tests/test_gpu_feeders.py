"""GPU parity of the two feeders and the bounds kernel: slot mapping and tile
bounds bit-exact against the oracle, the LSE merge within tolerance."""
import json
import math
import os

import numpy as np
import pytest
import torch

import paged_sliding_window_swa_gb300 as swa
import workloads as W
from oracle import swa_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture
def err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device="cuda")


def _i64(a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int64, device="cuda")


# ---------------------------------------------------------------------------
# slot mapping
# ---------------------------------------------------------------------------
def test_slot_mapping_pages_example(golden_dir, err):
    g = json.load(open(os.path.join(golden_dir, "slot_mapping_pages_example.json")))
    out = swa.swa_slot_mapping(_i32(g["query_start_loc"]), _i64(g["positions"]), _i32(g["block_table"]),
                               g["block_size"], g["max_num_tokens"], err=err)
    out = out.cpu().numpy()
    assert out[:10].tolist() == g["expect_first"]
    assert np.all(out[10:] == -1)
    assert err.item() == 0


@pytest.mark.parametrize("name", ["tiny", "geometry", "gemma_like", "chunked_prefill", "decode"])
def test_slot_mapping_named_layouts(name, err):
    lay = W.NAMED[name]()
    d = W.device_layout(lay, "cuda")
    out = swa.swa_slot_mapping(d["query_start_loc"], d["positions"], d["block_table"], lay.block_size,
                               lay.max_num_tokens, err=err)
    ref, bad = O.slot_mapping(lay.query_start_loc, lay.positions, lay.block_table, lay.block_size,
                              lay.num_tokens, lay.max_num_tokens)
    assert np.array_equal(out.cpu().numpy(), ref) and bad == [] and err.item() == 0


@pytest.mark.parametrize("name", ["tiny", "gemma_like", "chunked_prefill", "decode"])
def test_slot_mapping_derived_positions_named_layouts(name, err):
    """positions = NULL: context length + index, the same slots as the layout's
    explicit positions (which are exactly that)."""
    lay = W.NAMED[name]()
    d = W.device_layout(lay, "cuda")
    out = swa.swa_slot_mapping(d["query_start_loc"], None, d["block_table"], lay.block_size, lay.max_num_tokens,
                               context_lens=d["context_lens"], num_tokens=lay.num_tokens, err=err)
    ref, bad = O.slot_mapping(lay.query_start_loc, None, lay.block_table, lay.block_size, lay.num_tokens,
                              lay.max_num_tokens, context_lens=lay.context_lens)
    assert np.array_equal(out.cpu().numpy(), ref) and bad == [] and err.item() == 0


@pytest.mark.parametrize("seed", range(8))
def test_slot_mapping_derived_positions_random(seed, err):
    """Random context lengths, some past the block-table row (reported, pad_id)."""
    rng = np.random.default_rng(40 + seed)
    S, B = int(rng.integers(1, 7)), int(rng.choice([16, 32, 64]))
    qlen = rng.integers(0, 500, size=S)
    ctx = rng.integers(0, 3000, size=S)
    qsl = np.concatenate([[0], np.cumsum(qlen)])
    stride = int(-(-(ctx + qlen).max() // B)) - (1 if seed % 3 == 0 else 0)   # sometimes one page short
    stride = max(stride, 1)
    bt = rng.permutation(S * stride + 5)[:S * stride].reshape(S, stride)
    T = int(qsl[-1])
    maxn = T + int(rng.integers(0, 33))
    out = swa.swa_slot_mapping(_i32(qsl), None, _i32(bt), B, maxn, context_lens=_i32(ctx), num_tokens=T, err=err)
    ref, bad = O.slot_mapping(qsl, None, bt, B, T, maxn, context_lens=ctx)
    assert np.array_equal(out.cpu().numpy(), ref)
    torch.cuda.synchronize()
    assert bool(err.item() & 0x02) == bool(bad)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("misaligned", [False, True])
def test_slot_mapping_random(seed, misaligned, err):
    lay = W.random_small(seed, max_seqs=8, max_q=700)
    pos = lay.positions
    if misaligned:    # positions at an 8-byte offset, odd tail length: scalar path
        buf = _i64(np.concatenate([[0], pos]))
        pos_t = buf[1:]
        maxn = lay.num_tokens + 3
    else:
        pos_t = _i64(pos)
        maxn = lay.max_num_tokens
    out = swa.swa_slot_mapping(_i32(lay.query_start_loc), pos_t, _i32(lay.block_table), lay.block_size,
                               maxn, pad_id=-7, err=err)
    ref, _ = O.slot_mapping(lay.query_start_loc, pos, lay.block_table, lay.block_size,
                            lay.num_tokens, maxn, pad_id=-7)
    assert np.array_equal(out.cpu().numpy(), ref) and err.item() == 0


def test_slot_mapping_bad_positions_are_padded_and_reported(err):
    lay = W.random_small(2, max_seqs=3, max_q=200)
    pos = lay.positions.copy()
    pos[0] = -5
    pos[-1] = lay.block_table.shape[1] * lay.block_size + 3
    out = swa.swa_slot_mapping(_i32(lay.query_start_loc), _i64(pos), _i32(lay.block_table),
                               lay.block_size, lay.max_num_tokens, err=err)
    ref, bad = O.slot_mapping(lay.query_start_loc, pos, lay.block_table, lay.block_size,
                              lay.num_tokens, lay.max_num_tokens)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert set(bad) == {0, lay.num_tokens - 1}
    assert err.item() & 0x02


def test_slot_mapping_bad_query_start_loc_is_reported(err):
    qsl = _i32([0, 6, 3, 9])
    pos = _i64(np.arange(9))
    bt = _i32(np.arange(12).reshape(3, 4))
    swa.swa_slot_mapping(qsl, pos, bt, 16, 16, err=err)
    torch.cuda.synchronize()
    assert err.item() & 0x04


def test_slot_mapping_large(err):
    """Four million tokens over 64 requests: the bandwidth-sized case."""
    rng = np.random.default_rng(0)
    lens = rng.integers(1, 2 * 65536, size=64)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(qsl[-1])
    B = 16
    pages = -(-lens // B)
    bt = np.full((64, int(pages.max())), -1, dtype=np.int32)
    perm = rng.permutation(int(pages.sum())).astype(np.int32)
    c = 0
    for s in range(64):
        bt[s, :pages[s]] = perm[c:c + pages[s]]
        c += pages[s]
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int64)
    maxn = -(-T // 8192) * 8192
    out = swa.swa_slot_mapping(_i32(qsl), _i64(pos), _i32(bt), B, maxn, err=err).cpu().numpy()
    # vectorised check of the definition, then the oracle on a sample of requests
    req = np.repeat(np.arange(64), lens)
    expect = bt[req, pos // B].astype(np.int64) * B + pos % B
    assert np.array_equal(out[:T], expect) and np.all(out[T:] == -1)
    for s in (0, 17, 63):
        sub = slice(int(qsl[s]), int(qsl[s + 1]))
        ref, _ = O.slot_mapping([0, lens[s]], pos[sub], bt[s:s + 1], B, int(lens[s]), int(lens[s]))
        assert np.array_equal(out[sub], ref)
    assert err.item() == 0


# ---------------------------------------------------------------------------
# tile bounds
# ---------------------------------------------------------------------------
def test_tile_bounds_pages_geometry(golden_dir, err):
    gd = json.load(open(os.path.join(golden_dir, "tile_bounds_pages.json")))
    g = gd["geometry"]
    for c in gd["cases"]:
        out = swa.swa_tile_bounds(_i32([0, g["query_len"]]), _i32([g["seq_len"]]),
                                  mm_ranges=_i32([c["mm_ranges"]]), window=g["window"], causal=c["causal"],
                                  tile_size=g["tile_size"], block_q=g["block_q"],
                                  max_qblocks_per_seq=g["q_block_local_idx"] + 1, err=err)
        got = out[0, g["q_block_local_idx"]].tolist()
        if "expect" in c:
            assert got == c["expect"]
        else:
            assert got[:2] == c["expect_lo_hi"]
    assert err.item() == 0


@pytest.mark.parametrize("seed", range(30))
def test_tile_bounds_random(seed, err):
    lay = W.random_small(seed, max_seqs=6, max_ctx=3000, max_q=900)
    rng = np.random.default_rng(seed)
    tile = int(rng.choice([16, 32, 64, 128]))
    bq = int(rng.choice([1, 8, 16, 64]))
    maxb = -(-lay.max_query_len // bq) + int(rng.integers(0, 3))
    window = int(rng.choice([-1, 0, 1, 64, 1024]))
    mm = None if lay.mm_ranges is None else _i32(lay.mm_ranges)
    out = swa.swa_tile_bounds(_i32(lay.query_start_loc), _i32(lay.seq_lens),
                              context_lens=_i32(lay.context_lens) if seed % 2 else None, mm_ranges=mm,
                              window=window, causal=lay.causal, tile_size=tile, block_q=bq,
                              max_qblocks_per_seq=maxb, err=err)
    ref = O.tile_bounds(lay.query_start_loc, lay.seq_lens, lay.mm_ranges, window, lay.causal, tile, bq, maxb)
    assert np.array_equal(out.cpu().numpy(), ref) and err.item() == 0


@pytest.mark.parametrize("name", ["tiny", "geometry", "gemma_like", "chunked_prefill"])
def test_tile_bounds_named_layouts(name, err):
    lay = W.NAMED[name]()
    d = W.device_layout(lay, "cuda")
    for tile, bq in ((32, 8), (64, 32), (128, 64)):
        maxb = -(-lay.max_query_len // bq)
        out = swa.swa_tile_bounds(d["query_start_loc"], d["seq_lens"], context_lens=d["context_lens"],
                                  mm_ranges=d["mm_ranges"], window=lay.window, causal=lay.causal,
                                  tile_size=tile, block_q=bq, max_qblocks_per_seq=maxb, err=err)
        ref = O.tile_bounds(lay.query_start_loc, lay.seq_lens, lay.mm_ranges, lay.window, lay.causal,
                            tile, bq, maxb)
        assert np.array_equal(out.cpu().numpy(), ref)
    assert err.item() == 0


def test_tile_bounds_inconsistent_lengths_are_reported(err):
    out = swa.swa_tile_bounds(_i32([0, 10]), _i32([30]), context_lens=_i32([5]), window=8, causal=True,
                              tile_size=4, block_q=4, max_qblocks_per_seq=3, err=err)
    assert out.cpu().numpy().sum() == 0 and err.item() & 0x08


# ---------------------------------------------------------------------------
# LSE merge
# ---------------------------------------------------------------------------
def _partials(P, T, H, D, dtype, seed, dead_frac=0.3):
    g = torch.Generator(device="cuda").manual_seed(seed)
    po = torch.randn((P, T, H, D), generator=g, device="cuda").to(dtype)
    pl = (torch.randn((P, T, H), generator=g, device="cuda") * 4).float()
    dead = torch.rand((P, T, H), generator=g, device="cuda") < dead_frac
    pl[dead] = -math.inf
    pl[:, 0, 0] = -math.inf                            # one all-dead row
    po[dead] = float("nan")                            # must never be read
    return po, pl


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("P", [1, 3, 32])
def test_lse_combine_random(dtype, D, P):
    po, pl = _partials(P, 37, 5, D, dtype, seed=D + P)
    out, lse = swa.lse_combine(po, pl)
    ro, rl = O.lse_combine(po.cpu(), pl.cpu())
    o = out.float().cpu().numpy()
    tol = (2e-2 if dtype == torch.bfloat16 else 1e-5)
    assert np.all(np.isfinite(o))
    assert np.abs(o - ro).max() <= tol + (8e-3 if dtype == torch.bfloat16 else 1e-6) * np.abs(ro).max()
    l = lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(l[fin] - rl[fin]).max() <= 1e-5 * max(1.0, np.abs(rl[fin]).max())
    assert np.all(o[0, 0] == 0)


def test_lse_combine_large_sampled():
    """T = 65536 tokens x 32 heads x 8 partitions: sampled rows vs the oracle."""
    P, T, H, D = 8, 65536, 32, 128
    po, pl = _partials(P, T, H, D, torch.bfloat16, seed=7, dead_frac=0.2)
    out, lse = swa.lse_combine(po, pl)
    rng = np.random.default_rng(0)
    ts = np.unique(rng.integers(0, T, 300))
    ro, rl = O.lse_combine(po[:, ts].cpu(), pl[:, ts].cpu())
    o = out[ts].float().cpu().numpy()
    assert np.abs(o - ro).max() <= 2e-2
    l = lse[ts].cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin) and np.abs(l[fin] - rl[fin]).max() < 1e-4


def test_slot_mapping_derived_positions_misaligned_output(err):
    """An output buffer at a 4-byte offset takes the scalar store path."""
    lay = W.random_small(3, max_seqs=4, max_q=300)
    d = W.device_layout(lay, "cuda")
    buf = torch.full((lay.max_num_tokens + 1,), 7, dtype=torch.int32, device="cuda")
    out = buf[1:]
    swa.swa_slot_mapping(d["query_start_loc"], None, d["block_table"], lay.block_size, lay.max_num_tokens,
                         context_lens=d["context_lens"], num_tokens=lay.num_tokens, out=out, err=err)
    ref, _ = O.slot_mapping(lay.query_start_loc, None, lay.block_table, lay.block_size, lay.num_tokens,
                            lay.max_num_tokens, context_lens=lay.context_lens)
    assert np.array_equal(out.cpu().numpy(), ref) and buf[0].item() == 7 and err.item() == 0
