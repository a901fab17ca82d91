"""GPU parity of the chunked-lookback and per-sequence causal modes against
the oracle: tile bounds bit-exact, attention within the 2e-2 (bf16) / 2e-3
(fp32) max-abs bar on every row of small layouts and on sampled rows of the
chunked-prefill workload.  Each call goes through the C ABI; the layouts are
routed to the tensor-core, decode and CUDA-core kernels by their shapes."""
import json
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import workloads as W
from _gpu_helpers import (LSE_ATOL, atol_for, gpu_inputs, max_errors, oracle_rows, run_attention,
                          sample_rows)
from oracle import swa_oracle as O
import paged_sliding_window_swa_gb300 as swa

pytestmark = pytest.mark.gpu


@pytest.fixture
def err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _i32(a):
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device="cuda")


def _all_rows(lay):
    return [(t, h) for t in range(lay.num_tokens) for h in range(lay.num_heads_q)]


def _check(lay, rows, err, data_seed=1):
    q, k, v, d = gpu_inputs(lay, data_seed=data_seed)
    out, lse = run_attention(lay, q, k, v, d, err=err)
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay), f"{lay.name}: max-abs {e_out}"
    assert e_lse <= LSE_ATOL, f"{lay.name}: lse max-abs {e_lse}"
    torch.cuda.synchronize()
    assert err.item() == 0, hex(err.item())
    return out, (q, k, v, d)


def _with_modes(lay, rng, chunk=True, per_seq=True):
    kw = {}
    if chunk:
        kw["window"] = int(rng.choice([48, 200, 1000]))
        kw["chunk_size"] = int(rng.choice([16, 64, 100, 256]))
        kw["chunk_lookback"] = int(rng.choice([0, 1, 3]))
    if per_seq:
        kw["seq_causal"] = rng.integers(0, 2, size=lay.num_seqs).astype(np.int32)
    return replace(lay, name=lay.name + "-modes", **kw)


# ---------------------------------------------------------------------------
# tile bounds
# ---------------------------------------------------------------------------
def test_tile_bounds_per_seq_causal_printed_geometry(golden_dir, err):
    gd = json.load(open(os.path.join(golden_dir, "tile_bounds_pages.json")))
    g, c = gd["geometry"], gd["cases"][1]
    out = swa.swa_tile_bounds(_i32([0, g["query_len"]]), _i32([g["seq_len"]]), mm_ranges=_i32([c["mm_ranges"]]),
                              window=g["window"], causal=True, per_seq_causal=True, tile_size=g["tile_size"],
                              block_q=g["block_q"], max_qblocks_per_seq=g["q_block_local_idx"] + 1, err=err)
    assert out[0, g["q_block_local_idx"], :2].tolist() == c["expect_lo_hi"] and err.item() == 0


@pytest.mark.parametrize("seed", range(30))
def test_tile_bounds_chunk_and_per_seq_random(seed, err):
    lay = W.random_small(500 + seed, max_seqs=6, max_ctx=3000, max_q=900)
    rng = np.random.default_rng(seed)
    tile = int(rng.choice([16, 32, 64, 128]))
    bq = int(rng.choice([1, 8, 16, 64]))
    maxb = -(-lay.max_query_len // bq) + int(rng.integers(0, 3))
    window = int(rng.choice([1, 64, 1024, 1 << 30]))
    C = int(rng.choice([1, 16, 100, 512, 2048]))
    L = int(rng.choice([-1, 0, 1, 3, 1 << 20]))
    per_seq = bool(rng.integers(0, 2))
    mm = None if lay.mm_ranges is None else _i32(lay.mm_ranges)
    out = swa.swa_tile_bounds(_i32(lay.query_start_loc), _i32(lay.seq_lens), mm_ranges=mm, window=window,
                              causal=lay.causal, per_seq_causal=per_seq, chunk_size=C, chunk_lookback=L,
                              tile_size=tile, block_q=bq, max_qblocks_per_seq=maxb, err=err)
    ref = O.tile_bounds(lay.query_start_loc, lay.seq_lens, lay.mm_ranges, window, lay.causal, tile, bq, maxb,
                        per_seq_causal=per_seq, chunk_size=C, chunk_lookback=L)
    assert np.array_equal(out.cpu().numpy(), ref) and err.item() == 0


# ---------------------------------------------------------------------------
# attention, every row of small layouts
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(16))
def test_chunked_all_rows(seed, err):
    rng = np.random.default_rng(40 + seed)
    dtype = "fp32" if seed % 4 == 3 else "bf16"
    lay = W.random_small(600 + seed, dtype=dtype, max_seqs=3, max_ctx=500, max_q=260, with_ranges=seed % 2 == 0)
    _check(_with_modes(lay, rng, chunk=True, per_seq=False), _all_rows(lay), err)


@pytest.mark.parametrize("seed", range(12))
def test_per_seq_causal_all_rows(seed, err):
    rng = np.random.default_rng(80 + seed)
    dtype = "fp32" if seed % 4 == 3 else "bf16"
    lay = W.random_small(700 + seed, dtype=dtype, max_seqs=4, max_ctx=400, max_q=260,
                         window=int(rng.choice([-1, 0, 7, 64, 300])))
    _check(_with_modes(lay, rng, chunk=False, per_seq=True), _all_rows(lay), err)


@pytest.mark.parametrize("D,G", [(128, 2), (256, 2), (128, 8), (256, 1), (64, 4)])
def test_both_modes_shapes_all_rows(D, G, err):
    rng = np.random.default_rng(D + G)
    lay = W.random_small(800 + D + G, head_dim=D, group=G, max_seqs=3, max_ctx=700, max_q=300,
                         with_ranges=True)
    _check(_with_modes(lay, rng), _all_rows(lay), err)


@pytest.mark.parametrize("seed", range(4))
def test_both_modes_split_partials_and_merge(seed, err):
    P = [2, 5, 8, 3][seed]
    rng = np.random.default_rng(900 + seed)
    lay = W.random_small(900 + seed, max_seqs=3, max_ctx=2000, max_q=40, num_splits=P, with_ranges=True,
                         dtype="fp32" if seed == 3 else "bf16")
    lay = _with_modes(lay, rng)
    q, k, v, d = gpu_inputs(lay)
    po, pl = run_attention(lay, q, k, v, d, err=err)
    rows = _all_rows(lay)
    ro, rl = oracle_rows(lay, q, k, v, rows, num_splits=P)
    pof, plc = po.float().cpu().numpy(), pl.cpu().numpy()
    for (p, t, h), val in ro.items():
        if rl[(p, t, h)] == -np.inf:
            assert plc[p, t, h] == -np.inf
        else:
            assert abs(plc[p, t, h] - rl[(p, t, h)]) <= LSE_ATOL
            assert np.abs(pof[p, t, h] - val).max() <= atol_for(lay)
    mo, ml = swa.lse_combine(po, pl)
    uo, ul = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(mo, ml, uo, ul, rows)
    assert e_out <= atol_for(lay) and e_lse <= LSE_ATOL
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("D,G,max_q", [(128, 4, 1), (256, 2, 3), (64, 8, 2)])
def test_both_modes_decode_kernel(D, G, max_q, err):
    rng = np.random.default_rng(D * G + max_q)
    lay = W.random_small(950 + D + G, head_dim=D, group=G, max_seqs=4, max_ctx=3000, max_q=max_q,
                         with_ranges=True)
    _check(_with_modes(lay, rng), _all_rows(lay), err)


# ---------------------------------------------------------------------------
# the image term reaching before the chunk, at size
# ---------------------------------------------------------------------------
def _straddling_layout(causal=True):
    """4 sequences of 4096 query tokens after 0-1000 cached ones, W = 1024,
    chunks of 512, lookback 0, bf16 / D 256 / G 2 (the tensor-core kernel);
    every image straddles a chunk boundary, so the window-clamped image mask
    re-enables keys before the chunk of its later rows."""
    rng = np.random.default_rng(11)
    S, B = 4, 16
    qlen = np.full(S, 4096, np.int32)
    ctx = rng.integers(0, 1001, size=S).astype(np.int32)
    seq = ctx + qlen
    per = []
    for s in range(S):
        lst = []
        for c in range(1, int(seq[s]) // 512):
            if rng.integers(0, 2):
                a = c * 512 - int(rng.integers(1, 300))
                lst.append((a, a + int(rng.integers(300, 700))))
        per.append(lst)
    R = max(1, max(len(p) for p in per))
    mm = np.zeros((S, R, 2), np.int32)
    for s, lst in enumerate(per):
        for i, (a, b) in enumerate(lst):
            mm[s, i] = (a, min(b, int(seq[s]) - 1))
    pages = -(-seq // B)
    bt = np.full((S, int(pages.max()) + 2), -1, np.int32)
    perm = rng.permutation(int(pages.sum()) + 8)
    o = 0
    for s in range(S):
        bt[s, :pages[s]] = perm[o:o + pages[s]]
        o += int(pages[s])
    return W.Layout("straddling-chunks", query_lens=qlen, seq_lens=seq.astype(np.int32), mm_ranges=mm,
                    block_table=bt, num_blocks=int(perm.max()) + 1, num_heads_q=4, num_heads_kv=2,
                    head_dim=256, block_size=B, window=1024, causal=causal, chunk_size=512, chunk_lookback=0)


@pytest.mark.parametrize("causal", [True, False])
def test_image_reaches_before_the_chunk_at_size(causal, err):
    lay = _straddling_layout(causal)
    qsl = lay.query_start_loc
    edges = []
    for s in range(lay.num_seqs):
        c = int(lay.context_lens[s])
        for a, b in lay.mm_ranges[s]:
            if a < b:
                for p in (a, (a // 512 + 1) * 512, b):     # image start, the chunk boundary inside, image end
                    if c <= p < lay.seq_lens[s]:
                        edges.append(qsl[s] + p - c)
    rows = sample_rows(lay, 300, extra_tokens=edges)
    out, (q, k, v, d) = _check(lay, rows, err)
    without, _ = run_attention(lay, q, k, v, d, err=err, mm=False)
    idx = torch.as_tensor(sorted({t for t in edges}), device="cuda")
    change = (out.float() - without.float())[idx].abs().max().item()
    assert change >= 1e-2, change


def test_chunked_prefill_workload_modes_sampled(err):
    """The chunked-prefill workload (8 requests, 4k-32k cached tokens, 2048-token
    chunks, W = 1024) with chunks of 2048 looked back one chunk and mixed
    per-sequence causal flags."""
    lay = W.chunked_prefill(True)
    lay = replace(lay, chunk_size=2048, chunk_lookback=1,
                  seq_causal=np.array([s % 2 for s in range(lay.num_seqs)], np.int32))
    qsl = lay.query_start_loc
    edges = []
    for s in range(lay.num_seqs):
        edges += [qsl[s], qsl[s] + 127, qsl[s] + 128, qsl[s + 1] - 1]
    _check(lay, sample_rows(lay, 300, extra_tokens=edges), err)


@pytest.mark.parametrize("seed", range(40))
def test_random_layouts_with_chunks_and_per_sequence_causal(seed, err):
    """Random layouts (dtype, head_dim, GQA group, split count, window, images, page
    size, lengths) with chunked lookback (chunks of 32-2048, 0-3 back) and random
    per-sequence causal flags, up to 2000 rows each against the oracle."""
    rng = np.random.default_rng(30000 + seed)
    D = int(rng.choice([64, 128, 256]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    dtype = "fp32" if rng.random() < 0.15 else "bf16"
    P = int(rng.choice([1, 1, 1, 2, 5]))
    window = int(rng.choice([1, 7, 64, 200, 1000]))      # chunked lookback needs a window
    lay = W.random_small(30000 + seed, head_dim=D, group=G, dtype=dtype, max_seqs=int(rng.integers(1, 4)),
                         max_ctx=int(rng.choice([50, 900, 3000])), max_q=int(rng.choice([1, 40, 300, 700])),
                         window=window, num_splits=P)
    lay = replace(lay, chunk_size=int(rng.choice([32, 128, 512, 2048])), chunk_lookback=int(rng.choice([0, 1, 3])),
                  seq_causal=rng.integers(0, 2, size=lay.num_seqs).astype(np.int32))
    q, k, v, d = gpu_inputs(lay, data_seed=seed)
    rows = _all_rows(lay)
    if len(rows) > 2000:
        rows = [rows[i] for i in sorted(rng.choice(len(rows), 2000, replace=False))]
    if P == 1:
        out, lse = run_attention(lay, q, k, v, d, err=err)
    else:
        po, pl = run_attention(lay, q, k, v, d, err=err)
        out, lse = swa.lse_combine(po, pl)
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay) and e_lse <= LSE_ATOL, (e_out, e_lse)
    torch.cuda.synchronize()
    assert err.item() == 0
