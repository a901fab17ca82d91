"""GPU parity of swa_mm_paged_attention against the fp64 oracle.

Small layouts are compared on every (token, head) row; the full-size
workloads on sampled rows (every sequence's first and last token, image
boundaries, and random rows), each sequence cut out with its own pages so the
oracle stays fast.  The bar is max-abs 2e-2 for bf16 inputs (fp32
accumulation) and 2e-3 for fp32 inputs; LSE within 5e-3.
"""
import numpy as np
import pytest
import torch

import paged_sliding_window_swa_gb300 as swa
import workloads as W
from _gpu_helpers import (LSE_ATOL, atol_for, gpu_inputs, max_errors, oracle_rows, run_attention,
                          sample_rows)
from oracle import swa_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture
def err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _all_rows(lay):
    return [(t, h) for t in range(lay.num_tokens) for h in range(lay.num_heads_q)]


def _check(lay, rows, poison=False, err=None, data_seed=1):
    q, k, v, d = gpu_inputs(lay, data_seed=data_seed, poison=poison)
    out, lse = run_attention(lay, q, k, v, d, err=err)
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay), f"{lay.name}: max-abs {e_out}"
    assert e_lse <= LSE_ATOL, f"{lay.name}: lse max-abs {e_lse}"
    if err is not None:
        torch.cuda.synchronize()
        assert err.item() == 0, hex(err.item())
    return out, lse, (q, k, v, d)


def test_tiny_all_rows(err):
    lay = W.tiny()
    _check(lay, _all_rows(lay), err=err)


@pytest.mark.parametrize("variant", ["causal", "noncausal", "noncausal-wide"])
def test_geometry_rows(variant, err):
    lay = W.geometry(variant)
    rows = [(t, h) for t in range(0, lay.num_tokens, 3) for h in range(lay.num_heads_q)]
    rows += [(t, h) for t in range(1100, 1300) for h in (0, 5)]
    _check(lay, sorted(set(rows)), err=err)


def test_gemma_like_sampled(err):
    lay = W.gemma_like()
    edges = []
    qsl = lay.query_start_loc
    for s in range(lay.num_seqs):
        for (a, b) in lay.mm_ranges[s][:6]:
            edges += [qsl[s] + a - 1, qsl[s] + a, qsl[s] + b, qsl[s] + b + 1]
    rows = sample_rows(lay, 600, extra_tokens=edges)
    _check(lay, rows, err=err)


@pytest.mark.parametrize("causal", [True, False])
def test_chunked_prefill_sampled(causal, err):
    lay = W.chunked_prefill(causal)
    qsl, ctx = lay.query_start_loc, lay.context_lens
    edges = []
    for s in range(lay.num_seqs):
        edges += [qsl[s], qsl[s] + 1, qsl[s] + 127, qsl[s] + 128]      # the straddling image
    _check(lay, sample_rows(lay, 500, extra_tokens=edges), err=err)


@pytest.mark.parametrize("seed", range(24))
def test_random_small_all_rows(seed, err):
    dtype = "fp32" if seed % 4 == 3 else "bf16"
    lay = W.random_small(seed, dtype=dtype, max_seqs=3, max_ctx=500, max_q=260)
    _check(lay, _all_rows(lay), err=err)


@pytest.mark.parametrize("D,B,G", [(128, 16, 2), (256, 16, 2), (128, 16, 4), (256, 32, 1),
                                   (128, 64, 8), (64, 128, 4), (128, 128, 16), (64, 16, 2), (64, 32, 16),
                                   (64, 64, 1)])
def test_shapes_all_rows(D, B, G, err):
    lay = W.random_small(100 + D + B + G, head_dim=D, block_size=B, group=G, max_seqs=3, max_ctx=700,
                         max_q=300, window=int(np.random.default_rng(D + B).choice([48, 300])),
                         with_ranges=True)
    _check(lay, _all_rows(lay), err=err)


@pytest.mark.parametrize("D,G,window,causal", [(256, 2, 48, True), (256, 1, 300, False), (128, 2, 300, True),
                                              (128, 4, 48, False), (64, 4, 300, True), (64, 8, 48, False)])
def test_many_image_ranges_per_tile_all_rows(D, G, window, causal, err):
    """Dozens of short, partly overlapping image ranges: a 128-row tile meets more of
    them than an item record holds, so the softmax scans the sequence's ranges itself."""
    rng = np.random.default_rng(7 * D + G)
    qlen = np.array([333, 517], dtype=np.int32)
    ctx = np.array([150, 41], dtype=np.int32)
    seq = (ctx + qlen).astype(np.int32)
    per = []
    for s in range(2):
        lst = []
        for a in range(3, int(seq[s]) - 12, 13):
            b = a + int(rng.integers(0, 12))          # 1 to 12 tokens, every 13th start
            lst.append((a, b))
        lst.append((int(seq[s]) // 3, int(seq[s]) // 3 + 90))   # one that overlaps several
        per.append(lst)
    bt, nb = W._block_table(rng, seq, 32, spare_blocks=5)
    lay = W.Layout(f"many_ranges_d{D}_g{G}", query_lens=qlen, seq_lens=seq, mm_ranges=W._pad_ranges(per),
                   block_table=bt, num_blocks=nb, num_heads_q=2 * G, num_heads_kv=2, head_dim=D,
                   block_size=32, window=window, causal=causal, dtype="bf16",
                   max_num_tokens=int(qlen.sum()) + 9)
    _check(lay, _all_rows(lay), err=err)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_output_aligned_to_16_bytes_only(D, err):
    """The library asks for 16-byte aligned outputs; one that is not 32-byte aligned
    must give the same rows as the oracle (the output tensor map and the plain
    copies of partial tiles need 16 bytes only)."""
    lay = W.random_small(300 + D, head_dim=D, block_size=32, group=2, max_seqs=3, max_ctx=400, max_q=300,
                         window=200, with_ranges=True)
    q, k, v, d = gpu_inputs(lay, data_seed=3)
    big = torch.empty(q.numel() + 8, dtype=q.dtype, device=q.device)
    out = big[8:].view(q.shape)
    assert out.data_ptr() % 32 == 16
    o, lse = swa.swa_mm_paged_attention(
        q, k, v, d["block_table"], d["query_start_loc"], d["seq_lens"], context_lens=d["context_lens"],
        mm_ranges=d["mm_ranges"], max_query_len=lay.max_query_len, window=lay.window, causal=lay.causal,
        scale=lay.scale, out=out, err=err)
    assert o.data_ptr() == out.data_ptr()
    rows = _all_rows(lay)
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay) and e_lse <= LSE_ATOL, (e_out, e_lse)
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_group_of_three_all_rows(dtype, err):
    """A GQA group that does not divide the 128-row tile (the CUDA-core kernel's case)."""
    lay = W.random_small(77, head_dim=128, block_size=16, group=3, dtype=dtype, max_seqs=3, max_ctx=300,
                         max_q=200, window=100, with_ranges=True)
    assert lay.num_heads_q == 3 * lay.num_heads_kv
    _check(lay, _all_rows(lay), err=err)


@pytest.mark.parametrize("dtype,D,G,P,max_q", [
    ("fp32", 256, 2, 1, 200),    # 32-key tiles (fp32 operand pairs at head_dim 256)
    ("fp32", 128, 4, 3, 150),    # fp32 split partials, then the merge
    ("bf16", 64, 32, 1, 120),    # a GQA group only the general tensor-core kernel takes
    ("bf16", 128, 1, 4, 300),    # split-KV prefill with more rows than the decode kernel takes
    ("bf16", 256, 8, 2, 260)])
def test_general_tensor_core_kernel_shapes(dtype, D, G, P, max_q, err):
    """Shapes that run on the general tcgen05 kernel, every row against the oracle
    (split cases through lse_combine)."""
    from paged_sliding_window_swa_gb300 import lse_combine
    lay = W.random_small(400 + D + G + P, head_dim=D, group=G, dtype=dtype, max_seqs=3, max_ctx=600,
                         max_q=max_q, window=int(np.random.default_rng(D * G).choice([0, 64, 300])),
                         with_ranges=True, num_splits=P)
    q, k, v, d = gpu_inputs(lay, data_seed=5)
    rows = _all_rows(lay)
    if P == 1:
        out, lse = run_attention(lay, q, k, v, d, err=err)
    else:
        po, pl = run_attention(lay, q, k, v, d, err=err)
        out, lse = lse_combine(po, pl)
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay), e_out
    assert e_lse <= LSE_ATOL, e_lse
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("seed", range(60))
def test_random_layout_sweep(seed, err):
    """Random dtype, head_dim, GQA group, split count, window, causal flag, image ranges,
    page size and lengths (up to 3000 tokens of context and 700 queries per sequence):
    every kernel the dispatch can choose, against the oracle on up to 2500 rows."""
    from paged_sliding_window_swa_gb300 import lse_combine
    rng = np.random.default_rng(9000 + seed)
    D = int(rng.choice([64, 128, 256]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    dtype = "fp32" if rng.random() < 0.2 else "bf16"
    P = int(rng.choice([1, 1, 1, 2, 5]))
    lay = W.random_small(9000 + seed, head_dim=D, group=G, dtype=dtype, max_seqs=int(rng.integers(1, 4)),
                         max_ctx=int(rng.choice([50, 900, 3000])), max_q=int(rng.choice([1, 40, 300, 700])),
                         num_splits=P)
    q, k, v, d = gpu_inputs(lay, data_seed=seed)
    rows = _all_rows(lay)
    if len(rows) > 2500:
        rows = [rows[i] for i in sorted(rng.choice(len(rows), 2500, replace=False))]
    if P == 1:
        out, lse = run_attention(lay, q, k, v, d, err=err)
    else:
        po, pl = run_attention(lay, q, k, v, d, err=err)
        out, lse = lse_combine(po, pl)
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay), e_out
    assert e_lse <= LSE_ATOL, e_lse
    torch.cuda.synchronize()
    assert err.item() == 0


def test_unused_cache_rows_never_reach_the_output(err):
    """Spare blocks and page tails hold NaN; the output must stay finite and exact."""
    for seed in range(4):
        lay = W.random_small(40 + seed, max_seqs=3, max_ctx=300, max_q=200, block_size=64,
                             with_ranges=True)
        out, _, _ = _check(lay, _all_rows(lay), poison=True, err=err)
        assert torch.isfinite(out.float()).all()


def test_removing_image_ranges_changes_output(err):
    lay = W.geometry("causal")
    q, k, v, d = gpu_inputs(lay)
    with_mm, _ = run_attention(lay, q, k, v, d, err=err)
    without, _ = run_attention(lay, q, k, v, d, err=err, mm=False)
    rows = [(t, h) for t in range(1024, 2304, 16) for h in range(lay.num_heads_q)]
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, _ = max_errors(with_mm, None, ro, rl, rows)
    change = (with_mm.float() - without.float()).abs()[1024:2304].max().item()
    assert change >= max(4 * e_out, 1e-3), (change, e_out)


def test_bad_block_id_is_reported(err):
    lay = W.random_small(9, max_seqs=2, max_q=100, max_ctx=100)
    q, k, v, d = gpu_inputs(lay)
    d["block_table"][0, 0] = lay.num_blocks + 5
    out, _ = run_attention(lay, q, k, v, d, err=err)
    torch.cuda.synchronize()
    assert err.item() & 0x01
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("seed", range(6))
def test_split_partials_and_merge(seed, err):
    from paged_sliding_window_swa_gb300 import lse_combine
    P = [2, 3, 5, 8, 16, 4][seed]
    lay = W.random_small(200 + seed, max_seqs=3, max_ctx=2000, max_q=40, num_splits=P,
                         with_ranges=seed % 2 == 0, dtype="fp32" if seed == 5 else "bf16")
    q, k, v, d = gpu_inputs(lay)
    po, pl = run_attention(lay, q, k, v, d, err=err)
    rows = _all_rows(lay)
    ro, rl = oracle_rows(lay, q, k, v, rows, num_splits=P)
    pof = po.float().cpu().numpy()
    plc = pl.cpu().numpy()
    for (p, t, h), val in ro.items():
        if rl[(p, t, h)] == -np.inf:
            assert plc[p, t, h] == -np.inf
        else:
            assert abs(plc[p, t, h] - rl[(p, t, h)]) <= LSE_ATOL
            assert np.abs(pof[p, t, h] - val).max() <= atol_for(lay)
    mo, ml = lse_combine(po, pl)
    uo, ul = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(mo, ml, uo, ul, rows)
    assert e_out <= atol_for(lay) and e_lse <= LSE_ATOL
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("D,G,max_q,P,window,ranges", [
    (128, 4, 1, 32, 0, False), (128, 4, 1, 1, 0, False), (64, 2, 2, 4, 100, True),
    (256, 1, 4, 3, 0, True), (128, 2, 1, 8, 37, False), (256, 4, 1, 5, 300, True),
    (64, 1, 3, 1, 0, True), (128, 4, 1, 16, 1, False)])
def test_decode_kernel_cases(D, G, max_q, P, window, ranges, err):
    """Few query tokens per sequence (the decode path), split or not, all rows."""
    from paged_sliding_window_swa_gb300 import lse_combine
    lay = W.random_small(300 + D + G + P, head_dim=D, group=G, max_seqs=4, max_ctx=3000, max_q=max_q,
                         window=window, with_ranges=ranges, num_splits=P)
    q, k, v, d = gpu_inputs(lay, poison=True)
    rows = _all_rows(lay)
    res = run_attention(lay, q, k, v, d, err=err)
    if P > 1:
        po, pl = res
        ro, rl = oracle_rows(lay, q, k, v, rows, num_splits=P)
        pof, plc = po.float().cpu().numpy(), pl.cpu().numpy()
        for (p, t, h), val in ro.items():
            if rl[(p, t, h)] == -np.inf:
                assert plc[p, t, h] == -np.inf
            else:
                assert abs(plc[p, t, h] - rl[(p, t, h)]) <= LSE_ATOL
                assert np.abs(pof[p, t, h] - val).max() <= atol_for(lay)
        out, lse = lse_combine(po, pl)
    else:
        out, lse = res
    uo, ul = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, uo, ul, rows)
    assert e_out <= atol_for(lay) and e_lse <= LSE_ATOL
    torch.cuda.synchronize()
    assert err.item() == 0


def test_decode_split_kv_sampled(err):
    """128 single-token queries over 4k-64k contexts, 8-32 partitions, merged."""
    from paged_sliding_window_swa_gb300 import lse_combine
    lay = W.decode()
    q, k, v, d = gpu_inputs(lay)
    po, pl = run_attention(lay, q, k, v, d, err=err)
    mo, ml = lse_combine(po, pl)
    rng = np.random.default_rng(0)
    seqs = sorted(set(rng.integers(0, lay.num_seqs, 6).tolist()) | {int(np.argmax(lay.seq_lens))})
    rows = [(int(s), int(h)) for s in seqs for h in rng.integers(0, lay.num_heads_q, 3)]
    ro, rl = oracle_rows(lay, q, k, v, rows, num_splits=lay.num_splits)
    pof, plc = po.float().cpu().numpy(), pl.cpu().numpy()
    for (p, t, h), val in ro.items():
        if rl[(p, t, h)] == -np.inf:
            assert plc[p, t, h] == -np.inf
        else:
            assert abs(plc[p, t, h] - rl[(p, t, h)]) <= LSE_ATOL
            assert np.abs(pof[p, t, h] - val).max() <= 2e-2
    uo, ul = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(mo, ml, uo, ul, rows)
    assert e_out <= 2e-2 and e_lse <= LSE_ATOL
    torch.cuda.synchronize()
    assert err.item() == 0


def test_split_attention_and_merge_replay_in_a_cuda_graph(err):
    """Split-KV attention followed by the merge (a programmatic dependent launch),
    captured into a CUDA graph with all prefill kernels of the library and replayed:
    bit-identical to the same calls made eagerly."""
    from paged_sliding_window_swa_gb300 import lse_combine
    lay = W.random_small(77, head_dim=128, block_size=16, group=4, max_seqs=3, max_ctx=1500, max_q=1,
                         num_splits=8, with_ranges=False)
    q, k, v, d = gpu_inputs(lay, data_seed=9)
    P = lay.num_splits
    po = torch.empty((P,) + tuple(q.shape), dtype=q.dtype, device=q.device)
    pl = torch.empty((P,) + tuple(q.shape[:2]), dtype=torch.float32, device=q.device)
    mo = torch.empty_like(q)
    ml = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    lay2 = W.random_small(12, head_dim=256, block_size=32, group=2, max_seqs=2, max_ctx=400, max_q=300,
                          window=200, with_ranges=True)
    q2, k2, v2, d2 = gpu_inputs(lay2, data_seed=4)
    o2 = torch.empty_like(q2)
    l2 = torch.empty(q2.shape[:2], dtype=torch.float32, device=q2.device)

    def calls():
        swa.swa_mm_paged_attention(q, k, v, d["block_table"], d["query_start_loc"], d["seq_lens"],
                                   context_lens=d["context_lens"], max_query_len=lay.max_query_len,
                                   window=lay.window, causal=lay.causal, scale=lay.scale, num_splits=P,
                                   splits_per_seq=d["splits_per_seq"], partial_out=po, partial_lse=pl, err=err)
        lse_combine(po, pl, out=mo, out_lse=ml)
        swa.swa_mm_paged_attention(q2, k2, v2, d2["block_table"], d2["query_start_loc"], d2["seq_lens"],
                                   context_lens=d2["context_lens"], mm_ranges=d2["mm_ranges"],
                                   max_query_len=lay2.max_query_len, window=lay2.window, causal=lay2.causal,
                                   scale=lay2.scale, out=o2, lse=l2, err=err)

    calls()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (mo, ml, o2, l2)]
    for t in (mo, ml, o2, l2):
        t.fill_(7)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls()                                    # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for t in (mo, ml, o2, l2):
        t.fill_(7)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for got, want in zip((mo, ml, o2, l2), ref):
        assert torch.equal(got, want)
    assert err.item() == 0


def test_repeated_calls_are_bit_identical(err):
    """No atomics in the arithmetic: any run-to-run difference is a race."""
    lay = W.gemma_like()
    q, k, v, d = gpu_inputs(lay)
    ref, ref_lse = run_attention(lay, q, k, v, d, err=err)
    ref, ref_lse = ref.clone(), ref_lse.clone()
    for _ in range(4):
        out, lse = run_attention(lay, q, k, v, d, err=err)
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("D,scale", [(256, -0.07), (128, -0.11), (256, 0.0), (128, 0.3), (64, -0.09), (64, 0.0)])
def test_scale_sign_and_zero_all_rows(D, scale, err):
    """Any finite scale: a negative one (the max is taken on -S), zero (every
    visible key weighs the same) and a large one, on the tensor-core path."""
    import paged_sliding_window_swa_gb300 as swa
    lay = W.random_small(700 + D, head_dim=D, block_size=16, group=2, max_seqs=2, max_ctx=400, max_q=200,
                         window=150, with_ranges=True, dtype="bf16")
    q, k, v, d = gpu_inputs(lay)
    out, lse = swa.swa_mm_paged_attention(
        q, k, v, d["block_table"], d["query_start_loc"], d["seq_lens"], context_lens=d["context_lens"],
        mm_ranges=d["mm_ranges"], max_query_len=lay.max_query_len, window=lay.window, causal=lay.causal,
        scale=scale, err=err)
    rows = _all_rows(lay)
    ro, rl = O.attention(q.cpu(), k.cpu(), v.cpu(), lay.block_table, lay.query_start_loc, lay.seq_lens,
                         lay.mm_ranges, lay.window, lay.causal, scale, rows=rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay) and e_lse <= LSE_ATOL, (e_out, e_lse)
    torch.cuda.synchronize()
    assert err.item() == 0
