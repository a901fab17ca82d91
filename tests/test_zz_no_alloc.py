"""swa_mm_paged_attention_split_static: split-KV attention and its LSE merge
for callers that cannot allocate device memory when they run attention (an
engine whose allocator holds the whole device, a plugin host that forbids
allocation while enqueuing, a loop that cannot take cudaMalloc's device-wide
synchronisation).  The split partials live in an array the library owns.

The GPU test calls the entry point through the C ABI three times in a row:

1. and 2. two different batches, each checked against the ordinary path
   (swa_mm_paged_attention with caller-allocated partials, then lse_combine)
   and, on sampled rows, against the CPU oracle, with the tolerances of the
   other parity tests;
3. the second batch's shapes again, with one sequence rejected on the device
   (a wrong context length) and the last tokens covered by no sequence.  The
   array still holds the second call's finite partials in those rows, so
   their output is 0 and their LSE -inf only if the call resets the array.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

import paged_sliding_window_swa_gb300 as swa
import workloads as W

SWA_E_SIZE, SWA_E_SCRATCH = -2, -6
SWA_ERR_LENS = 0x08


def _call_static(lay, q, k, v, d, out, lse, err):
    """One call of the entry point through the raw C ABI (ctypes)."""
    P = lay.num_splits
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())   # noqa: E731
    import torch
    mm = d["mm_ranges"]
    return swa.lib().swa_mm_paged_attention_split_static(
        p(q), p(k), p(v), k.shape[0], p(d["block_table"]), d["block_table"].shape[1],
        p(d["query_start_loc"]), p(d["seq_lens"]), p(d["context_lens"]), p(mm),
        0 if mm is None else mm.shape[1], lay.num_seqs, q.shape[0], lay.max_query_len,
        q.shape[1], k.shape[2], q.shape[2], k.shape[1], lay.window, int(lay.causal),
        p(d.get("seq_causal")), lay.chunk_size, lay.chunk_lookback, float(lay.scale),
        swa.DTYPE_BF16 if q.dtype == torch.bfloat16 else swa.DTYPE_FP32, P, p(d["splits_per_seq"]),
        p(out), p(lse), p(err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _static(lay, q, k, v, d):
    import torch
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _call_static(lay, q, k, v, d, out, lse, err)
    torch.cuda.synchronize()
    return rc, out, lse, int(err.item())


def _check_rows(out, lse, ref_out, ref_lse, rows, atol, lse_atol, what):
    o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
    l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
    t, h = rows
    assert np.isfinite(o[t, h]).all(), what
    assert np.abs(o[t, h] - r[t, h]).max() <= atol, what
    a, b = l[t, h], rl[t, h]
    assert (np.isneginf(a) == np.isneginf(b)).all(), what
    both = np.isneginf(a) & np.isneginf(b)
    assert np.abs(np.where(both, 0.0, a - b)).max() <= lse_atol, what


@pytest.mark.gpu
def test_static_scratch_matches_the_allocating_path_on_two_calls_in_a_row():
    import torch
    from _gpu_helpers import LSE_ATOL, atol_for, gpu_inputs, oracle_rows, run_attention, sample_rows

    layouts = [
        # decode-like: one query per sequence, full attention, 8 partitions
        W.random_small(901, head_dim=128, group=4, max_seqs=4, max_ctx=3000, max_q=1, window=0,
                       with_ranges=False, num_splits=8),
        # a few queries per sequence, SWA with image ranges, 5 partitions
        W.random_small(902, head_dim=256, group=2, max_seqs=4, max_ctx=2000, max_q=40, window=300,
                       with_ranges=True, num_splits=5, dtype="bf16"),
    ]
    kept = None
    for call, lay in enumerate(layouts):
        q, k, v, d = gpu_inputs(lay, data_seed=7 + call)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        po, pl = run_attention(lay, q, k, v, d, err=err)
        ref_out, ref_lse = swa.lse_combine(po, pl)

        rc, out, lse, err2 = _static(lay, q, k, v, d)
        assert rc == 0, f"call {call}: rc {rc}"
        assert err.item() == 0 and err2 == 0
        T, H = q.shape[0], q.shape[1]
        every = (np.repeat(np.arange(T), H), np.tile(np.arange(H), T))
        _check_rows(out, lse, ref_out, ref_lse, every, atol_for(lay), LSE_ATOL, f"call {call}")

        # the same result straight against the oracle, on sampled rows
        rows = sample_rows(lay, 48, seed=call)
        o_ref, l_ref = oracle_rows(lay, q.cpu(), k.cpu(), v.cpu(), rows)
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        for t, h in rows:
            assert np.abs(o[t, h] - o_ref[(t, h)]).max() <= atol_for(lay), (call, t, h)
            if np.isneginf(l_ref[(t, h)]):
                assert np.isneginf(l[t, h])
            else:
                assert abs(float(l[t, h]) - l_ref[(t, h)]) <= LSE_ATOL, (call, t, h)
        kept = (lay, q, k, v, d, out, lse)

    # Third call, the second call's shapes: sequence 0 is rejected on the
    # device (its context length is off by one) and the last 3 tokens belong
    # to no sequence (the last sequence loses its last 3 queries and keys).
    lay, q, k, v, d, out2, lse2 = kept
    S = lay.num_seqs
    assert S >= 2 and int(lay.query_lens[S - 1]) > 3
    d3 = dict(d)
    ctx = d["context_lens"].clone()
    ctx[0] += 1
    qsl = d["query_start_loc"].clone()
    qsl[S] -= 3
    seq = d["seq_lens"].clone()
    seq[S - 1] -= 3
    d3.update(context_lens=ctx, query_start_loc=qsl, seq_lens=seq)
    rc, out3, lse3, err3 = _static(lay, q, k, v, d3)
    assert rc == 0
    assert err3 & SWA_ERR_LENS
    T, H = q.shape[0], q.shape[1]
    q0, q1 = int(lay.query_start_loc[0]), int(lay.query_start_loc[1])
    dead = list(range(q0, q1)) + list(range(T - 3, T))
    o3, l3 = out3.float().cpu().numpy(), lse3.cpu().numpy()
    assert np.isfinite(out2.float().cpu().numpy()[dead]).all()      # the array held finite partials there
    assert not np.isneginf(lse2.cpu().numpy()[dead]).all()
    assert (o3[dead] == 0).all() and np.isneginf(l3[dead]).all()
    # the sequences in between are untouched by the change: bit-identical to call 2
    live = list(range(q1, int(lay.query_start_loc[S - 1])))
    if live:
        assert np.array_equal(o3[live], out2.float().cpu().numpy()[live])
        assert np.array_equal(l3[live], lse2.cpu().numpy()[live])


def test_static_scratch_rejects_oversized_and_unsplit_calls():
    """Size checks return before any CUDA work, so they need no GPU."""
    lib = swa.lib()
    dummy = ctypes.c_void_p(256)
    args = lambda T, P: (dummy, dummy, dummy, 1, dummy, 1, dummy, dummy, None, None, 0, 1, T, 1,   # noqa: E731
                         32, 8, 128, 16, 0, 1, None, 0, -1, 0.088, swa.DTYPE_BF16, P, None, dummy,
                         None, None, None)
    # 32 partitions x 128 tokens x 32 heads x 128 bf16 = 32 MiB of partials > 16 MiB
    assert lib.swa_mm_paged_attention_split_static(*args(128, 32)) == SWA_E_SCRATCH
    assert lib.swa_mm_paged_attention_split_static(*args(128, 1)) == SWA_E_SIZE
    assert swa.STATIC_SCRATCH_BYTES == 16 << 20
