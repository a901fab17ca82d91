"""swa_mm_paged_attention_split_static: split-KV attention and its LSE merge
for callers that cannot allocate device memory when they run attention (an
engine whose allocator holds the whole device, a plugin host that forbids
allocation while enqueuing, a loop that cannot take cudaMalloc's device-wide
synchronisation).  The split partials live in an array the library owns.

The GPU test calls the entry point through the C ABI twice in a row, on two
different batches, and checks each result against the ordinary path
(swa_mm_paged_attention with caller-allocated partials, then lse_combine) with
the tolerances of the other parity tests.  The second call checks that what the
first left in the shared array does not leak into its result.  This file is
named to be collected last, so a run that stops at the first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest

import paged_sliding_window_swa_gb300 as swa
import workloads as W

SWA_E_SIZE, SWA_E_SCRATCH = -2, -6


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


@pytest.mark.gpu
def test_static_scratch_matches_the_allocating_path_on_two_calls_in_a_row():
    import torch
    from _gpu_helpers import LSE_ATOL, atol_for, gpu_inputs, run_attention

    layouts = [
        # decode-like: one query per sequence, full attention, 8 partitions
        W.random_small(901, head_dim=128, group=4, max_seqs=4, max_ctx=3000, max_q=1, window=0,
                       with_ranges=False, num_splits=8),
        # a few queries per sequence, SWA with image ranges, 5 partitions
        W.random_small(902, head_dim=256, group=2, max_seqs=4, max_ctx=2000, max_q=40, window=300,
                       with_ranges=True, num_splits=5, dtype="bf16"),
    ]
    for call, lay in enumerate(layouts):
        q, k, v, d = gpu_inputs(lay, data_seed=7 + call)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        po, pl = run_attention(lay, q, k, v, d, err=err)
        ref_out, ref_lse = swa.lse_combine(po, pl)

        out = torch.full_like(q, float("nan"))
        lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
        err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _call_static(lay, q, k, v, d, out, lse, err2)
        assert rc == 0, f"call {call}: rc {rc}"
        torch.cuda.synchronize()
        assert err.item() == 0 and err2.item() == 0

        o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
        assert np.isfinite(o).all()
        assert np.abs(o - r).max() <= atol_for(lay), f"call {call}"
        l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
        both_inf = np.isneginf(l) & np.isneginf(rl)
        assert (np.isneginf(l) == np.isneginf(rl)).all()
        assert np.abs(np.where(both_inf, 0.0, l - rl)).max() <= LSE_ATOL, f"call {call}"


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
