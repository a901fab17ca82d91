"""Failure detection in the tensor-core attention kernels, on a GPU, without a
fault: every pipeline wait of the tcgen05 kernels is bounded, and a call made
after swa_set_watchdog(limit, stall=True) makes one wait per CTA wait on a
barrier that nothing signals.  That wait runs out after the limit, the CTA
stops through its timeout path (abort flag, drain of its own copies and
MMAs, TMEM released) and the call reports SWA_ERR_TIMEOUT.  The context must
stay usable: an ordinary call right after it matches the oracle.

Both tensor-core kernels are covered: head_dim 128 (two query tiles per work
item) and head_dim 256."""
import time

import pytest
import torch

import paged_sliding_window_swa_gb300 as swa
import workloads as W
from _gpu_helpers import LSE_ATOL, atol_for, gpu_inputs, max_errors, oracle_rows, run_attention

pytestmark = pytest.mark.gpu

SWA_ERR_TIMEOUT = 0x10


def _layout(head_dim):
    # bf16, GQA group 2, several query rows per sequence: the tcgen05 kernels
    return W.random_small(41 + head_dim, head_dim=head_dim, group=2, block_size=16, dtype="bf16", max_seqs=3,
                          max_ctx=400, max_q=300, window=96, causal=True, with_ranges=True)


@pytest.mark.parametrize("head_dim", [128, 256])
def test_gpu_timeout_reports_and_recovers(head_dim):
    lay = _layout(head_dim)
    q, k, v, d = gpu_inputs(lay, data_seed=5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        swa.swa_set_watchdog(2_000_000, stall=True)        # 2 ms bound, a wait that cannot complete
        t0 = time.perf_counter()
        run_attention(lay, q, k, v, d, err=err)
        torch.cuda.synchronize()
        stalled_s = time.perf_counter() - t0
    finally:
        swa.swa_set_watchdog(0, stall=False)
    assert err.item() & SWA_ERR_TIMEOUT, hex(err.item())
    assert stalled_s < 10.0, stalled_s                    # the drains end well inside their own bound

    # an ordinary call right after: no error, every row matches the oracle
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_attention(lay, q, k, v, d, err=err2)
    torch.cuda.synchronize()
    assert err2.item() == 0, hex(err2.item())
    rows = [(t, h) for t in range(lay.num_tokens) for h in range(lay.num_heads_q)]
    ro, rl = oracle_rows(lay, q, k, v, rows)
    e_out, e_lse = max_errors(out, lse, ro, rl, rows)
    assert e_out <= atol_for(lay), e_out
    assert e_lse <= LSE_ATOL, e_lse


def test_gpu_short_bound_without_stall_is_harmless():
    """A 1 ms bound is far above any real wait of a small call: no timeout,
    same result as with the default bound."""
    lay = _layout(128)
    q, k, v, d = gpu_inputs(lay, data_seed=6)
    ref_out, ref_lse = run_attention(lay, q, k, v, d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        swa.swa_set_watchdog(1_000_000, stall=False)
        out, lse = run_attention(lay, q, k, v, d, err=err)
        torch.cuda.synchronize()
    finally:
        swa.swa_set_watchdog(0, stall=False)
    assert err.item() == 0, hex(err.item())
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
