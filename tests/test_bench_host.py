"""Host-side checks of bench.py: its visible-pair count (the FLOP numerator)
equals the oracle's per-pair count."""
import numpy as np
import pytest

import bench
import workloads as W
from oracle import swa_oracle as O


@pytest.mark.parametrize("lay", [W.tiny(), W.geometry("causal"), W.geometry("noncausal")]
                         + [W.random_small(s, max_seqs=3, max_ctx=200, max_q=150) for s in range(8)],
                         ids=lambda l: l.name)
def test_visible_pair_count_matches_oracle(lay):
    ref = O.allowed_pair_count(lay.query_start_loc, lay.seq_lens, lay.mm_ranges, lay.window, lay.causal)
    assert bench.visible_pairs_per_head(lay) == ref


def test_gemma_like_count_is_stable():
    lay = W.gemma_like()
    n = bench.visible_pairs_per_head(lay)
    # about W + half an image per query beyond the window
    assert 60e6 < n < 90e6


@pytest.mark.parametrize("seed", range(8))
def test_visible_pair_count_with_chunks_and_flags_matches_oracle(seed):
    from dataclasses import replace
    rng = np.random.default_rng(seed)
    lay = W.random_small(60 + seed, max_seqs=3, max_ctx=200, max_q=150, with_ranges=True,
                         window=int(rng.choice([5, 40, 300])))
    lay = replace(lay, chunk_size=int(rng.choice([1, 16, 50])), chunk_lookback=int(rng.choice([-1, 0, 2])),
                  seq_causal=rng.integers(0, 2, size=lay.num_seqs).astype(np.int32))
    ref = O.allowed_pair_count(lay.query_start_loc, lay.seq_lens, lay.mm_ranges, lay.window, lay.causal,
                               seq_causal=lay.seq_causal, chunk_size=lay.chunk_size,
                               chunk_lookback=lay.chunk_lookback)
    assert bench.visible_pairs_per_head(lay) == ref


def test_workload_text_names_each_layout():
    g = bench.workload_text(W.gemma_like())
    assert g.startswith("gemma_like") and "D=256" in g and "73728" in g
    c = bench.workload_text(W.chunked_prefill(True))
    assert c.startswith("chunked_prefill") and "D=128" in c and "causal" in c and "Hq=32" in c


def test_traffic_is_reported_only_for_the_measured_workload():
    # another request count than the one the counters were taken on: no traffic
    assert bench.kernel_traffic(1) is None
    t = bench.kernel_traffic(bench.MEASURED_TRAFFIC["requests"])
    assert t is None or t == bench.MEASURED_TRAFFIC["bytes"]


def test_clock_samples_are_taken_from_the_timed_region():
    import datetime
    base = datetime.datetime(2026, 1, 1, 12, 0, 0)
    def line(ms, sm, sw_power="Not Active", hw="Not Active"):
        ts = (base + datetime.timedelta(milliseconds=ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, {sm}, 2070, 900.00, 0x0, {hw}, Not Active, Not Active, {sw_power}"
    out = "\n".join([line(0, 1200), line(50, 2070), line(100, 2070, sw_power="Active"), line(150, 2070),
                     line(400, 990, hw="Active")])
    t0 = base.timestamp()
    c = bench.summarise_clocks(out, window=(t0 + 0.06, t0 + 0.14), margin_s=0.05)
    assert c["samples"] == 3 and c["in_region"] and c["sm_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]            # the idle and the late samples are left out
    short = bench.summarise_clocks(out, window=(t0 + 0.3, t0 + 0.301), margin_s=0.01)
    assert short["samples"] == 2 and not short["in_region"]
