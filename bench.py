#!/usr/bin/env python3
"""Benchmark: Gemma-like multimodal prefill through the paged SWA library.

One step = the whole hot path over one batch: slot mapping (with the PAD tail
up to a multiple of 8192 tokens), tile bounds, and paged attention with the
sliding window and the window-clamped image mask, on 4 requests of ~16,550
tokens with 60 images of 256 tokens each (Hq=16, Hkv=8, D=256, bf16, W=1024,
causal, paged KV block 16).  Inputs are synthetic (seeded N(0,1)).

Metric: attention TFLOP/s counting only visible (query, key) pairs
(4 * D * Hq * pairs), plus prefill tokens/s and the fraction of the measured
bf16 dense tensor-core peak.  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
(N > 1: launched by torchrun, one independent replica per GPU.)
``--workload chunked_prefill`` (``chunked_prefill_d64``) runs the causal
chunked-prefill layout at head_dim 128 (64) as the step instead, for profiling
that kernel; the default line is the Gemma-like one.
"""
import os

for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")     # each oracle process runs one thread; one process per core

import argparse
import dataclasses
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "allowed-pair attention TFLOP/s & prefill tok/s (1×GB300), % of bf16 TC peak"
UNIT = "TFLOP/s"


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------
def visible_pairs_per_head(lay) -> int:
    """Visible (query, key) pairs of one head.

    The visible keys of a query form one interval: left edge the base
    window's (q-W+1, or with chunked lookback the start of the chunk L chunks
    back), lowered to max(s, q-W+1) by every image range [s, e] holding q;
    right edge the larger of the base window's right edge and the end of every
    such range.  So the count is a sum of interval lengths.
    """
    total = 0
    ctx = lay.context_lens
    chunked = lay.window > 0 and lay.chunk_lookback >= 0
    for s in range(lay.num_seqs):
        n = int(lay.seq_lens[s])
        causal = lay.causal if lay.seq_causal is None else bool(lay.seq_causal[s])
        q = ctx[s] + np.arange(int(lay.query_lens[s]), dtype=np.int64)
        if lay.window > 0:
            if chunked:
                lo = (q // lay.chunk_size - lay.chunk_lookback) * lay.chunk_size
            else:
                lo = q - lay.window + 1
            hi = q.copy() if causal else q + lay.window - 1
        else:
            lo = np.zeros_like(q)
            hi = q.copy() if causal else np.full_like(q, n - 1)
        if lay.mm_ranges is not None:
            for a, b in lay.mm_ranges[s]:
                if a < b:
                    sel = (q >= a) & (q <= b)
                    hi[sel] = np.maximum(hi[sel], b)
                    if lay.window > 0:
                        lo[sel] = np.minimum(lo[sel], np.maximum(a, q[sel] - lay.window + 1))
        lo = np.maximum(lo, 0)
        hi = np.minimum(hi, n - 1)
        total += int(np.maximum(hi - lo + 1, 0).sum())
    return total


# Every source the head_dim-256 attention kernel is compiled from: a change to
# any of them makes the stored DRAM counters stale.
TRAFFIC_SOURCES = ("paged_sliding_window_swa_gb300/csrc/attention_tc.cu",
                   "paged_sliding_window_swa_gb300/csrc/attn_tc_common.cuh",
                   "paged_sliding_window_swa_gb300/csrc/tc_ptx.cuh",
                   "paged_sliding_window_swa_gb300/csrc/common.cuh",
                   "paged_sliding_window_swa_gb300/csrc/launch.h",
                   "include/swa.h")


def kernel_source_sha():
    """sha256 (16 hex digits) over the attention kernel's sources, in order."""
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(num_requests):
    """DRAM bytes per attention launch on the 4-request workload, from the ncu
    launch list taken of the kernel built from the sources whose hash is stored
    with them; None for another workload or once any of those sources changed."""
    if num_requests != MEASURED_TRAFFIC["requests"]:
        return None
    try:
        sha = kernel_source_sha()
    except OSError:
        return None
    return MEASURED_TRAFFIC["bytes"] if sha == MEASURED_TRAFFIC["kernel_sha"] else None


# dram__bytes_read.sum + dram__bytes_write.sum of one attention launch (ncu, 1 pass)
MEASURED_TRAFFIC = {"kernel_sha": "1e51a5d60c518219", "requests": 4, "bytes": (1085.5 + 518.4) * 1e6}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of the SM clock and the throttle reasons.  Only the
    samples taken inside the timed region (host wall clock, a margin of one
    interval) are kept; when the region is shorter than the interval, the
    nearest samples stand in and `in_region` says so."""
    INTERVAL_MS = 50
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        return summarise_clocks(out, window, self.INTERVAL_MS / 1e3)


def summarise_clocks(out, window=None, margin_s=0.05):
    """Median SM clock, maximum clock and throttle reasons from nvidia-smi CSV
    lines (timestamp first); `window` = (t0, t1) host epoch seconds."""
    import datetime
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    rows = []
    for line in out.strip().splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            rows.append((ts, float(f[1]), float(f[2]), [n for n, v in zip(names, f[5:9]) if v.lower() == "active"]))
        except ValueError:
            continue
    inside = rows
    if window is not None and rows:
        inside = [r for r in rows if window[0] - margin_s <= r[0] <= window[1] + margin_s]
        if not inside:                      # region shorter than the interval: the nearest samples
            mid = 0.5 * (window[0] + window[1])
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
    reasons = sorted({n for r in inside for n in r[3]})
    return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
            "sm_max_mhz": max(r[2] for r in inside) if inside else None,
            "reasons": reasons, "samples": len(inside),
            "in_region": window is not None and bool(inside) and
            all(window[0] - margin_s <= r[0] <= window[1] + margin_s for r in inside)}


# ---------------------------------------------------------------------------
# the GPU path
# ---------------------------------------------------------------------------
class PrefillStep:
    """Device-resident inputs and outputs of one Gemma-like prefill step."""

    TILE, BLOCK_Q = 64, 32      # tile-bounds geometry reported alongside the attention

    def __init__(self, lay, device, data_seed=1):
        import paged_sliding_window_swa_gb300 as swa
        self.swa, self.lay, self.dev = swa, lay, device
        self.q, self.k, self.v = W.make_tensors(lay, device=device, data_seed=data_seed)
        self.d = W.device_layout(lay, device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.slots = torch.empty(lay.max_num_tokens, dtype=torch.int32, device=device)
        self.maxb = -(-lay.max_query_len // self.BLOCK_Q)
        self.bounds = torch.empty((lay.num_seqs, self.maxb, 3), dtype=torch.int32, device=device)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((lay.num_tokens, lay.num_heads_q), dtype=torch.float32, device=device)

    def feeders(self):
        lay, d, swa = self.lay, self.d, self.swa
        swa.swa_slot_mapping(d["query_start_loc"], d["positions"], d["block_table"], lay.block_size,
                             lay.max_num_tokens, out=self.slots, err=self.err)
        swa.swa_tile_bounds(d["query_start_loc"], d["seq_lens"], context_lens=d["context_lens"],
                            mm_ranges=d["mm_ranges"], window=lay.window, causal=lay.causal,
                            tile_size=self.TILE, block_q=self.BLOCK_Q, max_qblocks_per_seq=self.maxb,
                            out=self.bounds, err=self.err)

    def attention(self):
        lay, d = self.lay, self.d
        self.swa.swa_mm_paged_attention(
            self.q, self.k, self.v, d["block_table"], d["query_start_loc"], d["seq_lens"],
            context_lens=d["context_lens"], mm_ranges=d["mm_ranges"], max_query_len=lay.max_query_len,
            window=lay.window, causal=lay.causal, scale=lay.scale, out=self.out, lse=self.lse,
            err=self.err)

    def launches_per_step(self):
        return 3

    def capture(self):
        """The two feeders and the attention as two CUDA graphs (the same three
        launches with their fixed device pointers), so the small feeder kernels
        run back to back without a launch gap each."""
        self.g_feed, self.g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_feed):
            self.feeders()
        with torch.cuda.graph(self.g_attn):
            self.attention()
        torch.cuda.synchronize(self.dev)


def max_over_ranks(ms, world, device):
    """The job's time: the slowest rank's (a MAX all-reduce over the process
    group; NCCL needs a CUDA tensor, gloo a CPU one)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Units per second of the whole job: every replica processes the same
    number of units in the (max-over-ranks) time."""
    return world * units_per_rank / (ms * 1e-3)


def run_gpu(args, rank, world, local_rank):
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if args.workload == "gemma_like":
        lay = W.gemma_like(num_requests=args.requests)
    elif args.workload == "chunked_prefill":
        lay = W.chunked_prefill(True)
    else:
        lay = dataclasses.replace(W.chunked_prefill(True), name="chunked_prefill-head_dim64", head_dim=64)
    step = PrefillStep(lay, dev)
    pairs = visible_pairs_per_head(lay)
    flops = 4.0 * lay.head_dim * lay.num_heads_q * pairs
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step.feeders()
        step.attention()
    barrier()
    run_feeders, run_attention = step.feeders, step.attention
    if not args.no_graph:
        step.capture()
        run_feeders, run_attention = step.g_feed.replay, step.g_attn.replay
        for _ in range(args.warmup):
            run_feeders()
            run_attention()
        barrier()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    wall0 = time.time()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        run_feeders()
        ev[i][1].record(stream)
        run_attention()
        ev[i][2].record(stream)
    t_end.record(stream)
    barrier()
    total_ms = t_start.elapsed_time(t_end)
    clk = clocks.stop(window=(wall0, time.time()))
    attn_ms = [a.elapsed_time(b) for _, a, b in ev]
    feed_ms = [a.elapsed_time(b) for a, b, _ in ev]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps

    # end to end through the public API: pinned host inputs -> device -> the
    # calls -> host, every step inside the timed region
    e2e = run_e2e(args, step, flops, barrier, stream, world, dev) if not args.no_e2e else None
    torch.cuda.synchronize(dev)
    err = int(step.err.item())
    if rank != 0:
        return None
    return report_line(args, lay, step, flops, pairs, ms_per_step, attn_ms, feed_ms, clk, e2e, err, world)


def run_e2e(args, step, flops, barrier, stream, world, dev):
    """The step end to end through the public API, as a prefill engine runs it:
    every step copies the new tokens' q, k and v rows and the batch metadata
    from pinned host memory, maps the tokens to cache slots, writes the new K/V
    rows into the paged cache by slot (swa_kv_cache_write), computes the tile
    bounds and the attention, and copies out and lse back to the host.  The
    work is cut per request on three streams (host->device, compute,
    device->host) so request r's copies overlap request r-1's kernels, and
    consecutive steps are pipelined as a serving loop runs them: the device
    copies of a step's inputs and outputs alternate between two sets, so step
    i+1's host->device copies run while step i computes and copies its output
    back; a set is refilled only after the step two back has finished reading
    it (events).  The last step's host output is compared with the
    device-resident step's."""
    swa, lay = step.swa, step.lay
    qsl = [int(x) for x in lay.query_start_loc]
    R = lay.num_seqs
    slots = step.slots[:lay.num_tokens].long()
    k_flat = step.k.view(-1, lay.num_heads_kv, lay.head_dim)
    v_flat = step.v.view(-1, lay.num_heads_kv, lay.head_dim)
    host = {"q": step.q.cpu().pin_memory(), "k_new": k_flat[slots].cpu().pin_memory(),
            "v_new": v_flat[slots].cpu().pin_memory()}
    meta = {key: t.cpu().pin_memory() for key, t in step.d.items() if t is not None}
    out_h = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    lse_h = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + list(meta.values()))
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    sets = []
    for _ in range(2):
        sets.append({"d": {key: torch.empty_like(t, device=dev) for key, t in meta.items()},
                     "q": torch.empty_like(step.q), "k_new": torch.empty_like(host["k_new"], device=dev),
                     "v_new": torch.empty_like(host["v_new"], device=dev), "out": torch.empty_like(step.out),
                     "lse": torch.empty_like(step.lse), "in_free": None, "out_free": None})
    # per-request views of the batch (request r alone, its query rows start at 0)
    sub_qsl = [torch.tensor([0, qsl[r + 1] - qsl[r]], dtype=torch.int32, device=dev) for r in range(R)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    mm = meta.get("mm_ranges") is not None

    def e2e_step(i):
        S = sets[i % 2]
        d = S["d"]
        if S["in_free"] is not None:
            s_h2d.wait_event(S["in_free"])              # the step two back no longer reads this set
        got_meta, got = torch.cuda.Event(), []
        with torch.cuda.stream(s_h2d):
            for key, t in meta.items():
                d[key].copy_(t, non_blocking=True)
            got_meta.record(s_h2d)
            for r in range(R):
                a, b = qsl[r], qsl[r + 1]
                S["q"][a:b].copy_(host["q"][a:b], non_blocking=True)
                S["k_new"][a:b].copy_(host["k_new"][a:b], non_blocking=True)
                S["v_new"][a:b].copy_(host["v_new"][a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_h2d)
                got.append(e)
        stream.wait_event(got_meta)
        if S["out_free"] is not None:
            stream.wait_event(S["out_free"])             # its output was copied back
        swa.swa_slot_mapping(d["query_start_loc"], d["positions"], d["block_table"], lay.block_size,
                             lay.max_num_tokens, out=step.slots, err=step.err, stream=stream)
        swa.swa_tile_bounds(d["query_start_loc"], d["seq_lens"], context_lens=d["context_lens"],
                            mm_ranges=d["mm_ranges"] if mm else None, window=lay.window, causal=lay.causal,
                            tile_size=step.TILE, block_q=step.BLOCK_Q, max_qblocks_per_seq=step.maxb,
                            out=step.bounds, err=step.err, stream=stream)
        done = []
        for r in range(R):
            a, b = qsl[r], qsl[r + 1]
            stream.wait_event(got[r])
            swa.swa_kv_cache_write(S["k_new"][a:b], S["v_new"][a:b], step.slots[a:b], step.k, step.v,
                                   err=step.err, stream=stream)
            swa.swa_mm_paged_attention(
                S["q"][a:b], step.k, step.v, d["block_table"][r:r + 1], sub_qsl[r], d["seq_lens"][r:r + 1],
                context_lens=d["context_lens"][r:r + 1], mm_ranges=d["mm_ranges"][r:r + 1] if mm else None,
                max_query_len=b - a, window=lay.window, causal=lay.causal, scale=lay.scale,
                out=S["out"][a:b], lse=S["lse"][a:b], err=step.err, stream=stream)
            e = torch.cuda.Event()
            e.record(stream)
            done.append(e)
        S["in_free"] = done[-1]
        with torch.cuda.stream(s_d2h):
            for r in range(R):
                a, b = qsl[r], qsl[r + 1]
                s_d2h.wait_event(done[r])
                out_h[a:b].copy_(S["out"][a:b], non_blocking=True)
                lse_h[a:b].copy_(S["lse"][a:b], non_blocking=True)
        back = torch.cuda.Event()
        back.record(s_d2h)
        S["out_free"] = back
        return back

    ref_out = step.out.clone()
    stream.wait_event(e2e_step(0))
    stream.wait_event(e2e_step(1))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 10))
    e0.record(stream)
    for i in range(e2e_steps):
        last = e2e_step(i)
    stream.wait_event(last)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    same = bool(torch.equal(out_h, ref_out.cpu()))
    return {"value": round(job_rate(flops, world, e2e_ms) / 1e12, 3), "unit": UNIT,
            "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "step": "per request on three streams: H2D of q/k_new/v_new, swa_kv_cache_write + "
                    "swa_mm_paged_attention, D2H of out/lse; slot mapping and tile bounds once per step; "
                    "consecutive steps pipelined over two sets of device buffers",
            "matches_device_step": same}


def workload_text(lay):
    if lay.name.startswith("gemma_like"):
        return (f"{lay.name}: {lay.num_seqs} request(s) of {'/'.join(str(int(x)) for x in lay.seq_lens)} tokens, "
                "60 images x 256 tokens each, causal SWA W=1024 with the window-clamped image mask, Hq=16, "
                f"Hkv=8, D=256, bf16, paged KV block 16, slot mapping padded to {lay.max_num_tokens}")
    return (f"{lay.name}: {lay.num_seqs} requests, cached context "
            f"{'/'.join(str(int(x)) for x in lay.context_lens)} + 2048-token chunks, 0-40 images x 256 tokens, "
            f"SWA W={lay.window} {'causal' if lay.causal else 'non-causal'}, Hq={lay.num_heads_q}, "
            f"Hkv={lay.num_heads_kv}, D={lay.head_dim}, bf16, paged KV block {lay.block_size}")


def l2_note(step):
    """How the timed region treats L2 (129 MB): the step's inputs are larger
    than it, so no flush is needed between steps."""
    q_gb = step.q.numel() * step.q.element_size() / 1e9
    kv_gb = 2 * step.k.numel() * step.k.element_size() / 1e9
    return (f"inputs larger than L2 (q {q_gb:.2f} GB, K/V caches {kv_gb:.2f} GB), no flush"
            if min(q_gb, kv_gb) * 1e3 > 129 else f"q {q_gb:.2f} GB, K/V caches {kv_gb:.2f} GB: not all larger than L2")


def report_line(args, lay, step, flops, pairs, ms_per_step, attn_ms, feed_ms, clk, e2e, err, world):
    pk = peaks()
    attn_avg = statistics.mean(attn_ms)
    achieved = flops / (attn_avg * 1e-3) / 1e12
    value = job_rate(flops, world, ms_per_step) / 1e12
    tok_s = job_rate(lay.num_tokens, world, ms_per_step)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": workload_text(lay),
            "global_batch": lay.num_seqs * world,
            "seq_len": int(lay.seq_lens.mean()),
            "tokens_per_step": lay.num_tokens,
            "visible_pairs_per_head": pairs,
            "tflop_per_step": round(flops / 1e12, 4),
            "step": "swa_slot_mapping + swa_tile_bounds + swa_mm_paged_attention",
            "launch": "eager" if args.no_graph else "CUDA graph replay (feeders, attention)",
            "l2": l2_note(step),
            "parallelism": f"replicas x{world}",
        },
        "tok_per_s": round(tok_s, 1),
        "pct_of_bf16_peak": round(100.0 * value / world / pk["bf16_tflops"], 2),
        "roofline": {
            "bound": "tensor",
            "kernel": "swa_mm_paged_attention",
            "achieved": round(achieved, 3),
            "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(achieved / pk["bf16_tflops"], 4),
            "traffic": kernel_traffic(args.requests) if args.workload == "gemma_like" else None,
            "peak_source": f"{pk['source']} bf16 dense (burst)",
            "peak_sustained": pk["bf16_tflops_sustained"],
            "frac_sustained": (round(achieved / pk["bf16_tflops_sustained"], 4)
                               if pk.get("bf16_tflops_sustained") else None),
            "avg_launch_ms": round(attn_avg, 4),
        },
        "feeders_ms": round(statistics.mean(feed_ms), 4),
        "e2e": e2e,
        "gpu_launches": args.steps * step.launches_per_step(),
        "clocks": clk,
        "device_errors": err,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(lay, step, budget_s=args.cpu_seconds)
    if not args.no_extras:
        line["extras"] = run_extras(step.dev, pk)
    return line


# ---------------------------------------------------------------------------
# the other workloads and the bandwidth kernels (reported under "extras")
# ---------------------------------------------------------------------------
def _time_ms(fn, reps=5, flush=None):
    """Median device time of fn() in ms over `reps` launches (events on the current stream)."""
    out = []
    for _ in range(reps):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return statistics.median(out)


def run_extras(dev, pk):
    import paged_sliding_window_swa_gb300 as swa
    res = {}
    scratch = torch.empty(512 << 20, dtype=torch.uint8, device=dev)     # 512 MB > L2: flush

    def flush():
        scratch.fill_(1)

    # chunked prefill over cached context (head_dim 128, GQA 4), causal and non-causal, and
    # causal with chunked lookback (chunks of 2048, one chunk back) and alternating
    # per-sequence causal flags; the causal layout again at head_dim 64
    chunk_lay = dataclasses.replace(W.chunked_prefill(True), name="chunked_prefill-chunk2048-lookback1-mixed",
                                    chunk_size=2048, chunk_lookback=1,
                                    seq_causal=np.array([s % 2 for s in range(8)], np.int32))
    d64_lay = dataclasses.replace(W.chunked_prefill(True), name="chunked_prefill-head_dim64", head_dim=64)
    for lay in (W.chunked_prefill(True), W.chunked_prefill(False), chunk_lay, d64_lay):
        q, k, v = W.make_tensors(lay, device=dev)
        d = W.device_layout(lay, dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)

        def attn():
            swa.swa_mm_paged_attention(q, k, v, d["block_table"], d["query_start_loc"], d["seq_lens"],
                                       context_lens=d["context_lens"], mm_ranges=d["mm_ranges"],
                                       max_query_len=lay.max_query_len, window=lay.window, causal=lay.causal,
                                       seq_causal=d["seq_causal"], chunk_size=lay.chunk_size,
                                       chunk_lookback=lay.chunk_lookback, scale=lay.scale, out=out, lse=lse)
        attn()
        ms = _time_ms(attn)
        fl = 4.0 * lay.head_dim * lay.num_heads_q * visible_pairs_per_head(lay)
        res[lay.name] = {"ms": round(ms, 4), "tflops_visible": round(fl / ms / 1e9, 2),
                         "frac_of_bf16_peak": round(fl / ms / 1e9 / pk["bf16_tflops"], 4),
                         "tok_per_s": round(lay.num_tokens / ms * 1e3, 1)}
        del q, k, v, out

    # decode: 128 single-token queries over 4k-64k contexts, split-KV + LSE merge
    lay = W.decode()
    q, k, v = W.make_tensors(lay, device=dev)
    d = W.device_layout(lay, dev)
    P = lay.num_splits
    po = torch.empty((P,) + tuple(q.shape), dtype=q.dtype, device=dev)
    pl = torch.empty((P,) + tuple(q.shape[:2]), dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)

    def dec_attn():
        swa.swa_mm_paged_attention(q, k, v, d["block_table"], d["query_start_loc"], d["seq_lens"],
                                   context_lens=d["context_lens"], max_query_len=1, window=lay.window,
                                   causal=True, scale=lay.scale, num_splits=P,
                                   splits_per_seq=d["splits_per_seq"], partial_out=po, partial_lse=pl)

    def dec_merge():
        swa.lse_combine(po, pl, out=out, out_lse=lse)
    def dec_step():
        dec_attn()
        dec_merge()
    dec_step()
    ms_a = _time_ms(dec_attn)
    ms_m = _time_ms(dec_merge, flush=flush)
    ms_s = _time_ms(dec_step, reps=9, flush=flush)      # the two launches back to back, as a step runs them
    kv_bytes = float(lay.seq_lens.sum()) * lay.num_heads_kv * lay.head_dim * 2 * 2
    live = float(lay.splits_per_seq.sum()) * lay.num_heads_q
    m_bytes = live * lay.head_dim * 2 + lay.num_tokens * lay.num_heads_q * (P * 4 + lay.head_dim * 2 + 4)
    res["decode"] = {"attention_ms": round(ms_a, 4), "kv_gbs": round(kv_bytes / ms_a / 1e6, 1),
                     "kv_frac_of_hbm": round(kv_bytes / ms_a / 1e6 / pk["hbm_gbs"], 4),
                     "lse_combine_ms": round(ms_m, 4), "lse_combine_gbs": round(m_bytes / ms_m / 1e6, 1),
                     "step_ms": round(ms_s, 4)}
    del q, k, v, po, pl

    # bandwidth sweeps at sizes where HBM, not launch latency, sets the time (cold L2)
    n_tok, B = 1 << 26, 16
    lens = np.full(64, n_tok // 64, dtype=np.int64)
    qsl = torch.as_tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    pos = torch.cat([torch.arange(int(x), device=dev, dtype=torch.int64) for x in lens])
    pages = int(-(-lens.max() // B))
    bt = torch.randperm(64 * pages, device=dev, dtype=torch.int64).to(torch.int32).view(64, pages)
    maxn = n_tok + 8192
    slots = torch.empty(maxn, dtype=torch.int32, device=dev)
    sm_ms = _time_ms(lambda: swa.swa_slot_mapping(qsl, pos, bt, B, maxn, out=slots), flush=flush)
    sm_bytes = n_tok * (8 + 4) + (maxn - n_tok) * 4 + 64 * pages * 4
    res["slot_mapping_64M_tokens"] = {"ms": round(sm_ms, 4), "gbs": round(sm_bytes / sm_ms / 1e6, 1),
                                      "frac_of_hbm": round(sm_bytes / sm_ms / 1e6 / pk["hbm_gbs"], 4)}
    cp_ms = _time_ms(lambda: swa.swa_slot_mapping_cp(qsl, pos, bt, B, maxn, kv_cache_block_size=B, cp_world_size=4,
                                                     cp_rank=1, cp_interleave=B, out=slots), flush=flush)
    res["slot_mapping_cp4_64M_tokens"] = {"ms": round(cp_ms, 4), "gbs": round(sm_bytes / cp_ms / 1e6, 1),
                                          "frac_of_hbm": round(sm_bytes / cp_ms / 1e6 / pk["hbm_gbs"], 4)}
    del pos, slots
    # the step's new K/V rows into the paged cache (Gemma-like sizes: 66,200 tokens x 8 kv heads x 256)
    T_kv, hkv, D_kv = 66200, 8, 256
    kn = torch.randn((T_kv, hkv, D_kv), device=dev).to(torch.bfloat16)
    vn = torch.randn((T_kv, hkv, D_kv), device=dev).to(torch.bfloat16)
    nblk = -(-T_kv // B) + 64
    kc = torch.empty((nblk, B, hkv, D_kv), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kv_slots = torch.randperm(nblk * B, device=dev)[:T_kv].to(torch.int32)
    kv_ms = _time_ms(lambda: swa.swa_kv_cache_write(kn, vn, kv_slots, kc, vc), flush=flush)
    kv_bytes = 2 * 2 * T_kv * hkv * D_kv * 2 + T_kv * 4
    res["kv_cache_write_66200_tokens"] = {"ms": round(kv_ms, 4), "gbs": round(kv_bytes / kv_ms / 1e6, 1),
                                          "frac_of_hbm": round(kv_bytes / kv_ms / 1e6 / pk["hbm_gbs"], 4)}
    del kn, vn, kc, vc
    P, T, H, D = 8, 65536, 32, 128
    po = torch.randn((P, T, H, D), device=dev).to(torch.bfloat16)
    pl = torch.randn((P, T, H), device=dev)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    cm_ms = _time_ms(lambda: swa.lse_combine(po, pl, out=out, out_lse=lse), flush=flush)
    cm_bytes = P * T * H * (D * 2 + 4) + T * H * (D * 2 + 4)
    res["lse_combine_T65536_P8"] = {"ms": round(cm_ms, 4), "gbs": round(cm_bytes / cm_ms / 1e6, 1),
                                    "frac_of_hbm": round(cm_bytes / cm_ms / 1e6 / pk["hbm_gbs"], 4)}
    return res


# ---------------------------------------------------------------------------
# the oracle leg (CPU)
# ---------------------------------------------------------------------------
def _oracle_subproblem(lay, q, k, v, seed):
    """One (sequence, kv head) of the layout as a small oracle problem on the host."""
    rng = np.random.default_rng(seed)
    qsl = lay.query_start_loc
    s = int(rng.integers(0, lay.num_seqs))
    hk = int(rng.integers(0, lay.num_heads_kv))
    n = int(lay.seq_lens[s])
    pages = lay.block_table[s, :-(-n // lay.block_size)].astype(np.int64)
    G = lay.group
    return {
        "s": s, "hk": hk, "n": n, "ctx": n - int(lay.query_lens[s]), "G": G, "seed": seed,
        "q": q[int(qsl[s]):int(qsl[s + 1]), hk * G:(hk + 1) * G].cpu(),
        "k": k[torch.as_tensor(pages)][:, :, hk:hk + 1].cpu(),
        "v": v[torch.as_tensor(pages)][:, :, hk:hk + 1].cpu(),
        "bt": np.arange(len(pages), dtype=np.int32)[None],
        "qs": np.array([0, int(lay.query_lens[s])]),
        "mm": None if lay.mm_ranges is None else lay.mm_ranges[s:s + 1],
        "window": lay.window, "causal": lay.causal, "scale": lay.scale, "head_dim": lay.head_dim,
    }


def _oracle_time_rows(sub, budget_s, rng):
    """Time the oracle on random (token, head) rows of one subproblem for ``budget_s``."""
    from oracle import swa_oracle as O
    nq = sub["q"].shape[0]
    t0 = time.perf_counter()
    rows_done, pairs = 0, 0
    while time.perf_counter() - t0 < budget_s:
        batch = [(int(t), int(h)) for t, h in zip(rng.integers(0, nq, 8), rng.integers(0, sub["G"], 8))]
        O.attention(sub["q"], sub["k"], sub["v"], sub["bt"], sub["qs"], [sub["n"]], sub["mm"], sub["window"],
                    sub["causal"], sub["scale"], rows=batch)
        for t, _ in batch:
            pairs += int(O.visible_keys(sub["ctx"] + t, sub["n"], sub["window"], sub["causal"],
                                        None if sub["mm"] is None else sub["mm"][0]).sum())
        rows_done += len(batch)
    return rows_done, pairs, time.perf_counter() - t0


def _oracle_worker_main(conn):
    """A spawned single-thread process: receives its subproblem once, then one
    time budget per sample, and answers (rows, visible pairs, seconds)."""
    sub = conn.recv()
    rng = np.random.default_rng(sub["seed"] + 7)
    while True:
        budget_s = conn.recv()
        if budget_s is None:
            break
        conn.send(_oracle_time_rows(sub, budget_s, rng))
    conn.close()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


class OracleTeam:
    """The oracle on every host core: one spawned single-thread process per
    core, each holding its own (sequence, kv head) sample of the layout."""

    def __init__(self, lay, q, k, v, seed=0, procs=None):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.lay = lay
        self.procs = host_cores() if procs is None else procs
        self.workers = []
        for i in range(self.procs):
            parent, child = ctx.Pipe()
            proc = ctx.Process(target=_oracle_worker_main, args=(child,), daemon=True)
            proc.start()
            parent.send(_oracle_subproblem(lay, q, k, v, seed * 1000 + i))
            self.workers.append((proc, parent))

    def sample(self, budget_s):
        """Whole-host TFLOP/s of visible-pair work over one budget."""
        for _, conn in self.workers:
            conn.send(budget_s)
        res = [conn.recv() for _, conn in self.workers]
        rows = sum(r[0] for r in res)
        pairs = sum(r[1] for r in res)
        wall = max(r[2] for r in res)
        flops = 4.0 * self.lay.head_dim * pairs
        return {"value": flops / wall / 1e12, "unit": UNIT, "cores": self.procs, "host_cores": host_cores(),
                "kind": "oracle",
                "sample": f"{rows} random (token, head) rows over {self.procs} (sequence, kv head) samples, "
                          f"{pairs} visible pairs, {wall:.1f} s on {self.procs} single-thread processes "
                          f"(fp64 numpy, per-pair mask)",
                "rows_per_s": rows / wall,
                "tok_per_s": rows / self.lay.num_heads_q / wall}

    def close(self):
        for proc, conn in self.workers:
            conn.send(None)
            conn.close()
        for proc, _ in self.workers:
            proc.join(timeout=30)


def _oracle_sample(lay, q, k, v, budget_s, seed=0, procs=None):
    team = OracleTeam(lay, q, k, v, seed=seed, procs=procs)
    try:
        return team.sample(budget_s)
    finally:
        team.close()


def cpu_baseline(lay, step, budget_s):
    return _oracle_sample(lay, step.q, step.k, step.v, budget_s)


def run_reference(args, rank, world):
    if rank != 0:
        return None
    lay = W.gemma_like()
    q, k, v = W.make_tensors(lay, device="cpu")
    per_step = args.cpu_seconds / max(1, args.steps)
    team = OracleTeam(lay, q, k, v, seed=0)
    try:
        for _ in range(args.warmup):
            team.sample(min(per_step, 0.2))
        vals = []
        t0 = time.perf_counter()
        for i in range(args.steps):
            vals.append(team.sample(per_step))
        total = time.perf_counter() - t0
    finally:
        team.close()
    value = statistics.mean(v["value"] for v in vals)
    flops_step = 4.0 * lay.head_dim * lay.num_heads_q * visible_pairs_per_head(lay)
    ms_per_step = flops_step / (value * 1e12) * 1e3       # extrapolated from the samples
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "ms_per_step_extrapolated": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "gemma_like (same as the GPU arm); each step times the CPU oracle "
                               "on a bounded sample of its rows on every host core and scales to "
                               "TFLOP/s; ms_per_step is that rate applied to the whole step",
                   "parallelism": f"{vals[0]['cores']} single-thread processes"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": vals[0]["cores"],
                         "host_cores": vals[0]["host_cores"], "kind": "oracle",
                         "sample": f"{args.steps} samples of about {per_step:.1f} s each on "
                                   f"{vals[0]['cores']} processes ({total:.1f} s total)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads and bandwidth sweeps")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels one by one instead of replaying CUDA graphs")
    ap.add_argument("--workload", default="gemma_like",
                    choices=["gemma_like", "chunked_prefill", "chunked_prefill_d64"],
                    help="the step's layout (gemma_like = the benchmark; the chunked-prefill layouts at "
                         "head_dim 128 and 64 = profiling cases)")
    ap.add_argument("--requests", type=int, default=4, choices=[1, 2, 3, 4],
                    help="Gemma-like requests per step (4 = the benchmark; fewer = profiling case)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_gpu(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
