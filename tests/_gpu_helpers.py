"""Helpers for the GPU parity tests: run the library on a layout, cut a
sequence out of a big batch as a small oracle problem, and compare rows."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import torch

import paged_sliding_window_swa_gb300 as swa
import workloads as W
from oracle import swa_oracle as O

BF16_ATOL = 2e-2      # max-abs bar for bf16 inputs with fp32 accumulation
FP32_ATOL = 2e-3
LSE_ATOL = 5e-3


def atol_for(lay):
    return BF16_ATOL if lay.dtype == "bf16" else FP32_ATOL


def gpu_inputs(lay, data_seed=1, poison=False):
    dev = torch.device("cuda")
    q, k, v = W.make_tensors(lay, device=dev, data_seed=data_seed, poison_unused=poison)
    return q, k, v, W.device_layout(lay, dev)


def run_attention(lay, q, k, v, d, err=None, num_splits=None, mm=True):
    P = lay.num_splits if num_splits is None else num_splits
    return swa.swa_mm_paged_attention(
        q, k, v, d["block_table"], d["query_start_loc"], d["seq_lens"],
        context_lens=d["context_lens"], mm_ranges=d["mm_ranges"] if mm else None,
        max_query_len=lay.max_query_len, window=lay.window, causal=lay.causal, scale=lay.scale,
        seq_causal=d.get("seq_causal"), chunk_size=lay.chunk_size, chunk_lookback=lay.chunk_lookback,
        num_splits=P, splits_per_seq=d["splits_per_seq"] if P > 1 else None, err=err)


def subproblem(lay, q, k, v, s):
    """Sequence s alone, with its pages copied to the host and renumbered."""
    B = lay.block_size
    n = int(lay.seq_lens[s])
    npages = -(-n // B)
    pages = torch.as_tensor(lay.block_table[s, :npages].astype(np.int64), device=k.device)
    qsl = lay.query_start_loc
    q_s = q[int(qsl[s]):int(qsl[s + 1])].cpu()
    k_s, v_s = k[pages].cpu(), v[pages].cpu()
    lay_s = replace(lay, name=f"{lay.name}-seq{s}", query_lens=lay.query_lens[s:s + 1].copy(),
                    seq_lens=lay.seq_lens[s:s + 1].copy(),
                    mm_ranges=None if lay.mm_ranges is None else lay.mm_ranges[s:s + 1].copy(),
                    block_table=np.arange(max(npages, 1), dtype=np.int32)[None],
                    num_blocks=npages,
                    splits_per_seq=None if lay.splits_per_seq is None else lay.splits_per_seq[s:s + 1].copy(),
                    seq_causal=None if lay.seq_causal is None else lay.seq_causal[s:s + 1].copy())
    return lay_s, q_s, k_s, v_s


def oracle_rows(lay, q, k, v, rows, mm=True, num_splits=1):
    """Oracle (out, lse) for global (token, head) rows, one sequence at a time."""
    qsl = lay.query_start_loc
    tok_seq = np.repeat(np.arange(lay.num_seqs), lay.query_lens)
    by_seq = {}
    for t, h in rows:
        by_seq.setdefault(int(tok_seq[t]), []).append((int(t), int(h)))
    out, lse = {}, {}
    for s, lst in by_seq.items():
        lay_s, q_s, k_s, v_s = subproblem(lay, q, k, v, s)
        local = [(t - int(qsl[s]), h) for t, h in lst]
        o, l = O.attention(q_s, k_s, v_s, lay_s.block_table, lay_s.query_start_loc, lay_s.seq_lens,
                           lay_s.mm_ranges if mm else None, lay.window, lay.causal, lay.scale,
                           rows=local, num_splits=num_splits, splits_per_seq=lay_s.splits_per_seq,
                           seq_causal=lay_s.seq_causal, chunk_size=lay.chunk_size,
                           chunk_lookback=lay.chunk_lookback)
        for key, val in o.items():
            if num_splits > 1:
                p, tl, h = key
                gk = (p, tl + int(qsl[s]), h)
            else:
                tl, h = key
                gk = (tl + int(qsl[s]), h)
            out[gk] = val
            lse[gk] = l[key]
    return out, lse


def sample_rows(lay, n, seed=0, extra_tokens=()):
    rng = np.random.default_rng(seed)
    T, H = lay.num_tokens, lay.num_heads_q
    rows = {(int(t), int(h)) for t, h in zip(rng.integers(0, T, n), rng.integers(0, H, n))}
    qsl = lay.query_start_loc
    for s in range(lay.num_seqs):        # first / last token of every sequence, every head
        for t in (int(qsl[s]), int(qsl[s + 1]) - 1):
            if qsl[s] < qsl[s + 1]:
                rows |= {(t, h) for h in range(H)}
    for t in extra_tokens:
        rows |= {(int(t), h) for h in range(H)}
    return sorted(rows)


def max_errors(out, lse, ref_out, ref_lse, rows):
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy() if lse is not None else None
    e_out = max(float(np.abs(o[t, h] - ref_out[(t, h)]).max()) for t, h in rows)
    e_lse = 0.0 if l is None else max(abs(float(l[t, h]) - ref_lse[(t, h)]) for t, h in rows)
    return e_out, e_lse
