"""Plain CPU oracle for paged sliding-window attention with a window-clamped
multimodal (image) prefix, and for its two feeders: slot mapping and the
log-sum-exp merge of split-KV partial outputs.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA library (``paged_sliding_window_swa_gb300``) and neither imports
the other.  Everything here is slow on purpose: per-token loops, a per-pair
visibility mask over every key of the sequence (no pruning), and fp64
softmax over the bf16/fp32 inputs widened to fp64.

Sources (page title, then the section):

* "vLLM PR #53147 summary: multimodal prefix restores SWA pruning"
  (prhub.com.cn) -- "Implementation breakdown" items 1-2 (the union
  semantics of the base window and the clamped image mask), the
  ``compute_tile_loop_bounds`` excerpt (tile bounds), and the geometry tests
  (expected bounds [3, 72, 4096] and [3, 68)).
* "vllm-ascend Triton operator: _compute_slot_mapping_kernel"
  (0539edu.com) -- section 2 "non-CP path" (slot formula), section 1 (the
  PAD tail for graph-fixed shapes), section 5 (worked example).
* the same slot-mapping article, section 3 "multi-CP domains" (the
  interleaved context-parallel slot formula, steps 1-5, and the example of
  section 3.3).
* "MLA DCP decode two-stream overlap and V-up fusion (PR #16977)"
  (huashanblogllm.xyz) -- section 1.1 and the LSE glossary entry: partial
  outputs merged with their LSE are equal to one softmax over the whole
  sequence.

Readings where the pages are silent or ambiguous:

* softmax scale is an argument (default 1/sqrt(head_dim) in the workloads);
  LSE is in natural log;
* the K/V cache is slot-major ``[num_blocks, block_size, num_kv_heads, D]``,
  slot = block * block_size + offset; query head h reads kv head
  h // (num_heads_q // num_heads_kv);
* image ranges are inclusive ``[s, e]`` in absolute positions; ``s >= e`` is
  padding (the pages' test pads with [0, 0]);
* tile bounds use the block's first row for the window's left edge
  (``ctx + qpos_lo - W + 1``, or its chunk's lookback start), the block's
  last row clamped to the query length, and ``max_seq_prefix_len = seq_len``
  whenever image ranges are enabled, attention is non-causal, or the
  per-sequence causal mode is on;
* chunked lookback (CHUNK_LOOKBACK >= 0) replaces only the base window's
  left edge; the image mask keeps the ordinary window clamp; it needs
  W > 0 and a positive chunk size (the excerpt applies it only inside the
  sliding-window branch);
* per-sequence causal: a flag per sequence replaces ``causal`` in the mask;
  the tile bounds do not read the flags and bound every sequence with the
  non-causal right edge, as the excerpt does;
* split-KV: a sequence with P_s partitions gives partition p the keys
  ``[p*L, min((p+1)*L, seq_len))`` with ``L = 128 * ceil(ceil(seq_len/P_s)/128)``;
  a row with no allowed key in a partition has partial LSE = -inf;
* LSE merge: partitions with LSE = -inf carry weight 0 and their partial
  output is never read; if every partition is -inf the output is 0 and the
  merged LSE is -inf.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -math.inf
SPLIT_ALIGN = 128


# ---------------------------------------------------------------------------
# slot mapping (vllm-ascend slot-mapping article, sections 1, 2 and 5)
# ---------------------------------------------------------------------------
def slot_mapping(query_start_loc, positions, block_table, block_size, num_tokens,
                 max_num_tokens, pad_id=-1, context_lens=None):
    """Physical KV slot of every token, then ``pad_id`` over the padded tail.

    For token t of request r: block index = pos // block_size, offset =
    pos - index * block_size, slot = block_table[r][index] * block_size +
    offset.  Tokens in ``[num_tokens, max_num_tokens)`` get ``pad_id``.  A
    token whose position is negative or whose block index lies outside the
    request's block-table row is not mapped (it gets ``pad_id``); its index is
    returned in ``bad``.  With ``positions`` None, the i-th token of request r
    sits at ``context_lens[r] + i`` (its cached context followed by the new
    tokens).
    """
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    if positions is None:
        ctx = np.asarray(context_lens, dtype=np.int64)
        positions = np.zeros(int(qsl[-1]) if len(qsl) else 0, dtype=np.int64)
        for r in range(len(qsl) - 1):
            for i, t in enumerate(range(int(qsl[r]), int(qsl[r + 1]))):
                positions[t] = ctx[r] + i
    pos_arr = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    stride = bt.shape[1]
    out = [pad_id] * int(max_num_tokens)
    bad = []
    for r in range(len(qsl) - 1):
        for t in range(int(qsl[r]), int(qsl[r + 1])):
            pos = int(pos_arr[t])
            index = pos // block_size
            if pos < 0 or index >= stride:
                bad.append(t)
                continue
            offset = pos - index * block_size
            out[t] = int(bt[r, index]) * block_size + offset
    del num_tokens  # the tail is everything after the last request's tokens
    return np.array(out, dtype=np.int64).astype(np.int32), bad


def slot_mapping_cp(query_start_loc, positions, block_table, block_size, max_num_tokens,
                    kv_cache_block_size, cp_world_size, cp_rank, cp_interleave, pad_id=-1):
    """Slot of every token on one context-parallel rank (section 3.1, steps 1-5).

    Token i of a sequence lives on rank (i // I) % W (I = interleave size, W =
    world size).  A virtual block spans kv_cache_block_size * W positions;
    the segments of it that this rank owns are concatenated into local
    offsets, which index this rank's blocks:

        v_idx, v_off = divmod(pos, kv_cache_block_size * W)
        local        = (v_off // I) % W == rank
        local_off    = (v_off // (W * I)) * I + v_off % I
        block_index  = v_idx * (kv_cache_block_size // block_size) + local_off // block_size
        slot         = block_table[r][block_index] * block_size + local_off % block_size

    Tokens owned by another rank, the padded tail and unmapped tokens get
    ``pad_id``; negative positions and block indices outside the row are
    returned in ``bad``.  With W = 1, I = 1 this is ``slot_mapping``.
    """
    W, rank, I = int(cp_world_size), int(cp_rank), int(cp_interleave)
    kvb, bs = int(kv_cache_block_size), int(block_size)
    if not (W >= 1 and 0 <= rank < W and I >= 1 and bs >= 1 and kvb % bs == 0 and kvb % I == 0):
        raise ValueError("cp geometry: need W >= 1, 0 <= rank < W, block_size | kv_cache_block_size, "
                         "interleave | kv_cache_block_size")
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    pos_arr = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    stride = bt.shape[1]
    blocks_per_kv_block = kvb // bs
    out = [pad_id] * int(max_num_tokens)
    bad = []
    for r in range(len(qsl) - 1):
        for t in range(int(qsl[r]), int(qsl[r + 1])):
            pos = int(pos_arr[t])
            if pos < 0:
                bad.append(t)
                continue
            v_idx, v_off = divmod(pos, kvb * W)
            if (v_off // I) % W != rank:
                continue                          # another rank's token
            local_off = (v_off // (W * I)) * I + v_off % I
            index = v_idx * blocks_per_kv_block + local_off // bs
            if index >= stride:
                bad.append(t)
                continue
            out[t] = int(bt[r, index]) * bs + local_off % bs
    return np.array(out, dtype=np.int64).astype(np.int32), bad


# ---------------------------------------------------------------------------
# KV-cache write by slot id (vllm-ascend slot-mapping article, section 1 and
# the closing summary: the cache-write and attention operators consume slots)
# ---------------------------------------------------------------------------
def kv_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache):
    """Copies of the two caches with token t's rows stored at slot
    ``slot_mapping[t]``.

    ``k_new``/``v_new``: [T, Hkv, D]; caches: [num_blocks, block_size, Hkv, D]
    (or already slot-major [num_slots, Hkv, D]).  A negative slot (padding)
    writes nothing; a slot >= num_slots writes nothing and is returned in
    ``bad``.  Two tokens with the same slot: unspecified (the scheduler never
    repeats a slot; here the later token wins).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    shape = kc.shape
    kc = kc.reshape(-1, shape[-2], shape[-1])
    vc = vc.reshape(-1, shape[-2], shape[-1])
    slots = np.asarray(slot_mapping, dtype=np.int64)
    kn, vn = np.asarray(k_new), np.asarray(v_new)
    bad = []
    for t in range(kn.shape[0]):
        s = int(slots[t])
        if s < 0:
            continue
        if s >= kc.shape[0]:
            bad.append(t)
            continue
        kc[s] = kn[t]
        vc[s] = vn[t]
    return kc.reshape(shape), vc.reshape(shape), bad


# ---------------------------------------------------------------------------
# the visibility rule (vLLM PR #53147 summary, implementation items 1-2)
# ---------------------------------------------------------------------------
def _check_chunk(window, chunk_size, chunk_lookback):
    """Chunked lookback replaces the sliding window's left edge, so it needs a
    window and a positive chunk size ("vLLM PR #53147 summary",
    compute_tile_loop_bounds excerpt: the chunk branch sits inside the
    SLIDING_WINDOW > 0 branch; CHUNK_LOOKBACK = -1 turns it off)."""
    if chunk_lookback is None or chunk_lookback < 0:
        return False
    if window <= 0 or chunk_size is None or chunk_size <= 0:
        raise ValueError("chunk_lookback >= 0 needs window > 0 and chunk_size > 0")
    return True


def visible_keys(q_abs, seq_len, window, causal, ranges, chunk_size=0, chunk_lookback=-1):
    """Boolean mask over every key k in [0, seq_len) for the query at q_abs.

    base(q, k): for W > 0, k >= left(q) and (causal: k <= q; non-causal:
    k <= q+W-1), where left(q) = q-W+1, or with chunked lookback
    (chunk_lookback L >= 0, chunk size C) the start of the chunk L chunks
    before q's chunk, ((q // C) - L) * C.  For W <= 0, causal: k <= q,
    non-causal: every key.
    mm(q, k): some valid range [s, e] holds both q and k, and (W > 0)
    k >= q-W+1 -- the ordinary window's edge, also under chunking (the
    reviewer's note on the same page: the image mask is OR-ed after the
    chunk restriction and clamped by the ordinary window, so it can reach
    keys before the chunk boundary).
    Visible = base OR mm, for 0 <= k < seq_len.
    """
    k = np.arange(int(seq_len), dtype=np.int64)
    q = int(q_abs)
    chunked = _check_chunk(window, chunk_size, chunk_lookback)
    if window > 0:
        right = q if causal else q + window - 1
        left = q - window + 1
        if chunked:
            left = ((q // int(chunk_size)) - int(chunk_lookback)) * int(chunk_size)
        base = (k >= left) & (k <= right)
    else:
        base = (k <= q) if causal else np.ones(k.shape, dtype=bool)
    mm = np.zeros(k.shape, dtype=bool)
    if ranges is not None:
        for s, e in np.asarray(ranges).reshape(-1, 2):
            s, e = int(s), int(e)
            if not s < e:
                continue                      # [0, 0] padding / empty range
            if s <= q <= e:
                inside = (k >= s) & (k <= e)
                if window > 0:
                    inside &= k >= q - window + 1   # clamped at the window's left edge
                mm |= inside
    return base | mm


def split_key_ranges(seq_len, parts):
    """Key range of each of ``parts`` split-KV partitions (possibly empty)."""
    seq_len, parts = int(seq_len), int(parts)
    per = -(-seq_len // parts) if parts > 0 else seq_len
    length = -(-per // SPLIT_ALIGN) * SPLIT_ALIGN
    return [(min(p * length, seq_len), min((p + 1) * length, seq_len)) for p in range(parts)]


def _gather(cache, table_row, seq_len, block_size, kv_head):
    """Rows of one kv head for keys 0..seq_len-1, fetched page by page."""
    d = cache.shape[-1]
    out = np.empty((int(seq_len), d), dtype=np.float64)
    for k in range(int(seq_len)):
        page = int(table_row[k // block_size])
        out[k] = cache[page, k % block_size, kv_head]
    return out


def _as_f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, mm_ranges,
              window, causal, scale, context_lens=None, rows=None, splits_per_seq=None,
              num_splits=1, seq_causal=None, chunk_size=0, chunk_lookback=-1):
    """Attention of every requested (token, head) row, fp64.

    ``seq_causal``: None, or one flag per sequence that replaces ``causal``
    for that sequence (the per-sequence causal mode).  ``chunk_size`` /
    ``chunk_lookback``: chunked lookback, see ``visible_keys``.

    ``rows``: iterable of (token, head) pairs, or None for all rows.  Returns
    dicts keyed by (token, head): ``out`` (D-vector) and ``lse`` (float).  With
    ``num_splits > 1`` the keys are further restricted to each partition and
    the results are keyed by (split, token, head); partitions >= P_s of a
    sequence, and rows with no allowed key in a partition, give lse = -inf and
    an all-zero output.
    """
    qf = _as_f64(q)
    kc = _as_f64(k_cache)
    vc = _as_f64(v_cache)
    bt = np.asarray(block_table)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    T, Hq, D = qf.shape
    Hkv = kc.shape[2]
    G = Hq // Hkv
    B = kc.shape[1]
    S = len(seq_lens)
    ctx = (seq_lens - np.diff(qsl)) if context_lens is None else np.asarray(context_lens, np.int64)
    tok_seq = np.repeat(np.arange(S), np.diff(qsl))
    if rows is None:
        rows = [(t, h) for t in range(T) for h in range(Hq)]
    by_group = {}
    for t, h in rows:
        by_group.setdefault((int(tok_seq[t]), h // G), []).append((int(t), int(h)))
    out, lse = {}, {}
    for (s, hk), lst in sorted(by_group.items()):
        K = _gather(kc, bt[s], seq_lens[s], B, hk)
        V = _gather(vc, bt[s], seq_lens[s], B, hk)
        rng = None if mm_ranges is None else np.asarray(mm_ranges)[s]
        parts = 1
        if num_splits > 1:
            parts = int(num_splits if splits_per_seq is None else splits_per_seq[s])
        key_ranges = split_key_ranges(seq_lens[s], parts)
        for t, h in lst:
            q_abs = int(ctx[s] + (t - qsl[s]))
            c_s = causal if seq_causal is None else bool(seq_causal[s])
            vis = visible_keys(q_abs, seq_lens[s], window, c_s, rng, chunk_size, chunk_lookback)
            for p in range(num_splits if num_splits > 1 else 1):
                sel = vis.copy()
                if num_splits > 1:
                    if p >= parts:
                        sel[:] = False
                    else:
                        lo, hi = key_ranges[p]
                        sel[:lo] = False
                        sel[hi:] = False
                idx = np.nonzero(sel)[0]
                if idx.size == 0:
                    o, l = np.zeros(D), NEG_INF
                else:
                    sc = scale * (K[idx] @ qf[t, h])
                    m = sc.max()
                    w = np.exp(sc - m)
                    o = (w @ V[idx]) / w.sum()
                    l = m + math.log(w.sum())
                key = (t, h) if num_splits == 1 else (p, t, h)
                out[key], lse[key] = o, l
    return out, lse


def allowed_pair_count(query_start_loc, seq_lens, mm_ranges, window, causal, context_lens=None,
                       seq_causal=None, chunk_size=0, chunk_lookback=-1):
    """Number of visible (query, key) pairs of one head, by the per-pair rule."""
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    ctx = (seq_lens - np.diff(qsl)) if context_lens is None else np.asarray(context_lens, np.int64)
    total = 0
    for s in range(len(seq_lens)):
        rng = None if mm_ranges is None else np.asarray(mm_ranges)[s]
        c_s = causal if seq_causal is None else bool(seq_causal[s])
        for i in range(int(qsl[s + 1] - qsl[s])):
            total += int(visible_keys(ctx[s] + i, seq_lens[s], window, c_s, rng, chunk_size,
                                      chunk_lookback).sum())
    return total


# ---------------------------------------------------------------------------
# tile bounds (vLLM PR #53147 summary, compute_tile_loop_bounds excerpt)
# ---------------------------------------------------------------------------
def tile_bounds(query_start_loc, seq_lens, mm_ranges, window, causal, tile_size, block_q,
                max_qblocks, context_lens=None, per_seq_causal=False, chunk_size=0,
                chunk_lookback=-1):
    """[loop_lo, loop_hi, max_seq_prefix_len] for every (sequence, query block).

    Blocks past the sequence's query length are left as [0, 0, 0].  The base
    window's left edge is the block's first row's, q_lo - W + 1, or with
    chunked lookback the start of the chunk L chunks before q_lo's chunk,
    ((q_lo // C) - L) * C.  Its right edge is q_hi (causal) or q_hi + W - 1
    (non-causal, and always in the per-sequence causal mode, which the
    excerpt bounds as non-causal).  With an image-range array present
    (``mm_ranges`` not None), every range that intersects the block's rows
    widens it: the left edge to max(start, q_lo - W + 1), the right edge to
    the range end; the right edge is then clamped to seq_len - 1 and both
    edges are converted to tiles.
    """
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    S = len(seq_lens)
    ctx = (seq_lens - np.diff(qsl)) if context_lens is None else np.asarray(context_lens, np.int64)
    use_mm = mm_ranges is not None and np.asarray(mm_ranges).size > 0
    chunked = _check_chunk(window, chunk_size, chunk_lookback)
    right_causal = causal and not per_seq_causal
    out = np.zeros((S, max_qblocks, 3), dtype=np.int64)
    for s in range(S):
        qlen = int(qsl[s + 1] - qsl[s])
        seq_len = int(seq_lens[s])
        c = int(ctx[s])
        for b in range(max_qblocks):
            qpos_lo = b * block_q
            if qpos_lo >= qlen:
                continue
            qpos_hi = min(qpos_lo + block_q - 1, qlen - 1)
            if use_mm or not right_causal:
                max_prefix = seq_len
            else:
                max_prefix = min(c + qpos_hi + 1, seq_len)
            num_tiles = -(-max_prefix // tile_size)
            if window <= 0:
                lo, hi = 0, num_tiles
            else:
                q_lo, q_hi = c + qpos_lo, c + qpos_hi
                if chunked:
                    first = ((q_lo // int(chunk_size)) - int(chunk_lookback)) * int(chunk_size)
                else:
                    first = q_lo - window + 1
                last = q_hi if right_causal else q_hi + window - 1
                if use_mm:
                    for rs, re_ in np.asarray(mm_ranges)[s].reshape(-1, 2):
                        rs, re_ = int(rs), int(re_)
                        if rs < re_ and rs <= q_hi and re_ >= q_lo:
                            first = min(first, max(rs, q_lo - window + 1))
                            last = max(last, re_)
                last = min(last, seq_len - 1)
                lo = max(0, first // tile_size)
                hi = min(last // tile_size + 1, num_tiles)
            out[s, b] = (lo, hi, max_prefix)
    return out.astype(np.int32)


# ---------------------------------------------------------------------------
def lse_combine(partial_out, partial_lse):
    """Merge P partial outputs [P, T, H, D] with their LSE [P, T, H].

    L = max_p lse_p; w_p = exp(lse_p - L); out = sum_p w_p o_p / sum_p w_p;
    lse = L + ln(sum_p w_p).  Partitions with lse = -inf have weight 0 and
    their output is not read.  All -inf: out = 0, lse = -inf.
    """
    po = _as_f64(partial_out)
    pl = _as_f64(partial_lse)
    P, T, H, D = po.shape
    out = np.zeros((T, H, D))
    lse = np.full((T, H), NEG_INF)
    for t in range(T):
        for h in range(H):
            vals = pl[:, t, h]
            live = [p for p in range(P) if vals[p] != NEG_INF]
            if not live:
                continue
            L = max(vals[p] for p in live)
            w = {p: math.exp(vals[p] - L) for p in live}
            tot = sum(w.values())
            acc = np.zeros(D)
            for p in live:
                acc += w[p] * po[p, t, h]
            out[t, h] = acc / tot
            lse[t, h] = L + math.log(tot)
    return out, lse
