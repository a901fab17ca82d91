"""Seeded synthetic inputs for paged sliding-window attention with image ranges.

This module builds batch *structure* (query/sequence/context lengths, token
positions, image ranges, paged block tables, split counts) and random q/k/v
tensors.  It is shared by the tests, the benchmark and the CPU oracle checks,
and it deliberately holds none of the method's arithmetic: no visibility mask,
no tile bounds, no slot formula, no softmax.  Every layout is drawn from a
numpy PCG64 generator seeded with ``structure_seed`` (default 0) and every
tensor from a ``torch.Generator`` seeded with ``data_seed`` (default 1).

The five named layouts follow the workloads the method is measured on:

* ``tiny``            one 256-token sequence, fp32, W=64, one image [40, 120]
* ``geometry``        one 4096-token sequence, W=1024, the tile-bounds example
* ``gemma_like``      4 requests of ~16,550 tokens with 60 images of 256 each
* ``chunked_prefill`` 8 requests, 4k-32k cached context + 2048-token chunks
* ``decode``          128 single-token queries over 4k-64k contexts, split-KV

Image ranges are inclusive ``[start, end]`` in absolute sequence positions;
``[0, 0]`` is padding.  Block-table entries that hold no page are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

try:  # torch is only needed for tensor generation
    import torch
except ImportError:  # pragma: no cover - torch is always present in this repo
    torch = None

DTYPES = ("bf16", "fp32")


@dataclass
class Layout:
    """Batch structure of one attention call (host numpy arrays)."""

    name: str
    query_lens: np.ndarray            # int32 [S]
    seq_lens: np.ndarray              # int32 [S]  (context + query)
    mm_ranges: Optional[np.ndarray]   # int32 [S, R, 2] inclusive, or None
    block_table: np.ndarray           # int32 [S, stride], -1 = no page
    num_blocks: int
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    window: int
    causal: bool
    dtype: str = "bf16"
    num_splits: int = 1
    splits_per_seq: Optional[np.ndarray] = None   # int32 [S] or None
    max_num_tokens: int = 0
    seq_causal: Optional[np.ndarray] = None       # int32 [S] per-sequence causal flags, or None
    chunk_size: int = 0                           # chunked lookback: chunk size (0 = off)
    chunk_lookback: int = -1                      # chunked lookback: chunks looked back (-1 = off)
    notes: dict = field(default_factory=dict)

    # ---- derived structure -------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(len(self.seq_lens))

    @property
    def num_tokens(self) -> int:
        return int(self.query_lens.sum())

    @property
    def query_start_loc(self) -> np.ndarray:
        qsl = np.zeros(self.num_seqs + 1, dtype=np.int32)
        qsl[1:] = np.cumsum(self.query_lens)
        return qsl

    @property
    def context_lens(self) -> np.ndarray:
        return (self.seq_lens - self.query_lens).astype(np.int32)

    @property
    def positions(self) -> np.ndarray:
        """Absolute position of every query token (context length + index)."""
        out = np.empty(self.num_tokens, dtype=np.int64)
        qsl = self.query_start_loc
        ctx = self.context_lens
        for s in range(self.num_seqs):
            out[qsl[s]:qsl[s + 1]] = ctx[s] + np.arange(self.query_lens[s], dtype=np.int64)
        return out

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    @property
    def max_mm_ranges(self) -> int:
        return 0 if self.mm_ranges is None else int(self.mm_ranges.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_heads_q // self.num_heads_kv

    def without_ranges(self) -> "Layout":
        return replace(self, name=self.name + "-noimg", mm_ranges=None)


# ---------------------------------------------------------------------------
# structure helpers
# ---------------------------------------------------------------------------
def _block_table(rng: np.random.Generator, seq_lens, block_size: int,
                 spare_blocks: int = 64, extra_stride: int = 0):
    pages = [(int(n) + block_size - 1) // block_size for n in seq_lens]
    num_blocks = sum(pages) + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    stride = max(max(pages) if pages else 0, 1) + extra_stride
    bt = np.full((len(seq_lens), stride), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[cur:cur + n]
        cur += n
    return bt, num_blocks


def _pad_ranges(per_seq, min_r: int = 1) -> np.ndarray:
    r = max(min_r, max((len(x) for x in per_seq), default=0))
    out = np.zeros((len(per_seq), r, 2), dtype=np.int32)
    for s, lst in enumerate(per_seq):
        for i, (a, b) in enumerate(lst):
            out[s, i] = (a, b)
    return out


def _place_images(rng, seq_len: int, n: int, img: int, forced=None, max_tries: int = 20000):
    """Non-overlapping ``img``-token ranges at random offsets in [0, seq_len)."""
    placed = []
    if forced is not None and n >= 1:
        placed.append(forced)
    tries = 0
    while len(placed) < n and tries < max_tries and seq_len >= img:
        tries += 1
        st = int(rng.integers(0, seq_len - img + 1))
        en = st + img - 1
        if all(en < a or st > b for a, b in placed):
            placed.append((st, en))
    return sorted(placed)


# ---------------------------------------------------------------------------
# the five named layouts
# ---------------------------------------------------------------------------
def tiny(structure_seed: int = 0) -> Layout:
    """1 x 256 tokens, causal, W=64, image [40,120], 2 q heads / 1 kv head, D=64, fp32."""
    rng = np.random.default_rng(structure_seed)
    seq = np.array([256], dtype=np.int32)
    bt, nb = _block_table(rng, seq, 16)
    return Layout("tiny", query_lens=seq.copy(), seq_lens=seq, mm_ranges=_pad_ranges([[(40, 120)]]),
                  block_table=bt, num_blocks=nb, num_heads_q=2, num_heads_kv=1, head_dim=64,
                  block_size=16, window=64, causal=True, dtype="fp32", max_num_tokens=256,
                  notes={"tile_size": 32})


def geometry(variant: str = "causal", structure_seed: int = 0) -> Layout:
    """1 x 4096 tokens, W=1024, 8 q heads / 4 kv heads, D=256, bf16, two range slots.

    variant ``causal``: image [1024, 2303] (wider than the window);
    ``noncausal``: image [1024, 1279] with the bidirectional right window;
    ``noncausal-wide``: image [1024, 2303] with the bidirectional right window.
    """
    rng = np.random.default_rng(structure_seed)
    seq = np.array([4096], dtype=np.int32)
    bt, nb = _block_table(rng, seq, 16)
    if variant == "causal":
        rngs, causal = [(1024, 2303)], True
    elif variant == "noncausal":
        rngs, causal = [(1024, 1279)], False
    elif variant == "noncausal-wide":
        rngs, causal = [(1024, 2303)], False
    else:
        raise ValueError(variant)
    mm = _pad_ranges([rngs], min_r=2)
    return Layout("geometry-" + variant, query_lens=seq.copy(), seq_lens=seq, mm_ranges=mm,
                  block_table=bt, num_blocks=nb, num_heads_q=8, num_heads_kv=4, head_dim=256,
                  block_size=16, window=1024, causal=causal, dtype="bf16", max_num_tokens=4096,
                  notes={"tile_size": 32, "block_q": 8})


def gemma_like(structure_seed: int = 0, num_requests: int = 4) -> Layout:
    """4 requests (16550, 16294, 16806, 16550 tokens), 60 images of 256 tokens each.

    Text spans between images are a seeded random composition of the remaining
    text tokens into 61 gaps of at least one token.  Causal, W=1024, 16 q heads
    / 8 kv heads, D=256, bf16, block size 16; slot mapping pads to a multiple of
    8192 tokens.  ``num_requests < 4`` keeps the first requests only (a smaller
    case of the same structure, for profiling).
    """
    rng = np.random.default_rng(structure_seed)
    lens = np.array([16550, 16294, 16806, 16550], dtype=np.int32)[:num_requests]
    n_img, img = 60, 256
    per_seq = []
    for n in lens:
        text = int(n) - n_img * img
        cuts = np.sort(rng.choice(np.arange(1, text), size=n_img, replace=False))
        gaps = np.diff(np.concatenate([[0], cuts, [text]]))
        ranges, pos = [], 0
        for i in range(n_img):
            pos += int(gaps[i])
            ranges.append((pos, pos + img - 1))
            pos += img
        per_seq.append(ranges)
    bt, nb = _block_table(rng, lens, 16)
    t = int(lens.sum())
    name = "gemma_like" if num_requests == 4 else f"gemma_like_{num_requests}req"
    return Layout(name, query_lens=lens.copy(), seq_lens=lens, mm_ranges=_pad_ranges(per_seq),
                  block_table=bt, num_blocks=nb, num_heads_q=16, num_heads_kv=8, head_dim=256,
                  block_size=16, window=1024, causal=True, dtype="bf16",
                  max_num_tokens=-(-t // 8192) * 8192)


def chunked_prefill(causal: bool = True, structure_seed: int = 0) -> Layout:
    """8 requests: context U[4096, 32768] + 2048-token chunk, 0-40 images of 256.

    In every request with at least one image, one image is forced to straddle
    the chunk boundary ([ctx-128, ctx+127]).  W=1024, 32 q heads / 8 kv heads,
    D=128, bf16, block size 16.
    """
    rng = np.random.default_rng(structure_seed)
    ctx = rng.integers(4096, 32768 + 1, size=8).astype(np.int32)
    qlen = np.full(8, 2048, dtype=np.int32)
    seq = ctx + qlen
    per_seq = []
    for s in range(8):
        n = int(rng.integers(0, 41))
        forced = (int(ctx[s]) - 128, int(ctx[s]) + 127)
        per_seq.append(_place_images(rng, int(seq[s]), n, 256, forced=forced))
    bt, nb = _block_table(rng, seq, 16)
    t = int(qlen.sum())
    return Layout("chunked_prefill-" + ("causal" if causal else "noncausal"), query_lens=qlen,
                  seq_lens=seq.astype(np.int32), mm_ranges=_pad_ranges(per_seq), block_table=bt,
                  num_blocks=nb, num_heads_q=32, num_heads_kv=8, head_dim=128, block_size=16,
                  window=1024, causal=causal, dtype="bf16", max_num_tokens=t)


def decode(structure_seed: int = 0, num_seqs: int = 128) -> Layout:
    """128 single-token queries, context U[4096, 65536], full attention, split-KV.

    Each sequence uses clamp(ceil(ctx / 2048), 8, 32) partitions of a 32-slot
    partial buffer.  32 q heads / 8 kv heads, D=128, bf16, block size 16.
    """
    rng = np.random.default_rng(structure_seed)
    ctx = rng.integers(4096, 65536 + 1, size=num_seqs).astype(np.int32)
    qlen = np.ones(num_seqs, dtype=np.int32)
    seq = (ctx + qlen).astype(np.int32)
    bt, nb = _block_table(rng, seq, 16)
    sps = np.clip(-(-ctx // 2048), 8, 32).astype(np.int32)
    return Layout("decode", query_lens=qlen, seq_lens=seq, mm_ranges=None, block_table=bt,
                  num_blocks=nb, num_heads_q=32, num_heads_kv=8, head_dim=128, block_size=16,
                  window=0, causal=True, dtype="bf16", num_splits=32, splits_per_seq=sps,
                  max_num_tokens=num_seqs)


def random_small(seed: int, *, head_dim=None, block_size=None, dtype=None, group=None,
                 max_seqs: int = 4, max_ctx: int = 600, max_q: int = 300,
                 window=None, causal=None, with_ranges=None, num_splits: int = 1) -> Layout:
    """A random small batch for parity sweeps (ragged lengths, empty queries allowed)."""
    rng = np.random.default_rng(1000 + seed)
    S = int(rng.integers(1, max_seqs + 1))
    D = head_dim or int(rng.choice([64, 128, 256]))
    B = block_size or int(rng.choice([16, 32, 64, 128]))
    G = group or int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2]))
    qlen = rng.integers(0, max_q + 1, size=S).astype(np.int32)
    if qlen.sum() == 0:
        qlen[0] = 1
    ctx = rng.integers(0, max_ctx + 1, size=S).astype(np.int32)
    seq = (ctx + qlen).astype(np.int32)
    W = window if window is not None else int(rng.choice([0, 1, 7, 64, 200, 100000]))
    c = causal if causal is not None else bool(rng.integers(0, 2))
    wr = with_ranges if with_ranges is not None else bool(rng.integers(0, 4))
    mm = None
    if wr:
        per = []
        for s in range(S):
            n = int(rng.integers(0, 5))
            lst = []
            for _ in range(n):
                if seq[s] < 2:
                    break
                a = int(rng.integers(0, seq[s] - 1))
                b = int(rng.integers(a, min(seq[s], a + 300)))
                lst.append((a, b))        # may overlap, may be a 1-token [a, a]
            per.append(lst)
        mm = _pad_ranges(per, min_r=int(rng.integers(1, 6)))
    bt, nb = _block_table(rng, seq, B, spare_blocks=int(rng.integers(0, 9)),
                          extra_stride=int(rng.integers(0, 3)))
    sps = None
    if num_splits > 1:
        sps = rng.integers(1, num_splits + 1, size=S).astype(np.int32)
    return Layout(f"random{seed}", query_lens=qlen, seq_lens=seq, mm_ranges=mm, block_table=bt,
                  num_blocks=nb, num_heads_q=G * Hkv, num_heads_kv=Hkv, head_dim=D, block_size=B,
                  window=W, causal=c, dtype=dtype or "bf16", num_splits=num_splits,
                  splits_per_seq=sps, max_num_tokens=int(qlen.sum()) + int(rng.integers(0, 40)))


NAMED = {
    "tiny": tiny,
    "geometry": geometry,
    "gemma_like": gemma_like,
    "chunked_prefill": chunked_prefill,
    "decode": decode,
}


# ---------------------------------------------------------------------------
# tensors
# ---------------------------------------------------------------------------
def _torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _fill_randn(t, gen, chunk: int = 1 << 26):
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n].copy_(torch.randn(n, generator=gen, device=t.device, dtype=torch.float32))
    return t


def make_tensors(layout: Layout, device="cpu", data_seed: int = 1, poison_unused: bool = False):
    """q [T, Hq, D] and paged k/v caches [num_blocks, block_size, Hkv, D], N(0,1).

    With ``poison_unused`` every cache row that holds no token of any sequence
    (spare blocks and the tail of each sequence's last page) is set to NaN, so a
    kernel that lets an unused row reach its output shows NaN.
    """
    dt = _torch_dtype(layout.dtype)
    gen = torch.Generator(device=device)
    gen.manual_seed(data_seed)
    T, Hq, Hkv, D, B = (layout.num_tokens, layout.num_heads_q, layout.num_heads_kv,
                        layout.head_dim, layout.block_size)
    q = _fill_randn(torch.empty((T, Hq, D), dtype=dt, device=device), gen)
    k = _fill_randn(torch.empty((layout.num_blocks, B, Hkv, D), dtype=dt, device=device), gen)
    v = _fill_randn(torch.empty((layout.num_blocks, B, Hkv, D), dtype=dt, device=device), gen)
    if poison_unused:
        used = np.zeros(layout.num_blocks, dtype=bool)
        for s in range(layout.num_seqs):
            n = int(layout.seq_lens[s])
            pages = (n + B - 1) // B
            row = layout.block_table[s, :pages]
            used[row] = True
            if pages and n % B:
                k[int(row[-1]), n % B:] = float("nan")
                v[int(row[-1]), n % B:] = float("nan")
        spare = torch.from_numpy(np.nonzero(~used)[0]).to(device)
        if spare.numel():
            k[spare] = float("nan")
            v[spare] = float("nan")
    return q, k, v


def device_layout(layout: Layout, device):
    """The integer structure arrays of ``layout`` as torch tensors on ``device``."""
    as_t = lambda a, dt=torch.int32: torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)
    out = {
        "query_start_loc": as_t(layout.query_start_loc),
        "seq_lens": as_t(layout.seq_lens),
        "context_lens": as_t(layout.context_lens),
        "positions": as_t(layout.positions, torch.int64),
        "block_table": as_t(layout.block_table),
        "mm_ranges": None if layout.mm_ranges is None else as_t(layout.mm_ranges),
        "splits_per_seq": None if layout.splits_per_seq is None else as_t(layout.splits_per_seq),
        "seq_causal": None if layout.seq_causal is None else as_t(layout.seq_causal),
    }
    return out
