"""Python binding of the GB300 paged sliding-window attention library.

A thin ctypes layer over the C ABI in ``include/swa.h``: it checks tensor
devices, dtypes and contiguity, allocates outputs with torch (device memory
only) and passes raw pointers plus the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no Python or CPU
fallback -- if the shared library is missing, every call raises.

Entry points (same names as the C ABI):

* ``swa_slot_mapping``       token position -> physical KV slot, PAD tail
* ``swa_tile_bounds``        pruned KV-tile loop range per query block
* ``swa_mm_paged_attention`` paged attention, SWA + window-clamped image mask
* ``lse_combine``            merge of split-KV partials by their LSE
* ``swa_mm_paged_attention_split_static``  split-KV attention and merge with
  the partials in a library-owned array, for callers that cannot allocate
* ``swa_set_watchdog``       bound of the tensor-core kernels' pipeline waits,
  and a switch that makes them run out (failure-detection tests)
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build_lib import LIB_PATH

__all__ = ["swa_slot_mapping", "swa_slot_mapping_cp", "swa_kv_cache_write", "swa_tile_bounds",
           "swa_mm_paged_attention", "lse_combine", "swa_mm_paged_attention_split_static", "swa_set_watchdog",
           "lib", "SwaError", "DTYPE_BF16", "DTYPE_FP32", "ERR_BITS"]

DTYPE_BF16 = 0
DTYPE_FP32 = 1
SPLIT_ALIGN = 128
_RC = {-1: "SWA_E_NULL", -2: "SWA_E_SIZE", -3: "SWA_E_UNSUPPORTED", -4: "SWA_E_ALIGN", -5: "SWA_E_CUDA", -6: "SWA_E_SCRATCH"}
ERR_BITS = {0x01: "BLOCK_ID", 0x02: "POSITION", 0x04: "QSL", 0x08: "LENS", 0x10: "TIMEOUT", 0x20: "SPLITS",
            0x40: "INTERNAL", 0x80: "SLOT"}

_c_i32, _c_i64, _c_f, _c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_SIGS = {
    "swa_slot_mapping": [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i64, _c_i64, _c_i32, _c_p, _c_p,
                         _c_p],
    "swa_slot_mapping_cp": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i64, _c_i64, _c_i32, _c_i32, _c_i32,
                            _c_i32, _c_i32, _c_p, _c_p, _c_p],
    "swa_kv_cache_write": [_c_p, _c_p, _c_p, _c_i64, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_i64, _c_p, _c_p],
    "swa_tile_bounds": [_c_p, _c_p, _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                        _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_p],
    "swa_mm_paged_attention": [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_i32,
                               _c_i32, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                               _c_p, _c_i32, _c_i32, _c_f, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_p,
                               _c_p, _c_p],
    "lse_combine": [_c_p, _c_p, _c_i32, _c_i64, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_p],
    "swa_mm_paged_attention_split_static": [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p,
                                            _c_i32, _c_i32, _c_i64, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                            _c_i32, _c_i32, _c_p, _c_i32, _c_i32, _c_f, _c_i32, _c_i32, _c_p,
                                            _c_p, _c_p, _c_p, _c_p],
}
# Bytes of the library-owned array behind swa_mm_paged_attention_split_static.
STATIC_SCRATCH_BYTES = 16 << 20
EXPORTED = tuple(_SIGS) + ("swa_version", "swa_set_watchdog")


class SwaError(RuntimeError):
    pass


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise SwaError(f"{LIB_PATH} is missing: build it with "
                           "`python -m paged_sliding_window_swa_gb300.build_lib` (needs nvcc)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        handle.swa_version.restype = ctypes.c_char_p
        handle.swa_version.argtypes = []
        handle.swa_set_watchdog.restype = ctypes.c_int
        handle.swa_set_watchdog.argtypes = [ctypes.c_uint64, ctypes.c_int32]
        _LIB = handle
    return _LIB


def _check(rc: int, name: str):
    if rc != 0:
        raise SwaError(f"{name} returned {rc} ({_RC.get(rc, 'unknown')})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise SwaError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise SwaError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise SwaError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise SwaError(f"unsupported dtype {t.dtype}")


def swa_slot_mapping(query_start_loc, positions, block_table, block_size: int, max_num_tokens: int,
                     *, context_lens=None, num_tokens=None, pad_id: int = -1, out=None, err=None,
                     stream=None):
    """int32 slots [max_num_tokens]; see ``swa_slot_mapping`` in include/swa.h.

    ``positions`` None: token i of request r sits at ``context_lens[r] + i``;
    ``num_tokens`` must then be given (no device read is made to find it)."""
    _dev(query_start_loc, "query_start_loc", torch.int32)
    _dev(positions, "positions", torch.int64)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    if positions is None:
        if context_lens is None or num_tokens is None:
            raise SwaError("swa_slot_mapping: without positions, context_lens and num_tokens are required")
    else:
        num_tokens = positions.numel()
    if out is None:
        out = torch.empty(max_num_tokens, dtype=torch.int32, device=block_table.device)
    _dev(out, "out", torch.int32)
    _dev(err, "err", torch.int32)
    rc = lib().swa_slot_mapping(_ptr(query_start_loc), _ptr(positions), _ptr(context_lens), _ptr(block_table),
                                block_table.shape[1], block_size, query_start_loc.numel() - 1,
                                int(num_tokens), max_num_tokens, pad_id, _ptr(out), _ptr(err),
                                _stream(stream))
    _check(rc, "swa_slot_mapping")
    return out


def swa_slot_mapping_cp(query_start_loc, positions, block_table, block_size: int, max_num_tokens: int, *,
                        kv_cache_block_size: int, cp_world_size: int, cp_rank: int, cp_interleave: int,
                        pad_id: int = -1, out=None, err=None, stream=None):
    """int32 slots [max_num_tokens] on one context-parallel rank; see ``swa_slot_mapping_cp``."""
    _dev(query_start_loc, "query_start_loc", torch.int32)
    _dev(positions, "positions", torch.int64)
    _dev(block_table, "block_table", torch.int32)
    if out is None:
        out = torch.empty(max_num_tokens, dtype=torch.int32, device=positions.device)
    _dev(out, "out", torch.int32)
    _dev(err, "err", torch.int32)
    rc = lib().swa_slot_mapping_cp(_ptr(query_start_loc), _ptr(positions), _ptr(block_table),
                                   block_table.shape[1], block_size, query_start_loc.numel() - 1,
                                   positions.numel(), max_num_tokens, pad_id, kv_cache_block_size,
                                   cp_world_size, cp_rank, cp_interleave, _ptr(out), _ptr(err), _stream(stream))
    _check(rc, "swa_slot_mapping_cp")
    return out


def swa_kv_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, *, err=None, stream=None):
    """Store rows t of ``k_new``/``v_new`` [T, Hkv, D] at slots ``slot_mapping[t]`` of the
    [num_blocks, block_size, Hkv, D] caches (in place); see ``swa_kv_cache_write``."""
    _dev(k_new, "k_new")
    code = _dtype_code(k_new)
    _dev(v_new, "v_new", k_new.dtype)
    _dev(k_cache, "k_cache", k_new.dtype)
    _dev(v_cache, "v_cache", k_new.dtype)
    _dev(slot_mapping, "slot_mapping", torch.int32)
    _dev(err, "err", torch.int32)
    T, Hkv, D = k_new.shape
    if tuple(v_new.shape) != (T, Hkv, D) or k_cache.shape[-2:] != (Hkv, D) or v_cache.shape != k_cache.shape:
        raise SwaError("swa_kv_cache_write: shape mismatch")
    if slot_mapping.numel() < T:
        raise SwaError("swa_kv_cache_write: slot_mapping shorter than the token count")
    num_slots = k_cache.numel() // (Hkv * D)
    rc = lib().swa_kv_cache_write(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, Hkv, D, code,
                                  _ptr(k_cache), _ptr(v_cache), num_slots, _ptr(err), _stream(stream))
    _check(rc, "swa_kv_cache_write")
    return k_cache, v_cache


def swa_tile_bounds(query_start_loc, seq_lens, *, context_lens=None, mm_ranges=None, window: int,
                    causal: bool, tile_size: int, block_q: int, max_qblocks_per_seq: int,
                    per_seq_causal: bool = False, chunk_size: int = 0, chunk_lookback: int = -1, out=None,
                    err=None, stream=None):
    """int32 [num_seqs, max_qblocks_per_seq, 3] = {lo, hi, max_seq_prefix_len}."""
    _dev(query_start_loc, "query_start_loc", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(mm_ranges, "mm_ranges", torch.int32)
    S = seq_lens.numel()
    if out is None:
        out = torch.empty((S, max_qblocks_per_seq, 3), dtype=torch.int32, device=seq_lens.device)
    _dev(out, "out", torch.int32)
    _dev(err, "err", torch.int32)
    R = 0 if mm_ranges is None else mm_ranges.shape[1]
    rc = lib().swa_tile_bounds(_ptr(query_start_loc), _ptr(seq_lens), _ptr(context_lens), _ptr(mm_ranges),
                               R, S, window, int(bool(causal)), int(bool(per_seq_causal)), int(chunk_size),
                               int(chunk_lookback), tile_size, block_q, max_qblocks_per_seq,
                               _ptr(out), _ptr(err), _stream(stream))
    _check(rc, "swa_tile_bounds")
    return out


def swa_mm_paged_attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, *,
                           context_lens=None, mm_ranges=None, max_query_len=None, window: int,
                           causal: bool, scale: float, seq_causal=None, chunk_size: int = 0,
                           chunk_lookback: int = -1, num_splits: int = 1, splits_per_seq=None,
                           out=None, lse=None, return_lse: bool = True, partial_out=None,
                           partial_lse=None, err=None, stream=None):
    """Paged attention; returns (out, lse) or, with num_splits > 1, (partial_out, partial_lse)."""
    _dev(q, "q")
    code = _dtype_code(q)
    _dev(k_cache, "k_cache", q.dtype)
    _dev(v_cache, "v_cache", q.dtype)
    for name, t in (("block_table", block_table), ("query_start_loc", query_start_loc),
                    ("seq_lens", seq_lens), ("context_lens", context_lens), ("mm_ranges", mm_ranges),
                    ("splits_per_seq", splits_per_seq), ("seq_causal", seq_causal), ("err", err)):
        _dev(t, name, torch.int32)
    T, Hq, D = q.shape
    num_blocks, B, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise SwaError("k/v cache shapes do not match q")
    S = seq_lens.numel()
    R = 0 if mm_ranges is None else mm_ranges.shape[1]
    if max_query_len is None:
        max_query_len = T
    if num_splits > 1:
        if partial_out is None:
            partial_out = torch.empty((num_splits, T, Hq, D), dtype=q.dtype, device=q.device)
        if partial_lse is None:
            partial_lse = torch.empty((num_splits, T, Hq), dtype=torch.float32, device=q.device)
        _dev(partial_out, "partial_out", q.dtype)
        _dev(partial_lse, "partial_lse", torch.float32)
    else:
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
        _dev(out, "out", q.dtype)
        _dev(lse, "lse", torch.float32)
    rc = lib().swa_mm_paged_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table), block_table.shape[1],
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(context_lens), _ptr(mm_ranges), R, S, T,
        int(max_query_len), Hq, Hkv, D, B, int(window), int(bool(causal)), _ptr(seq_causal),
        int(chunk_size), int(chunk_lookback), float(scale), code,
        int(num_splits), _ptr(splits_per_seq), _ptr(out), _ptr(lse), _ptr(partial_out),
        _ptr(partial_lse), _ptr(err), _stream(stream))
    _check(rc, "swa_mm_paged_attention")
    if num_splits > 1:
        return partial_out, partial_lse
    return out, lse


def lse_combine(partial_out, partial_lse, *, out=None, out_lse=None, return_lse: bool = True,
                stream=None):
    """Merge [P, T, H, D] partials with their [P, T, H] LSE into (out, lse)."""
    _dev(partial_out, "partial_out")
    code = _dtype_code(partial_out)
    _dev(partial_lse, "partial_lse", torch.float32)
    P, T, H, D = partial_out.shape
    if out is None:
        out = torch.empty((T, H, D), dtype=partial_out.dtype, device=partial_out.device)
    if out_lse is None and return_lse:
        out_lse = torch.empty((T, H), dtype=torch.float32, device=partial_out.device)
    _dev(out, "out", partial_out.dtype)
    _dev(out_lse, "out_lse", torch.float32)
    rc = lib().lse_combine(_ptr(partial_out), _ptr(partial_lse), P, T, H, D, code, _ptr(out),
                           _ptr(out_lse), _stream(stream))
    _check(rc, "lse_combine")
    return out, out_lse


def swa_mm_paged_attention_split_static(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, *,
                                        context_lens=None, mm_ranges=None, max_query_len=None,
                                        window: int, causal: bool, scale: float, seq_causal=None,
                                        chunk_size: int = 0, chunk_lookback: int = -1, num_splits: int,
                                        splits_per_seq=None, out=None, lse=None, return_lse: bool = True,
                                        err=None, stream=None):
    """Split-KV attention merged by LSE in one call that allocates no device
    memory: the partials live in the library's fixed array, so the caller
    passes (or here, torch allocates) only ``out`` and ``lse``.  Calls that
    overlap on the GPU share that array and race; returns (out, lse)."""
    _dev(q, "q")
    code = _dtype_code(q)
    _dev(k_cache, "k_cache", q.dtype)
    _dev(v_cache, "v_cache", q.dtype)
    for name, t in (("block_table", block_table), ("query_start_loc", query_start_loc),
                    ("seq_lens", seq_lens), ("context_lens", context_lens), ("mm_ranges", mm_ranges),
                    ("splits_per_seq", splits_per_seq), ("seq_causal", seq_causal), ("err", err)):
        _dev(t, name, torch.int32)
    T, Hq, D = q.shape
    num_blocks, B, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise SwaError("k/v cache shapes do not match q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    _dev(out, "out", q.dtype)
    _dev(lse, "lse", torch.float32)
    rc = lib().swa_mm_paged_attention_split_static(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, _ptr(block_table), block_table.shape[1],
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(context_lens), _ptr(mm_ranges),
        0 if mm_ranges is None else mm_ranges.shape[1], seq_lens.numel(), T,
        int(T if max_query_len is None else max_query_len), Hq, Hkv, D, B, int(window), int(bool(causal)),
        _ptr(seq_causal), int(chunk_size), int(chunk_lookback), float(scale), code, int(num_splits),
        _ptr(splits_per_seq), _ptr(out), _ptr(lse), _ptr(err), _stream(stream))
    _check(rc, "swa_mm_paged_attention_split_static")
    return out, lse


def swa_set_watchdog(wait_limit_ns: int = 0, stall: bool = False):
    """Bound of every pipeline wait in the tensor-core attention kernels for
    later calls (0 = the default 200 ms) and, with ``stall``, a wait that can
    only run out, so those calls report SWA_ERR_TIMEOUT.  Process-wide."""
    _check(lib().swa_set_watchdog(int(wait_limit_ns), int(bool(stall))), "swa_set_watchdog")
