"""CPU-side checks of the C ABI library: it builds for sm_103a, loads without a
GPU, exports every symbol the header declares, and its host-side argument
checks reject bad calls before any CUDA work (these calls never reach a
kernel, so they are safe without a GPU)."""
import ctypes
import os
import re

import pytest

import paged_sliding_window_swa_gb300 as swa
from paged_sliding_window_swa_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NULL = None


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(build_lib.LIB_PATH):
        build_lib.build()
    return swa.lib()


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("swa_slot_mapping", "swa_tile_bounds", "swa_mm_paged_attention", "lse_combine"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_binding_names_match_the_abi():
    for n in ("swa_slot_mapping", "swa_tile_bounds", "swa_mm_paged_attention", "lse_combine"):
        assert callable(getattr(swa, n))


def test_version(lib):
    assert b"sm_103a" in lib.swa_version()


def test_slot_mapping_rejects_bad_sizes(lib):
    assert lib.swa_slot_mapping(NULL, NULL, NULL, NULL, 4, 16, 1, 10, 5, -1, NULL, NULL, NULL) == -2
    assert lib.swa_slot_mapping(NULL, NULL, NULL, NULL, 4, 0, 1, 10, 20, -1, NULL, NULL, NULL) == -2
    assert lib.swa_slot_mapping(NULL, NULL, NULL, NULL, 4, 16, 1, 10, 20, -1, NULL, NULL, NULL) == -1
    assert lib.swa_slot_mapping(NULL, NULL, NULL, NULL, 4, 16, 0, 0, 0, -1, NULL, NULL, NULL) == 0
    # positions or context lengths: one of the two is needed once there are tokens
    p = ctypes.c_void_p(0x1000)
    assert lib.swa_slot_mapping(p, NULL, NULL, p, 4, 16, 1, 10, 20, -1, p, NULL, NULL) == -1


def test_tile_bounds_rejects_bad_sizes(lib):
    assert lib.swa_tile_bounds(NULL, NULL, NULL, NULL, 0, 1, 64, 1, 0, 0, -1, 0, 8, 4, NULL, NULL, NULL) == -2
    assert lib.swa_tile_bounds(NULL, NULL, NULL, NULL, 0, 1, 64, 1, 0, 0, -1, 32, 8, 4, NULL, NULL, NULL) == -1
    # chunked lookback needs a window and a chunk size
    assert lib.swa_tile_bounds(NULL, NULL, NULL, NULL, 0, 1, 0, 1, 0, 16, 2, 32, 8, 4, NULL, NULL, NULL) == -2
    assert lib.swa_tile_bounds(NULL, NULL, NULL, NULL, 0, 1, 64, 1, 0, 0, 2, 32, 8, 4, NULL, NULL, NULL) == -2
    assert lib.swa_tile_bounds(NULL, NULL, NULL, NULL, 0, 1, 64, 1, 1, 16, 2, 32, 8, 4, NULL, NULL, NULL) == -1


def _attn(lib, **kw):
    args = dict(q=NULL, k=NULL, v=NULL, nb=10, bt=NULL, stride=4, qsl=NULL, seq=NULL, ctx=NULL,
                mm=NULL, R=0, S=1, T=8, mq=8, hq=8, hkv=2, d=128, b=16, w=64, causal=1, seq_causal=NULL,
                chunk_size=0, chunk_lookback=-1, scale=0.1,
                dtype=0, P=1, sps=NULL, out=NULL, lse=NULL, po=NULL, pl=NULL, err=NULL, st=NULL)
    args.update(kw)
    return lib.swa_mm_paged_attention(*args.values())


def test_attention_rejects_bad_arguments(lib):
    assert _attn(lib, hkv=3) == -2                      # Hq % Hkv != 0
    assert _attn(lib, d=96) == -3                       # head_dim not built
    assert _attn(lib, b=8) == -3                        # block size not built
    assert _attn(lib, dtype=7) == -3
    assert _attn(lib, scale=float("nan")) == -2
    assert _attn(lib, chunk_lookback=1) == -2           # chunking without a chunk size
    assert _attn(lib, chunk_lookback=0, chunk_size=64, w=0) == -2   # chunking without a window
    assert _attn(lib, chunk_lookback=0, chunk_size=64) == -1        # valid: reaches the NULL check
    assert _attn(lib) == -1                             # NULL tensors
    assert _attn(lib, T=0) == 0                         # nothing to do
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    full = dict(q=p, k=p, v=p, bt=p, qsl=p, seq=p, out=p)
    assert _attn(lib, **{**full, "q": odd}) == -4       # misaligned
    assert _attn(lib, **{**full, "P": 4}) == -1         # split mode needs partial buffers


def test_lse_combine_rejects_bad_arguments(lib):
    assert lib.lse_combine(NULL, NULL, 0, 4, 2, 128, 0, NULL, NULL, NULL) == -2
    assert lib.lse_combine(NULL, NULL, 2, 4, 2, 100, 0, NULL, NULL, NULL) == -3
    assert lib.lse_combine(NULL, NULL, 2, 4, 2, 128, 0, NULL, NULL, NULL) == -1
    p, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1008)
    assert lib.lse_combine(odd, p, 2, 4, 2, 128, 0, p, NULL, NULL) == -4


def test_product_path_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(swa, "_LIB", None)
    monkeypatch.setattr(swa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(swa.SwaError):
        swa.lib()


def test_binding_exposes_the_cache_write_and_cp_calls():
    for n in ("swa_slot_mapping_cp", "swa_kv_cache_write"):
        assert n in _declared() and callable(getattr(swa, n))


def test_slot_mapping_cp_rejects_bad_geometry(lib):
    def call(kvb=32, W=2, r=0, I=16, bs=16):
        return lib.swa_slot_mapping_cp(NULL, NULL, NULL, 4, bs, 1, 10, 20, -1, kvb, W, r, I, NULL, NULL, NULL)
    assert call(kvb=24) == -2                           # block size 16 does not divide 24
    assert call(I=12) == -2                             # interleave does not divide 32
    assert call(r=2) == -2                              # rank >= world size
    assert call(W=0) == -2
    assert call() == -1                                 # geometry fine, pointers missing
    assert lib.swa_slot_mapping_cp(NULL, NULL, NULL, 4, 16, 0, 0, 0, -1, 32, 2, 0, 16, NULL, NULL, NULL) == 0


def test_kv_cache_write_rejects_bad_arguments(lib):
    def call(T=4, hkv=2, d=128, dtype=0, nslots=64):
        return lib.swa_kv_cache_write(NULL, NULL, NULL, T, hkv, d, dtype, NULL, NULL, nslots, NULL, NULL)
    assert call(d=100) == -2                            # rows of 16-byte vectors need D % 8 == 0
    assert call(hkv=0) == -2
    assert call(dtype=5) == -3
    assert call() == -1
    assert call(T=0) == 0


def test_watchdog_rejects_out_of_range_bounds(lib):
    """The bound must be 0 (default) or within [1 us, 10 s]; a refused call changes nothing."""
    assert lib.swa_set_watchdog(999, 0) == -2
    assert lib.swa_set_watchdog(10_000_000_001, 0) == -2
    assert lib.swa_set_watchdog(1000, 0) == 0
    assert lib.swa_set_watchdog(0, 0) == 0
