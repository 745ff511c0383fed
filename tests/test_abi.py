"""The C-ABI library loads, exports every declared symbol, and validates
arguments on the host (no compute call; runs without a GPU)."""

import ctypes
import os
import re

import pytest

from sparse_long_context_locks_gb300 import build as B
from sparse_long_context_locks_gb300 import locks as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "locks.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(locks_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) <= set(L._SIGS), "binding misses a declared entry point"


def test_device_accessible_refuses_null_and_pageable_host_memory(lib):
    assert lib.locks_device_accessible(None) == 0
    buf = ctypes.create_string_buffer(4096)      # pageable host memory
    assert lib.locks_device_accessible(ctypes.addressof(buf)) == 0


def test_sizes_and_status_strings(lib):
    assert L.locks_summary_bytes(8) == 784
    # unquantised fp32 records: mu, V (128 x r), C (16 x r), tail + pad
    for r in (1, 8, 16):
        assert L.locks_summary_bytes(8, quant=0, rank=r) == 4 * (128 + 128 * r + 16 * r + 4)
        assert L.record_bytes(0, r) == L.locks_summary_bytes(8, quant=0, rank=r)
    cfg_bad = L.locks_cfg(128, 16, 8, 8, 3, 1)   # G = 3 unsupported
    assert lib.locks_summary_bytes(ctypes.byref(cfg_bad)) == 0
    small = L.locks_workspace_bytes(8, 1, 257, 16)
    big = L.locks_workspace_bytes(8, 1, 8193, 128)
    assert 0 < small < big
    assert L.locks_workspace_bytes(8, 64, 16385, 128) > big
    for s in range(6):
        assert L.locks_status_str(s)


def test_host_validation_rejects_before_launch(lib):
    cfg = L.make_cfg(8)
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: validation fails first
    misaligned = ctypes.c_void_p(0x10001)
    # unsupported shapes
    for bad in (L.locks_cfg(64, 16, 8, 8, 4, 1), L.locks_cfg(128, 32, 8, 8, 4, 1),
                L.locks_cfg(128, 16, 4, 8, 4, 1), L.locks_cfg(128, 16, 17, 8, 4, 0),
                L.locks_cfg(128, 16, 0, 8, 4, 0), L.locks_cfg(128, 16, 8, 8, 4, 2),
                L.locks_cfg(128, 16, 8, 3, 4, 1), L.locks_cfg(128, 16, 8, 12, 4, 1)):
        assert lib.locks_score(ctypes.byref(bad), fake, fake, 10, fake, fake, 1, 4, None, fake,
                               1 << 20, None) == UNSUPPORTED
    # null / misaligned pointers
    assert lib.locks_build_summaries(ctypes.byref(cfg), None, 10, fake, 4, fake, None, 0, None) == INVALID
    assert lib.locks_build_summaries(ctypes.byref(cfg), misaligned, 10, fake, 4, fake, None, 0, None) == INVALID
    assert lib.locks_score(ctypes.byref(cfg), fake, None, 10, fake, fake, 1, 4, None, fake, 1 << 20, None) == INVALID
    assert lib.locks_select(ctypes.byref(cfg), fake, 1, 4, 2, None, None, fake, fake, 1 << 20, None) == INVALID
    # negative sizes, bad scale
    assert lib.locks_score(ctypes.byref(cfg), fake, fake, 10, fake, fake, -1, 4, None, fake, 1 << 20, None) == INVALID
    assert lib.locks_select(ctypes.byref(cfg), fake, 1, 4, -2, None, fake, fake, fake, 1 << 20, None) == INVALID
    assert lib.locks_sparse_decode(ctypes.byref(cfg), fake, fake, fake, 10, fake, fake, fake, fake, 1, 4,
                                   2, ctypes.c_float(-1.0), fake, fake, 1 << 20, None) == INVALID
    # workspace too small
    need = L.locks_workspace_bytes(8, 1, 4, 2)
    assert lib.locks_score(ctypes.byref(cfg), fake, fake, 10, fake, fake, 1, 4, None, fake, need - 1, None) == WORKSPACE
    assert lib.locks_sparse_decode(ctypes.byref(cfg), fake, fake, fake, 10, fake, fake, fake, fake, 1, 4,
                                   2, ctypes.c_float(0.088), fake, fake, need - 1, None) == WORKSPACE
    assert lib.locks_dense_decode(ctypes.byref(cfg), fake, fake, fake, 10, fake, fake, 1, 4,
                                  ctypes.c_float(0.088), fake, fake, need - 1, None) == WORKSPACE
    # empty batch is a no-op
    assert lib.locks_score(ctypes.byref(cfg), fake, fake, 10, fake, fake, 0, 4, None, fake, 0, None) == OK
    # read_status needs a workspace
    v = ctypes.c_uint32(0)
    assert lib.locks_read_status(None, ctypes.byref(v), None) == INVALID


def test_noalloc_validates_like_the_workspace_entry_point_before_any_cuda_call(lib):
    """The allocation-free entry point shares the workspace path's
    configuration check and split plan, and rejects a batch whose partial
    states exceed its fixed 8 MiB scratch before making any CUDA call (so this
    runs without a GPU)."""
    fake = ctypes.c_void_p(0x10000)
    scale = ctypes.c_float(0.088)

    def call(cfg, batch, budget=128):
        return lib.locks_sparse_decode_noalloc(ctypes.byref(cfg), fake, fake, fake, 10, fake, fake, fake,
                                               fake, batch, 8, budget, scale, fake, None)

    # KV-head counts the scorer's head grouping cannot tile are rejected by
    # both entry points
    for H in (3, 12):
        bad = L.locks_cfg(128, 16, 8, H, 4, 1)
        assert call(bad, 1) == UNSUPPORTED
        assert lib.locks_sparse_decode(ctypes.byref(bad), fake, fake, fake, 10, fake, fake, fake, fake, 1,
                                       8, 2, scale, fake, fake, 1 << 20, None) == UNSUPPORTED
    # 4025 (request, KV head) units fit, 4026 do not: the limit in locks.h
    assert call(L.make_cfg(1), 4026) == WORKSPACE
    assert call(L.make_cfg(2), 2013 + 1) == WORKSPACE     # 4028 units
    assert call(L.make_cfg(8), 504) == WORKSPACE          # 4032 units
    assert call(L.make_cfg(8), 10_000, budget=0) == WORKSPACE
    # argument errors come first, as on the workspace path
    assert lib.locks_sparse_decode_noalloc(ctypes.byref(L.make_cfg(8)), None, fake, fake, 10, fake, fake,
                                           fake, fake, 600, 8, 128, scale, fake, None) == INVALID
    assert lib.locks_noalloc_read_status(None, None) == INVALID


def test_binding_raises_on_missing_library(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "LIB", str(tmp_path / "nope.so"))
    monkeypatch.setattr(L, "_lib", None)
    with pytest.raises(ImportError):
        L.load()
