"""Thin ctypes binding of liblocks.so (declared in include/locks.h).

Argument marshalling only: tensors are passed as raw device pointers, the
current torch CUDA stream as the cudaStream_t.  Every computation happens in
the library's kernels.  There is no fallback: if the library is missing or
fails to load, importing the first entry point raises.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

from . import build as _build

LOCKS_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
                3: "workspace too small", 4: "CUDA error", 5: "device wait timed out"}
FLAG_BAD_BLOCK, FLAG_BAD_SEQLEN, FLAG_TIMEOUT, FLAG_BAD_SELECT = 1, 2, 4, 8

HEAD_DIM, PAGE_SIZE, RANK, GROUP = 128, 16, 8, 4
RECORD_BYTES = 784   # one page-head summary record


class LocksError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} (status {status})")
        self.status = status


class locks_cfg(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("quant", ctypes.c_int32)]


def make_cfg(num_kv_heads: int, group_size: int = GROUP, quant: int = 1, rank: int = RANK) -> locks_cfg:
    """quant=1: the 784-byte int4/int8 records at rank 8; quant=0: unquantised
    fp32 records of rank 1..16 (record_bytes(0, rank) bytes)."""
    return locks_cfg(HEAD_DIM, PAGE_SIZE, rank, num_kv_heads, group_size, quant)


def record_bytes(quant: int = 1, rank: int = RANK) -> int:
    """Bytes of one page-head summary record (see include/locks.h)."""
    return RECORD_BYTES if quant == 1 else 528 + 576 * rank


_lib = None
_P = ctypes.c_void_p
_I32, _I64, _SZ, _F = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_CFG = ctypes.POINTER(locks_cfg)

_SIGS = {
    "locks_summary_bytes": (_SZ, [_CFG]),
    "locks_workspace_bytes": (_I32, [_CFG, _I32, _I32, _I32, ctypes.POINTER(_SZ)]),
    "locks_workspace_init": (_I32, [_P, _SZ, _P]),
    "locks_read_status": (_I32, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "locks_device_accessible": (_I32, [_P]),
    "locks_build_summaries": (_I32, [_CFG, _P, _I64, _P, _I32, _P, _P, _SZ, _P]),
    "locks_build_pending": (_I32, [_CFG, _P, _I64, _P, _P, _I32, _P, _P, _SZ, _P]),
    "locks_score": (_I32, [_CFG, _P, _P, _I64, _P, _P, _I32, _I32, _P, _P, _SZ, _P]),
    "locks_select": (_I32, [_CFG, _P, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "locks_score_select": (_I32, [_CFG, _P, _P, _I64, _P, _P, _I32, _I32, _I32, _P, _P, _P,
                                  _P, _SZ, _P]),
    "locks_sparse_decode": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _P, _P, _I32, _I32, _I32,
                                   _F, _P, _P, _SZ, _P]),
    "locks_dense_decode": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _I32, _I32, _F, _P, _P, _SZ,
                                  _P]),
    "locks_select_sparse_decode": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _I32, _I32, _I32, _P, _P,
                                          _P, _F, _P, _P, _SZ, _P]),
    "locks_decode_step": (_I32, [_CFG, _P, _P, _P, _P, _I64, _P, _P, _I32, _I32, _I32, _F, _P, _P,
                                 _P, _P, _P, _SZ, _P]),
    "locks_decode_step_crossing": (_I32, [_CFG, _P, _P, _P, _P, _I64, _P, _P, _I32, _I32, _I32, _F, _P, _P,
                                          _P, _P, _P, _SZ, _P]),
    "locks_status_str": (ctypes.c_char_p, [_I32]),
    "locks_sparse_decode_noalloc": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _P, _P, _I32, _I32,
                                           _I32, _F, _P, _P]),
    "locks_noalloc_read_status": (_I32, [ctypes.POINTER(ctypes.c_uint32), _P]),
    "locks_check_bounded_wait": (_I32, [_P, _P, ctypes.c_uint32, _P, _SZ, _P]),
    "locks_shared_basis_build": (_I32, [_CFG, _P, _I64, _P, _I32, _P, _I32, _P, _P, _SZ, _P]),
    "locks_shared_basis_score": (_I32, [_CFG, _P, _P, _I32, _P, _I64, _P, _P, _I32, _I32, _P, _P, _SZ, _P]),
    "locks_cp_score_pairs": (_I32, [_CFG, _P, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "locks_cp_select_local": (_I32, [_CFG, _P, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _P, _P, _SZ,
                                     _P]),
    "locks_cp_merge_select": (_I32, [_CFG, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "locks_cp_sparse_decode_partial": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _P, _P, _I32, _I32, _I32,
                                              _F, _P, _P, _SZ, _P]),
    "locks_cp_merge_attention": (_I32, [_CFG, _I32, _I32, _P, _P, _P]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load liblocks.so (optionally building it first) and declare signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"liblocks.so not found at {path}; run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, where: str) -> None:
    if status != LOCKS_OK:
        raise LocksError(status, where)


# ------------------------------------------------------------------ sizes
def locks_summary_bytes(num_kv_heads: int, quant: int = 1, rank: int = RANK) -> int:
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    return int(load().locks_summary_bytes(ctypes.byref(cfg)))


def locks_workspace_bytes(num_kv_heads: int, batch: int, max_pages: int, budget_pages: int) -> int:
    cfg = make_cfg(num_kv_heads)
    out = _SZ(0)
    _check(load().locks_workspace_bytes(ctypes.byref(cfg), batch, max_pages, budget_pages,
                                        ctypes.byref(out)), "locks_workspace_bytes")
    return int(out.value)


def locks_workspace_init(workspace, stream=None) -> None:
    _check(load().locks_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "locks_workspace_init")


LOCKS_ERR_TIMEOUT = 5


def _check_status_read(status: int, where: str) -> None:
    # LOCKS_ERR_TIMEOUT only says that the flags read include FLAG_TIMEOUT
    if status not in (LOCKS_OK, LOCKS_ERR_TIMEOUT):
        raise LocksError(status, where)


def locks_read_status(workspace, stream=None) -> int:
    """Flags of the status word (read and cleared; synchronises the stream)."""
    v = ctypes.c_uint32(0)
    _check_status_read(load().locks_read_status(_ptr(workspace), ctypes.byref(v), _stream(stream)),
                       "locks_read_status")
    return int(v.value)


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


# ------------------------------------------------------------------ argument checks
# The C ABI receives bare pointers, so the layouts it assumes (include/locks.h)
# are checked here, before any pointer is passed: a contiguous CUDA tensor of
# the stated dtype and shape.  A mismatch raises ValueError.
def _req(t, name: str, dtype: str, shape=None, optional: bool = False) -> None:
    """shape: a tuple of sizes, None for a free axis (its rank is checked)."""
    import torch
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    want = getattr(torch, dtype)
    if t.dtype != want:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None:
        if t.dim() != len(shape) or any(n is not None and t.shape[i] != n for i, n in enumerate(shape)):
            want_s = "[" + ", ".join("*" if n is None else str(n) for n in shape) + "]"
            raise ValueError(f"{name} must have shape {want_s}, got {list(t.shape)}")


def _req_out(out, B: int, H: int) -> None:
    """out [batch, H*G, 128] fp32: a CUDA tensor, or a pinned host tensor the
    device addresses with the same pointer (the kernels then store the result
    straight into host memory)."""
    import torch
    if isinstance(out, torch.Tensor) and not out.is_cuda:
        if not out.is_pinned():
            raise ValueError("out must be a CUDA tensor or a pinned host tensor")
        if out.dtype != torch.float32 or not out.is_contiguous() or \
                tuple(out.shape) != (B, H * GROUP, HEAD_DIM):
            raise ValueError(f"out must be a contiguous float32 tensor of shape [{B}, {H * GROUP}, {HEAD_DIM}]")
        if load().locks_device_accessible(out.data_ptr()) != 1:
            raise ValueError("out: this pinned host memory is not addressable by the device")
        return
    _req(out, "out", "float32", (B, H * GROUP, HEAD_DIM))


def _req_cache(t, name: str, H: int) -> None:
    _req(t, name, "bfloat16", (None, H, PAGE_SIZE, HEAD_DIM))


def _req_step(H, q, block_table, seq_lens) -> tuple:
    """q [batch, H*G, 128] bf16; block_table [batch, max_pages] int32;
    seq_lens [batch] int32.  Returns (batch, max_pages)."""
    _req(block_table, "block_table", "int32", (None, None))
    B, MP = block_table.shape
    _req(seq_lens, "seq_lens", "int32", (B,))
    if q is not None:
        _req(q, "q", "bfloat16", (B, H * GROUP, HEAD_DIM))
    return B, MP


def _req_selection(H, B, budget_pages, selected, n_selected) -> None:
    _req(n_selected, "n_selected", "int32", (B, H))
    _req(selected, "selected", "int32", (B, H, budget_pages) if budget_pages > 0 else None,
         optional=budget_pages == 0)


# ------------------------------------------------------------------ calls
def locks_build_summaries(num_kv_heads, k_cache, block_ids, summaries, workspace=None, stream=None,
                          quant=1, rank=RANK):
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(block_ids, "block_ids", "int32", (None,))
    _req(summaries, "summaries", "uint8", (k_cache.shape[0], num_kv_heads, record_bytes(quant, rank)))
    _req(workspace, "workspace", "uint8", optional=True)
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    _check(load().locks_build_summaries(
        ctypes.byref(cfg), _ptr(k_cache), k_cache.shape[0], _ptr(block_ids), block_ids.numel(),
        _ptr(summaries), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_build_summaries")


def locks_build_pending(num_kv_heads, k_cache, block_ids, n_pending, summaries, workspace=None,
                        stream=None, quant=1, rank=RANK):
    """Build the records of block_ids[0, n_pending[0]) (n_pending: a device
    int32 tensor, read by the kernel); block_ids holds room for the most pages
    any step can finalise."""
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(block_ids, "block_ids", "int32", (None,))
    _req(n_pending, "n_pending", "int32", (None,))
    _req(summaries, "summaries", "uint8", (k_cache.shape[0], num_kv_heads, record_bytes(quant, rank)))
    _req(workspace, "workspace", "uint8", optional=True)
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    _check(load().locks_build_pending(
        ctypes.byref(cfg), _ptr(k_cache), k_cache.shape[0], _ptr(block_ids), _ptr(n_pending),
        block_ids.numel(), _ptr(summaries), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_build_pending")


def locks_score(num_kv_heads, q, summaries, block_table, seq_lens, workspace, scores=None,
                stream=None, quant=1, rank=RANK):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req(summaries, "summaries", "uint8", (None, num_kv_heads, record_bytes(quant, rank)))
    _req(scores, "scores", "float32", (B, num_kv_heads, MP, GROUP), optional=True)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    _check(load().locks_score(
        ctypes.byref(cfg), _ptr(q), _ptr(summaries), summaries.shape[0], _ptr(block_table),
        _ptr(seq_lens), block_table.shape[0], block_table.shape[1], _ptr(scores), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "locks_score")


def locks_select(num_kv_heads, seq_lens, max_pages, budget_pages, selected, n_selected, workspace,
                 scores=None, stream=None):
    _req(seq_lens, "seq_lens", "int32", (None,))
    B = seq_lens.shape[0]
    _req(scores, "scores", "float32", (B, num_kv_heads, max_pages, GROUP), optional=True)
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_select(
        ctypes.byref(cfg), _ptr(seq_lens), seq_lens.shape[0], max_pages, budget_pages, _ptr(scores),
        _ptr(selected), _ptr(n_selected), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_select")


def locks_score_select(num_kv_heads, q, summaries, block_table, seq_lens, budget_pages, selected,
                       n_selected, workspace, scores=None, stream=None, quant=1, rank=RANK):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req(summaries, "summaries", "uint8", (None, num_kv_heads, record_bytes(quant, rank)))
    _req(scores, "scores", "float32", (B, num_kv_heads, MP, GROUP), optional=True)
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    _check(load().locks_score_select(
        ctypes.byref(cfg), _ptr(q), _ptr(summaries), summaries.shape[0], _ptr(block_table),
        _ptr(seq_lens), block_table.shape[0], block_table.shape[1], budget_pages, _ptr(scores),
        _ptr(selected), _ptr(n_selected), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_score_select")


def locks_sparse_decode(num_kv_heads, q, k_cache, v_cache, block_table, seq_lens, selected,
                        n_selected, budget_pages, out, workspace, sm_scale=None, stream=None):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req_out(out, B, num_kv_heads)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_sparse_decode(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_table), _ptr(seq_lens), _ptr(selected), _ptr(n_selected),
        block_table.shape[0], block_table.shape[1], budget_pages, scale, _ptr(out),
        _ptr(workspace), _nbytes(workspace), _stream(stream)), "locks_sparse_decode")


def locks_select_sparse_decode(num_kv_heads, q, k_cache, v_cache, block_table, seq_lens,
                               budget_pages, selected, n_selected, out, workspace, scores=None,
                               sm_scale=None, stream=None):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req(scores, "scores", "float32", (B, num_kv_heads, MP, GROUP), optional=True)
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req_out(out, B, num_kv_heads)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_select_sparse_decode(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_table), _ptr(seq_lens), block_table.shape[0], block_table.shape[1],
        budget_pages, _ptr(scores), _ptr(selected), _ptr(n_selected), scale, _ptr(out),
        _ptr(workspace), _nbytes(workspace), _stream(stream)), "locks_select_sparse_decode")


def locks_decode_step(num_kv_heads, q, summaries, k_cache, v_cache, block_table, seq_lens,
                      budget_pages, selected, n_selected, out, workspace, scores=None,
                      sm_scale=None, stream=None, quant=1, rank=RANK):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req(summaries, "summaries", "uint8", (None, num_kv_heads, record_bytes(quant, rank)))
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req(scores, "scores", "float32", (B, num_kv_heads, MP, GROUP), optional=True)
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req_out(out, B, num_kv_heads)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_decode_step(
        ctypes.byref(cfg), _ptr(q), _ptr(summaries), _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(block_table), _ptr(seq_lens), block_table.shape[0],
        block_table.shape[1], budget_pages, scale, _ptr(scores), _ptr(selected),
        _ptr(n_selected), _ptr(out), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_decode_step")


def locks_decode_step_crossing(num_kv_heads, q, summaries, k_cache, v_cache, block_table, seq_lens,
                               budget_pages, selected, n_selected, out, workspace, scores=None,
                               sm_scale=None, stream=None, quant=1, rank=RANK):
    """locks_decode_step after building the page each request's current token
    completed (requests with L_b % 16 == 0), overlapped with the scoring."""
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req(summaries, "summaries", "uint8", (k_cache.shape[0], num_kv_heads, record_bytes(quant, rank)))
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req(scores, "scores", "float32", (B, num_kv_heads, MP, GROUP), optional=True)
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req_out(out, B, num_kv_heads)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads, quant=quant, rank=rank)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_decode_step_crossing(
        ctypes.byref(cfg), _ptr(q), _ptr(summaries), _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], _ptr(block_table), _ptr(seq_lens), block_table.shape[0],
        block_table.shape[1], budget_pages, scale, _ptr(scores), _ptr(selected),
        _ptr(n_selected), _ptr(out), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_decode_step_crossing")


def locks_dense_decode(num_kv_heads, q, k_cache, v_cache, block_table, seq_lens, out, workspace,
                       sm_scale=None, stream=None):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req_out(out, B, num_kv_heads)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_dense_decode(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_table), _ptr(seq_lens), block_table.shape[0], block_table.shape[1], scale,
        _ptr(out), _ptr(workspace), _nbytes(workspace), _stream(stream)), "locks_dense_decode")


def locks_sparse_decode_noalloc(num_kv_heads, q, k_cache, v_cache, block_table, seq_lens, selected,
                                n_selected, budget_pages, out, sm_scale=None, stream=None):
    """locks_sparse_decode for callers that cannot allocate: the library's own
    fixed device scratch replaces the workspace (see include/locks.h)."""
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req_out(out, B, num_kv_heads)
    cfg = make_cfg(num_kv_heads)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_sparse_decode_noalloc(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
        _ptr(block_table), _ptr(seq_lens), _ptr(selected), _ptr(n_selected),
        block_table.shape[0], block_table.shape[1], budget_pages, scale, _ptr(out),
        _stream(stream)), "locks_sparse_decode_noalloc")


def locks_noalloc_read_status(stream=None) -> int:
    """Flags accumulated by locks_sparse_decode_noalloc since the last read
    (the read clears them); synchronises the stream."""
    v = ctypes.c_uint32(0)
    _check_status_read(load().locks_noalloc_read_status(ctypes.byref(v), _stream(stream)),
                       "locks_noalloc_read_status")
    return int(v.value)


def locks_check_bounded_wait(src, result, limit_us, workspace, stream=None) -> None:
    """Diagnostic: make one bounded wait run out after limit_us (see locks.h).
    src: 256 bytes on the device; result: device int32/uint32 [4]."""
    _req(src, "src", "uint8", (256,))
    _req(result, "result", "int32", (4,))
    _req(workspace, "workspace", "uint8")
    _check(load().locks_check_bounded_wait(_ptr(src), _ptr(result), int(limit_us), _ptr(workspace),
                                           _nbytes(workspace), _stream(stream)),
           "locks_check_bounded_wait")


# ------------------------------------------------------------------ shared-basis ablation
def shared_basis_record_bytes(rho: int) -> int:
    return 512 + 64 * rho


def locks_shared_basis_build(num_kv_heads, k_cache, block_ids, basis, records, workspace=None, stream=None):
    """basis: float32 [H_kv, 128, rho]; records: uint8 [num_blocks, H_kv, 512 + 64 rho]."""
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(block_ids, "block_ids", "int32", (None,))
    _req(basis, "basis", "float32", (num_kv_heads, HEAD_DIM, None))
    rho = basis.shape[2]
    _req(records, "records", "uint8", (k_cache.shape[0], num_kv_heads, shared_basis_record_bytes(rho)))
    _req(workspace, "workspace", "uint8", optional=True)
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_shared_basis_build(
        ctypes.byref(cfg), _ptr(k_cache), k_cache.shape[0], _ptr(block_ids), block_ids.numel(), _ptr(basis), rho,
        _ptr(records), _ptr(workspace), _nbytes(workspace), _stream(stream)), "locks_shared_basis_build")


def locks_shared_basis_score(num_kv_heads, q, basis, records, block_table, seq_lens, workspace, scores=None,
                             stream=None):
    B, MP = _req_step(num_kv_heads, q, block_table, seq_lens)
    _req(basis, "basis", "float32", (num_kv_heads, HEAD_DIM, None))
    rho = basis.shape[2]
    _req(records, "records", "uint8", (None, num_kv_heads, shared_basis_record_bytes(rho)))
    _req(scores, "scores", "float32", (B, num_kv_heads, MP, GROUP), optional=True)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_shared_basis_score(
        ctypes.byref(cfg), _ptr(q), _ptr(basis), rho, _ptr(records), records.shape[0], _ptr(block_table),
        _ptr(seq_lens), B, MP, _ptr(scores), _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "locks_shared_basis_score")


# ------------------------------------------------------------------ context-parallel shards
# One request's pages split over several GPUs; see include/locks.h.  Every
# tensor is this shard's own; *_all tensors stack every shard's result on a
# leading axis (gathered by the caller).
def locks_cp_score_pairs(num_kv_heads, shard_lens, max_pages, pairs, workspace, scores=None, stream=None):
    _req(shard_lens, "shard_lens", "int32", (None,))
    B = shard_lens.shape[0]
    _req(pairs, "pairs", "float32", (B, num_kv_heads, GROUP, 2))
    _req(scores, "scores", "float32", (B, num_kv_heads, max_pages, GROUP), optional=True)
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_cp_score_pairs(ctypes.byref(cfg), _ptr(shard_lens), B, max_pages, _ptr(scores),
                                       _ptr(pairs), _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "locks_cp_score_pairs")


def locks_cp_select_local(num_kv_heads, shard_lens, page_offset, max_pages, budget_pages, pairs_all,
                          cand_pages, cand_keys, cand_counts, workspace, scores=None, stream=None):
    _req(shard_lens, "shard_lens", "int32", (None,))
    B = shard_lens.shape[0]
    _req(page_offset, "page_offset", "int32", (B,))
    _req(pairs_all, "pairs_all", "float32", (None, B, num_kv_heads, GROUP, 2))
    _req(scores, "scores", "float32", (B, num_kv_heads, max_pages, GROUP), optional=True)
    _req(cand_pages, "cand_pages", "int32", (B, num_kv_heads, max(1, budget_pages)))
    _req(cand_keys, "cand_keys", "int32", (B, num_kv_heads, max(1, budget_pages)))
    _req(cand_counts, "cand_counts", "int32", (B, num_kv_heads))
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_cp_select_local(
        ctypes.byref(cfg), _ptr(shard_lens), _ptr(page_offset), B, max_pages, budget_pages, _ptr(scores),
        _ptr(pairs_all), pairs_all.shape[0], _ptr(cand_pages), _ptr(cand_keys), _ptr(cand_counts),
        _ptr(workspace), _nbytes(workspace), _stream(stream)), "locks_cp_select_local")


def locks_cp_merge_select(num_kv_heads, page_offset, budget_pages, shard, cand_pages_all, cand_keys_all,
                          cand_counts_all, selected, n_selected, stream=None):
    _req(page_offset, "page_offset", "int32", (None,))
    B = page_offset.shape[0]
    R = cand_counts_all.shape[0]
    _req(cand_pages_all, "cand_pages_all", "int32", (R, B, num_kv_heads, max(1, budget_pages)))
    _req(cand_keys_all, "cand_keys_all", "int32", (R, B, num_kv_heads, max(1, budget_pages)))
    _req(cand_counts_all, "cand_counts_all", "int32", (R, B, num_kv_heads))
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_cp_merge_select(
        ctypes.byref(cfg), _ptr(page_offset), B, budget_pages, R, shard, _ptr(cand_pages_all),
        _ptr(cand_keys_all), _ptr(cand_counts_all), _ptr(selected), _ptr(n_selected), _stream(stream)),
        "locks_cp_merge_select")


def locks_cp_sparse_decode_partial(num_kv_heads, q, k_cache, v_cache, block_table, shard_lens, selected,
                                   n_selected, budget_pages, states, workspace, sm_scale=None, stream=None):
    B, MP = _req_step(num_kv_heads, q, block_table, shard_lens)
    _req_cache(k_cache, "k_cache", num_kv_heads)
    _req(v_cache, "v_cache", "bfloat16", tuple(k_cache.shape))
    _req_selection(num_kv_heads, B, budget_pages, selected, n_selected)
    _req(states, "states", "float32", (B, num_kv_heads * GROUP, 2 + HEAD_DIM))
    _req(workspace, "workspace", "uint8")
    cfg = make_cfg(num_kv_heads)
    scale = 1.0 / math.sqrt(HEAD_DIM) if sm_scale is None else sm_scale
    _check(load().locks_cp_sparse_decode_partial(
        ctypes.byref(cfg), _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(block_table),
        _ptr(shard_lens), _ptr(selected), _ptr(n_selected), B, MP, budget_pages, scale, _ptr(states),
        _ptr(workspace), _nbytes(workspace), _stream(stream)), "locks_cp_sparse_decode_partial")


def locks_cp_merge_attention(num_kv_heads, states_all, out, stream=None):
    R, B = states_all.shape[0], states_all.shape[1]
    _req(states_all, "states_all", "float32", (R, B, num_kv_heads * GROUP, 2 + HEAD_DIM))
    _req_out(out, B, num_kv_heads)
    cfg = make_cfg(num_kv_heads)
    _check(load().locks_cp_merge_attention(ctypes.byref(cfg), B, R, _ptr(states_all), _ptr(out),
                                           _stream(stream)), "locks_cp_merge_attention")


def locks_status_str(status: int) -> str:
    return load().locks_status_str(status).decode()


# ------------------------------------------------------------------ helper
class DecodeBuffers:
    """Device buffers of one decode step for a batch shape (allocated by torch)."""

    def __init__(self, num_kv_heads: int, batch: int, max_pages: int, budget_pages: int,
                 device="cuda"):
        import torch
        self.num_kv_heads, self.batch = num_kv_heads, batch
        self.max_pages, self.budget_pages = max_pages, budget_pages
        nbytes = locks_workspace_bytes(num_kv_heads, batch, max_pages, budget_pages)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        locks_workspace_init(self.workspace)
        self.scores = torch.empty(batch, num_kv_heads, max_pages, GROUP, dtype=torch.float32,
                                  device=device)
        self.selected = torch.full((batch, num_kv_heads, max(1, budget_pages)), -1,
                                   dtype=torch.int32, device=device)
        self.n_selected = torch.zeros(batch, num_kv_heads, dtype=torch.int32, device=device)
        self.out = torch.empty(batch, num_kv_heads * GROUP, HEAD_DIM, dtype=torch.float32,
                               device=device)
