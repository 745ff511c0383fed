"""locks_sparse_decode_noalloc, the entry point for callers that cannot
allocate device memory (an engine that gave all of HBM to its KV-cache pool,
a latency-critical path where cudaMalloc would synchronise the device, a host
integration without an allocator).  Its scratch is a fixed array inside the
library; its output must match locks_sparse_decode, called with a workspace,
within the attention tolerance the other GPU tests use -- on two calls in a
row, since calls share (and do not re-zero all of) that array.  The calls
must not change the device's free memory, and the flags the kernel raises
must reach the caller through locks_noalloc_read_status.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test."""

import pytest
import torch

from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import ATTN_ATOL

pytestmark = pytest.mark.gpu


def _workspace_reference(w, d):
    H = w.num_kv_heads
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ, bufs.workspace)
    L.locks_score_select(H, d["q"], summ, d["block_table"], d["seq_lens"], w.budget_pages,
                         bufs.selected, bufs.n_selected, bufs.workspace, scores=bufs.scores)
    L.locks_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                          bufs.selected, bufs.n_selected, w.budget_pages, bufs.out, bufs.workspace)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    ref = bufs.out.clone()
    assert torch.isfinite(ref).all()
    return bufs, ref


def _noalloc(w, d, bufs, out):
    L.locks_sparse_decode_noalloc(w.num_kv_heads, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                  d["seq_lens"], bufs.selected, bufs.n_selected, w.budget_pages, out)


def test_noalloc_sparse_decode_matches_workspace_entry_point():
    w = W.Workload(name="noalloc", batch=2, context=16 * 400 + 5, context_hi=16 * 520,
                   num_kv_heads=8, group=4, budget_tokens=16 * 32, carriers_per_head=4, seed=77)
    d = W.generate(w, device="cuda", tail_fill="nan")
    bufs, ref = _workspace_reference(w, d)
    L.locks_noalloc_read_status()            # start from a clear status word
    # the first call in this process looks the scratch array up (and may load
    # the module that holds it); the free-memory check starts after it
    out = torch.full_like(ref, float("nan"))
    _noalloc(w, d, bufs, out)
    torch.cuda.synchronize()
    assert (out - ref).abs().max().item() <= ATTN_ATOL
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    alloc0 = torch.cuda.memory_allocated()
    for call in range(2):
        _noalloc(w, d, bufs, outs[call])
    torch.cuda.synchronize()
    # nothing allocated by the two calls: neither device memory nor torch's pool
    assert torch.cuda.mem_get_info()[0] == free0, "the calls changed the device's free memory"
    assert torch.cuda.memory_allocated() == alloc0
    for call in range(2):
        err = (outs[call] - ref).abs().max().item()
        assert err <= ATTN_ATOL, f"call {call}: max-abs difference {err}"
    assert L.locks_noalloc_read_status() == 0


def test_noalloc_near_its_size_limit():
    """4,024 (request, KV head) units, one below the documented 4,025-unit
    limit: 503 requests of 2-3 full pages with partial tails."""
    w = W.Workload(name="noalloc_limit", batch=503, context=16 * 2 + 3, context_hi=16 * 3 + 9,
                   num_kv_heads=8, group=4, budget_tokens=16 * 2, carriers_per_head=0, seed=79)
    d = W.generate(w, device="cuda", tail_fill="huge")
    bufs, ref = _workspace_reference(w, d)
    L.locks_noalloc_read_status()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        _noalloc(w, d, bufs, out)
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert err <= ATTN_ATOL, f"call {call}: max-abs difference {err}"
    assert L.locks_noalloc_read_status() == 0
    # one request more does not fit the fixed scratch
    w2 = w.scaled(batch=504)
    bt = torch.zeros(504, w.max_pages, dtype=torch.int32, device="cuda")
    lens = torch.full((504,), 40, dtype=torch.int32, device="cuda")
    q = torch.zeros(504, 32, 128, dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros(504, 8, w.budget_pages, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(504, 8, dtype=torch.int32, device="cuda")
    out = torch.empty(504, 32, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(L.LocksError) as e:
        L.locks_sparse_decode_noalloc(8, q, d["k_cache"], d["v_cache"], bt, lens, sel, nsel,
                                      w2.budget_pages, out)
    assert e.value.status == 3


def test_noalloc_reports_device_flags():
    """A selected index past the unit's full pages and a block id outside the
    cache are skipped by the kernel and reported, without a fault."""
    w = W.Workload(name="noalloc_flags", batch=2, context=16 * 64 + 5, num_kv_heads=8, group=4,
                   budget_tokens=16 * 8, carriers_per_head=0, seed=81)
    d = W.generate(w, device="cuda")
    bufs, ref = _workspace_reference(w, d)
    L.locks_noalloc_read_status()
    out = torch.empty_like(ref)
    sel_bad = bufs.selected.clone()
    sel_bad[0, 3, 0] = 64 + 7                     # request 0 has 64 full pages
    L.locks_sparse_decode_noalloc(8, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                  sel_bad, bufs.n_selected, w.budget_pages, out)
    assert L.locks_noalloc_read_status() == L.FLAG_BAD_SELECT
    assert L.locks_noalloc_read_status() == 0     # the read cleared it
    bt_bad = d["block_table"].clone()
    page = int(bufs.selected[1, 5, 2])
    bt_bad[1, page] = d["num_blocks"] + 11
    L.locks_sparse_decode_noalloc(8, d["q"], d["k_cache"], d["v_cache"], bt_bad, d["seq_lens"],
                                  bufs.selected, bufs.n_selected, w.budget_pages, out)
    assert L.locks_noalloc_read_status() == L.FLAG_BAD_BLOCK
    torch.cuda.synchronize()
    # request 0 never reads the altered block-table row
    assert (out[0] - ref[0]).abs().max().item() <= ATTN_ATOL
