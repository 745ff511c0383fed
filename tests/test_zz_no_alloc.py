"""locks_sparse_decode_noalloc, the entry point for callers that cannot
allocate device memory (an engine that gave all of HBM to its KV-cache pool,
a latency-critical path where cudaMalloc would synchronise the device, a host
integration without an allocator).  Its scratch is a fixed array inside the
library; its output must match locks_sparse_decode, called with a workspace,
within the attention tolerance the other GPU tests use -- on two calls in a
row, since calls share (and do not re-zero all of) that array.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test."""

import pytest
import torch

from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import ATTN_ATOL

pytestmark = pytest.mark.gpu


def test_noalloc_sparse_decode_matches_workspace_entry_point():
    w = W.Workload(name="noalloc", batch=2, context=16 * 400 + 5, context_hi=16 * 520,
                   num_kv_heads=8, group=4, budget_tokens=16 * 32, carriers_per_head=4, seed=77)
    d = W.generate(w, device="cuda", tail_fill="nan")
    H = w.num_kv_heads
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ, bufs.workspace)
    L.locks_score_select(H, d["q"], summ, d["block_table"], d["seq_lens"], w.budget_pages,
                         bufs.selected, bufs.n_selected, bufs.workspace, scores=bufs.scores)
    L.locks_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                          bufs.selected, bufs.n_selected, w.budget_pages, bufs.out, bufs.workspace)
    torch.cuda.synchronize()
    ref = bufs.out.clone()
    assert torch.isfinite(ref).all()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        L.locks_sparse_decode_noalloc(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                      d["seq_lens"], bufs.selected, bufs.n_selected, w.budget_pages,
                                      out)
        torch.cuda.synchronize()
        err = (out - ref).abs().max().item()
        assert err <= ATTN_ATOL, f"call {call}: max-abs difference {err}"
