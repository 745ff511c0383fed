"""The fused select + attend cluster kernel (locks_select_sparse_decode) and
the whole decode step (locks_decode_step, which uses that kernel when every
unit's cluster fits on the GPU at once and the selection kernel plus split-K
attention otherwise) against the separate calls and the fp64 oracle, on small
edge cases and on the named workloads."""

import numpy as np
import pytest
import torch

from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run, check_fused_unit, check_unit

pytestmark = pytest.mark.gpu


def _w(**kw):
    base = dict(name="t", batch=1, context=16 * 300 + 7, num_kv_heads=8, group=4,
                budget_tokens=16 * 24, carriers_per_head=4, seed=11)
    base.update(kw)
    return W.Workload(**base)


@pytest.mark.parametrize("ctx,heads,budget", [
    (16 * 300 + 7, 8, 24), (16 * 150 - 1, 2, 24), (16 * 150, 1, 24),     # tail 7 / 15 / 0
    (16 * 10 + 2, 8, 24), (5, 8, 24), (15, 4, 24),                         # n <= budget, tiny
    (16 * 2000 + 3, 8, 128), (16 * 64 + 9, 8, 100),                        # many pages / all
    (16 * 3000 + 1, 4, 1000),                                              # > 8 items per warp
])
def test_fused_matches_separate_and_oracle(ctx, heads, budget):
    w = _w(context=ctx, num_kv_heads=heads, budget_tokens=16 * budget, seed=ctx % 97 + heads)
    run = Run(w, tail_fill="nan", fused=True)
    assert run.status == 0
    for h in range(heads):
        check_unit(run, 0, h, check_scores_too=False)
        check_fused_unit(run, 0, h)


def test_fused_ragged_batch_and_ties():
    w = _w(batch=4, context=16 * 90, context_hi=16 * 700, budget_tokens=16 * 40, seed=5)
    run = Run(w, tail_fill="huge", fused=True, step=True)
    assert run.status == 0
    for b in range(4):
        for h in (0, 7):
            check_fused_unit(run, b, h)
            check_fused_unit(run, b, h, which="step")   # 32 units x 8 CTAs: the separate path


@pytest.mark.parametrize("batch,heads", [(1, 8), (2, 8), (19, 1), (20, 8)])
def test_decode_step_both_paths(batch, heads):
    # batch x heads x 8 CTAs <= 152 SMs takes the fused kernel, more the separate path
    w = _w(batch=batch, num_kv_heads=heads, context=16 * 120, context_hi=16 * 400,
           budget_tokens=16 * 32, seed=batch + heads)
    run = Run(w, tail_fill="nan", step=True)
    assert run.status == 0
    for b in sorted({0, batch // 2, batch - 1}):
        for h in sorted({0, heads - 1}):
            check_fused_unit(run, b, h, which="step")


def test_fused_step_in_a_graph_is_stable():
    w = _w(context=16 * 800 + 5, seed=9)
    run = Run(w, step=True)
    first = run.step["out"].clone()
    d, H, bufs, f = run.d, run.H, run.bufs, run.step
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.locks_decode_step(H, d["q"], run.summ, d["k_cache"], d["v_cache"], d["block_table"],
                            d["seq_lens"], w.budget_pages, f["selected"], f["n_selected"], f["out"],
                            bufs.workspace)
    f["out"].zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first, f["out"])
    assert L.locks_read_status(bufs.workspace) == 0


@pytest.mark.parametrize("name", ["llama8b_128k", "ctx1m"])
def test_fused_named_workloads(name):
    run = Run(W.CONFIGS[name], fused=True)
    assert run.status == 0
    for h in range(8):
        check_fused_unit(run, 0, h)


def test_fused_rejects_unsupported_budget():
    w = _w(context=16 * 100, budget_tokens=16 * 2048)
    d = W.generate(w, device="cuda")
    bufs = L.DecodeBuffers(8, 1, w.max_pages, w.budget_pages)
    summ = torch.zeros(d["num_blocks"], 8, 784, dtype=torch.uint8, device="cuda")
    with pytest.raises(L.LocksError) as e:
        L.locks_select_sparse_decode(8, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                     d["seq_lens"], w.budget_pages, bufs.selected, bufs.n_selected,
                                     bufs.out, bufs.workspace)
    assert e.value.status == 2


@pytest.mark.parametrize("kernel", ["select", "fused"])
def test_selection_takes_lowest_index_copies_of_tied_rows(kernel):
    """Score rows copied bit for bit across pages that straddle the budget
    boundary: the copies have equal keys, and both selection kernels must
    take the lowest-index ones (LOCKS summary §2: ties go to the lower page
    index).  The scores are planted straight into the table, so the scorer's
    own rounding plays no part."""
    import oracle as O
    from gpu_helpers import check_selection

    w = _w(context=16 * 700 + 5, budget_tokens=16 * 40, seed=34)
    run = Run(w)
    H, bufs, d = run.H, run.bufs, run.d
    n, k = run.lens[0] // 16, w.budget_pages
    rng = np.random.default_rng(8)
    tied = {}
    for h in range(H):
        base = (rng.normal(size=(n, 4)) * 2.0).astype(np.float32)
        _, avg = O.select_pages(base.astype(np.float64), k)
        order = np.argsort(-avg, kind="stable")
        # copy one row to six lower-ranked pages; the copies move Z_g, so try
        # source ranks from k - 3 upwards until the seven rows straddle the
        # boundary in the oracle's own ranking
        for r in range(k - 3, -1, -1):
            table = base.copy()
            src = order[r]
            copies = rng.choice(order[r + 1:k + 40], size=6, replace=False)
            table[copies] = table[src]
            pages = np.sort(np.append(copies, src))
            sel_or, _ = O.select_pages(table.astype(np.float64), k)
            taken = np.intersect1d(sel_or, pages)
            if 0 < taken.size < pages.size:
                break
        assert 0 < taken.size < pages.size, "the copies must straddle the boundary"
        tied[h] = (pages, taken)
        bufs.scores[0, h, :n] = torch.from_numpy(table).cuda()
    sel = torch.full_like(bufs.selected, -1)
    nsel = torch.full_like(bufs.n_selected, -1)
    if kernel == "select":
        L.locks_select(H, d["seq_lens"], w.max_pages, k, sel, nsel, bufs.workspace, scores=bufs.scores)
    else:
        out = torch.empty_like(bufs.out)
        L.locks_select_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                     k, sel, nsel, out, bufs.workspace, scores=bufs.scores)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    for h in range(H):
        pages, taken = tied[h]
        got = sel[0, h, :int(nsel[0, h])].cpu().numpy().astype(np.int64)
        check_selection(got, bufs.scores[0, h, :n].double().cpu().numpy(), k)
        got_tied = np.intersect1d(got, pages)
        assert got_tied.tolist() == pages[:got_tied.size].tolist(), (h, pages, got_tied)
        assert got_tied.tolist() == taken.tolist(), (h, got_tied, taken)
