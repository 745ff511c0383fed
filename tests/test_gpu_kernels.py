"""GPU parity of each LOCKS kernel against the fp64 oracle on small seeded
cases (several tiles, ragged tails, edge cases).  All calls go through the C
ABI (liblocks.so) via the ctypes binding."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import (Run, check_attention, check_records, check_scores, check_selection,
                         check_unit)

pytestmark = pytest.mark.gpu


def _w(**kw):
    base = dict(name="t", batch=1, context=16 * 300 + 7, num_kv_heads=8, group=4,
                budget_tokens=16 * 24, carriers_per_head=4, seed=11)
    base.update(kw)
    return W.Workload(**base)


# ------------------------------------------------------------------ a1/a2 build
@pytest.mark.parametrize("noise", [0.05, 0.1])
def test_build_summaries_parity(noise):
    w = W.CONFIGS["pr1_4k"].scaled(noise_std=noise, seed=3)
    run = Run(w)
    assert run.status == 0
    n = run.lens[0] // 16
    K = run.pages_f64(run.d["k_cache"], 0, 0, range(n))
    info = check_records(run.records(0, 0), K)
    assert info["well_conditioned"] > 0.75 * n


def test_build_summaries_fullrank_and_multihead():
    w = _w(key_regime="fullrank", context=16 * 64 + 3, num_kv_heads=2)
    run = Run(w)
    for h in range(2):
        n = run.lens[0] // 16
        check_records(run.records(0, h), run.pages_f64(run.d["k_cache"], 0, h, range(n)))


def test_build_special_pages():
    """Equal keys, exact low rank, zero page, large and tiny magnitudes."""
    rng = np.random.default_rng(5)
    pages = []
    k = rng.normal(size=128)
    pages.append(np.tile(k, (16, 1)))                                   # all keys equal
    mu = rng.integers(-3, 4, 128)
    U = rng.integers(-2, 3, (128, 3))
    C = rng.integers(-3, 4, (16, 3))
    pages.append(mu + C @ U.T)                                          # rank 3
    pages.append(np.zeros((16, 128)))                                   # zero page
    pages.append(rng.normal(size=(16, 128)) * 300.0)                    # large
    pages.append(rng.normal(size=(16, 128)) * 1e-3)                     # tiny
    K = torch.tensor(np.stack(pages), dtype=torch.bfloat16)            # bf16-exact inputs
    kc = K[:, None].contiguous().cuda()                                 # [P, 1, 16, 128]
    summ = torch.zeros(K.shape[0], 1, 784, dtype=torch.uint8, device="cuda")
    ids = torch.arange(K.shape[0], dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(1, kc, ids, summ, ws)
    torch.cuda.synchronize()
    assert L.locks_read_status(ws) == 0
    rec = summ[:, 0].cpu().numpy()
    Kd = K.double().numpy()
    check_records(rec, Kd)
    g = O.decode_records(rec)
    # equal keys and the zero page: no basis at all
    for p in (0, 2):
        assert g["sV"][p] == 0 and g["sC"][p] == 0
        assert np.all(g["Vq"][p] == 0) and np.all(g["Cq"][p] == 0)
    # rank 3: directions 3..7 are zero
    assert np.all(g["Vq"][1][:, 3:] == 0) and np.all(g["Cq"][1][:, 3:] == 0)


def test_build_flags_bad_block_ids():
    kc = torch.randn(4, 2, 16, 128, device="cuda").to(torch.bfloat16)
    summ = torch.full((4, 2, 784), 7, dtype=torch.uint8, device="cuda")
    ids = torch.tensor([1, 9, -3, 2], dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(2, kc, ids, summ, ws)
    torch.cuda.synchronize()
    assert L.locks_read_status(ws) & L.FLAG_BAD_BLOCK
    untouched = summ.cpu()
    assert torch.all(untouched[0] == 7) and torch.all(untouched[3] == 7)
    assert not torch.all(untouched[1] == 7) and not torch.all(untouched[2] == 7)


# ------------------------------------------------------------------ a3-a6 pipeline
def test_pipeline_pr1_config():
    run = Run(W.CONFIGS["pr1_4k"])
    assert run.status == 0
    res = check_unit(run, 0, 0)
    assert res["band"] <= 2


@pytest.mark.parametrize("tail", [0, 1, 15])
@pytest.mark.parametrize("heads", [1, 2, 8])
def test_pipeline_tail_lengths_and_head_counts(tail, heads):
    w = _w(context=16 * 150 + tail - 1 if tail else 16 * 150 - 1, num_kv_heads=heads, seed=tail + 10 * heads)
    run = Run(w, tail_fill="nan")
    assert run.status == 0
    assert run.lens[0] % 16 == tail
    for h in range(heads):
        check_unit(run, 0, h)


def test_pipeline_fewer_pages_than_budget_and_tiny_contexts():
    for ctx, seed in ((16 * 10 + 2, 1), (16 * 24 - 1, 2), (5, 3), (15, 4), (16, 5)):
        run = Run(_w(context=ctx, seed=seed, carriers_per_head=1), tail_fill="nan")
        assert run.status == 0
        for h in range(8):
            n = run.lens[0] // 16
            assert run.gpu_selected(0, h).tolist() == list(range(min(n, 24)))
            check_unit(run, 0, h)


def test_pipeline_ragged_batch():
    w = _w(batch=3, context=16 * 90, context_hi=16 * 200, budget_tokens=16 * 32, seed=21)
    run = Run(w, tail_fill="huge")
    assert run.status == 0
    assert len(set(run.lens)) > 1
    for b in range(3):
        for h in (0, 3, 7):
            check_unit(run, b, h)


@pytest.mark.parametrize("q_scale", [30.0, 100.0, 300.0])
def test_scores_with_huge_deviation_logits(q_scale):
    """Queries scaled until a page's 16-token sum of 2^x passes 2^100 (x in
    log2 units): those rows take the max-shifted log-sum-exp, the rest of the
    warp's rows follow it, and every score must still match the oracle.
    Selection is not compared here: the shares of most pages underflow in fp32
    while fp64 keeps them apart."""
    w = _w(context=16 * 200 + 3, seed=71)
    d = W.generate(w, device="cuda")
    d["q"] = (d["q"].float() * q_scale).to(torch.bfloat16)
    run = Run(w, data=d)
    assert run.status == 0
    n = run.lens[0] // 16
    past = 0
    for h in range(w.num_kv_heads):
        qg = run.q_group(0, h)
        dq = O.dequantize(O.decode_records(run.records(0, h)))
        s_ref = O.page_scores(qg, dq["mu"], dq["V"], dq["C"])
        check_scores(run.gpu_scores(0, h), s_ref)
        lse_dev = s_ref - dq["mu"] @ qg.T / math.sqrt(128)        # natural log of the deviation sum
        past += int(np.sum(lse_dev * (1 / math.log(2)) > 100.0))
    assert past > 0, "no row reached the max-shifted branch"
    assert past < w.num_kv_heads * n * w.group, "every row reached it"


def test_pipeline_exact_ties_go_to_lower_page_index():
    """Identical pages give identical records and scores: ties at the budget
    boundary must be broken by the lower page index."""
    w = _w(context=16 * 40, num_kv_heads=1, budget_tokens=16 * 5, carriers_per_head=0, seed=8)
    d = W.generate(w, device="cuda")
    bt = d["block_table"].cpu()
    src = int(bt[0, 3])
    q = d["q"][0, :4].float().mean(0)
    d["k_cache"][src, 0, 0] = (8 * q / q.norm()).to(torch.bfloat16)   # page 3: clear winner
    copies = (7, 12, 30, 35, 38)          # six identical top pages for a budget of five
    for j in copies:
        d["k_cache"][int(bt[0, j])] = d["k_cache"][src]
    run = Run(w, data=d)
    s = run.gpu_scores(0, 0)
    # identical records (the builder is deterministic) ...
    r3 = run.summ[int(bt[0, 3]), 0]
    for j in copies:
        assert torch.equal(run.summ[int(bt[0, j]), 0], r3)
    # ... and bit-identical scores, whatever slot of its group of four a page
    # takes (pages 3, 7, 35 sit in slot 3, page 12 in slot 0, 30 and 38 in
    # slot 2): the scorer's arithmetic does not depend on the slot
    for j in copies:
        assert np.array_equal(s[j], s[3]), (j, s[j], s[3])
    sel = run.gpu_selected(0, 0).tolist()
    assert sel == [3, 7, 12, 30, 35]
    check_unit(run, 0, 0)


def test_sparse_with_all_pages_equals_dense():
    w = _w(context=16 * 64 + 9, budget_tokens=16 * 100, seed=31)
    run = Run(w, dense=True)
    for h in range(8):
        np.testing.assert_allclose(run.gpu_out(0, h), run.gpu_out(0, h, dense=True), atol=2e-3)


def test_dense_decode_parity():
    w = _w(batch=2, context=16 * 700 + 3, context_hi=16 * 900, seed=41)
    run = Run(w, dense=True, tail_fill="nan")
    for b in range(2):
        for h in (0, 5):
            L_b = run.lens[b]
            n = L_b // 16
            kc, vc, bt_row = run.unit_cache(b, h, range(n))
            ref = O.dense_attend_unit(run.q_group(b, h), kc, vc, bt_row, 0, L_b, 1 / math.sqrt(128))
            check_attention(run.gpu_out(b, h, dense=True), ref)


def test_repeated_calls_and_graph_capture_are_stable():
    w = _w(context=16 * 500 + 4, seed=51)
    run = Run(w)
    first = run.bufs.out.clone()
    d, H, bufs = run.d, run.H, run.bufs
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            L.locks_score_select(H, d["q"], run.summ, d["block_table"], d["seq_lens"], w.budget_pages,
                                 bufs.selected, bufs.n_selected, bufs.workspace, scores=bufs.scores,
                                 stream=s)
            L.locks_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                  d["seq_lens"], bufs.selected, bufs.n_selected, w.budget_pages,
                                  bufs.out, bufs.workspace, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(first, bufs.out)
    g = torch.cuda.CUDAGraph()
    bufs.out.zero_()
    with torch.cuda.graph(g):
        L.locks_score_select(H, d["q"], run.summ, d["block_table"], d["seq_lens"], w.budget_pages,
                             bufs.selected, bufs.n_selected, bufs.workspace, scores=bufs.scores)
        L.locks_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                              bufs.selected, bufs.n_selected, w.budget_pages, bufs.out, bufs.workspace)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first, bufs.out)
    assert L.locks_read_status(bufs.workspace) == 0


def test_bad_block_ids_are_flagged_not_faulted():
    w = _w(context=16 * 60 + 3, seed=61)
    d = W.generate(w, device="cuda")
    run = Run(w, data=d)
    assert run.status == 0
    bt = d["block_table"].clone()
    bt[0, 5] = d["num_blocks"] + 1000
    bt[0, 9] = -7
    bufs = run.bufs
    L.locks_score_select(8, d["q"], run.summ, bt, d["seq_lens"], w.budget_pages, bufs.selected,
                         bufs.n_selected, bufs.workspace, scores=bufs.scores)
    L.locks_dense_decode(8, d["q"], d["k_cache"], d["v_cache"], bt, d["seq_lens"], bufs.out,
                         bufs.workspace)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) & L.FLAG_BAD_BLOCK
    assert torch.isfinite(bufs.out).all()
