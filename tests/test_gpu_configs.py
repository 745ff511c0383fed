"""GPU parity on the five named workloads at full size, in the launch
configuration bench.py times.  The oracle checks every unit where that is
cheap and sampled (request, KV head) units where the cache is too large to
check whole (batch 16: 4 requests x 8 heads; batch 64: 3 requests x 8 heads);
the builder is checked on sampled pages."""

import gc

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run, check_fused_unit, check_records, check_unit

pytestmark = pytest.mark.gpu


def _check_build_sample(run, b, h, n_pages, rng):
    n = run.lens[b] // 16
    pages = np.sort(rng.choice(n, size=min(n_pages, n), replace=False))
    K = run.pages_f64(run.d["k_cache"], b, h, pages)
    blocks = torch.from_numpy(run.bt[b, pages].astype(np.int64)).cuda()
    rec = run.summ[blocks, h].cpu().numpy()
    return check_records(rec, K)


def _free(run):
    del run.d, run.summ, run.bufs
    gc.collect()
    torch.cuda.empty_cache()


def test_pr1_4k():
    run = Run(W.CONFIGS["pr1_4k"], dense=True)
    assert run.status == 0
    check_unit(run, 0, 0)


def test_llama8b_128k_all_heads():
    run = Run(W.CONFIGS["llama8b_128k"])
    assert run.status == 0
    rng = np.random.default_rng(0)
    for h in range(8):
        check_unit(run, 0, h)
    _check_build_sample(run, 0, 3, 1024, rng)
    _free(run)


def test_batch16_32k_sampled_requests():
    w = W.CONFIGS["batch16_32k"]
    run = Run(w, tail_fill="nan")
    assert run.status == 0
    assert len(set(run.lens)) > 1
    for b in (0, 5, 10, 15):
        for h in range(8):
            check_unit(run, b, h)
    _free(run)


def test_ctx1m_all_heads():
    run = Run(W.CONFIGS["ctx1m"])
    assert run.status == 0
    rng = np.random.default_rng(1)
    for h in range(8):
        check_unit(run, 0, h, check_scores_too=(h in (0, 5)))
    _check_build_sample(run, 0, 6, 2048, rng)
    lens = run.lens
    by = W.algorithmic_bytes(lens, 8, 4, run.w.budget_pages)
    assert by["dense_kv"] / (by["score"] + by["sparse_kv"]) >= 9.0
    _free(run)


def test_staged_selection_ragged_requests():
    """Requests of 70K-300K tokens: 2,344-page slices per selecting CTA, so
    the selection kernel copies each CTA's scores to shared memory first; the
    shorter requests leave slices with ragged ends and under 1,024 pages."""
    w = W.Workload("ragged_300k", batch=3, context=70000, context_hi=300000, num_kv_heads=8, group=4,
                   budget_tokens=2048, carriers_per_head=8, seed=105)
    run = Run(w)
    assert run.status == 0
    assert len(set(run.lens)) == 3 and min(run.lens) // 16 < 8 * 1024 < w.max_pages
    for b in range(w.batch):
        for h in range(8):
            check_unit(run, b, h, check_scores_too=(h == b))
    _free(run)


@pytest.mark.parametrize("regime", ["batch64_256k_lowrank", "batch64_256k_fullrank"])
def test_batch64_256k_sampled_requests(regime):
    run = Run(W.CONFIGS[regime])
    assert run.status == 0
    rng = np.random.default_rng(2)
    for b in (0, 31, 63):
        for h in range(8):
            check_unit(run, b, h, check_scores_too=(h % 4 == 0))
    _check_build_sample(run, 17, 2, 512, rng)
    _free(run)


def test_maximum_context_and_budget():
    """The largest request the fused step accepts: 131,072 pages (2,097,151
    tokens, so a 15-token tail), each selecting CTA's 16,384 keys and block ids
    filling its 128 KB ring, and a 2,047-page budget (32 items for each of the
    cluster's 64 warps with the tail).  Scores of one head against the oracle,
    every head's selection from its scores and the step's attention."""
    w = W.Workload("max_2m", batch=1, context=16 * 131072 - 1, num_kv_heads=8, group=4,
                   budget_tokens=16 * 2047, carriers_per_head=16, seed=77)
    assert w.max_pages == 131072 and w.budget_pages == 2047
    run = Run(w, step=True)
    assert run.status == 0
    rng = np.random.default_rng(3)
    for h in range(8):
        check_unit(run, 0, h, check_scores_too=(h == 3))
        check_fused_unit(run, 0, h, which="step")
    _check_build_sample(run, 0, 1, 1024, rng)
    _free(run)
