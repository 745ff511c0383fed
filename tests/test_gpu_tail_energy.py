"""The spectral tail energy the builder stores with every record (sum of the
Gram eigenvalues beyond rank 8; "LOCKS: Page-Local Compact Key Summaries for
Efficient Long-Context Decoding", technical summary §3, Thm. 1: the error of a
page's reconstruction is controlled by that energy) tracks how far the page's
summary score lies from its exact log page mass."""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run

pytestmark = pytest.mark.gpu


def _ranks(x):
    r = np.empty(len(x))
    r[np.argsort(x, kind="stable")] = np.arange(len(x))
    return r


def test_tail_energy_orders_the_score_error():
    w = W.Workload(name="t", batch=1, context=16 * 400, num_kv_heads=2, group=4,
                   budget_tokens=16 * 16, carriers_per_head=0, seed=17)
    d = W.generate(w, device="cuda")
    n = (w.context + 1) // 16
    bt = d["block_table"][0, :n].long()
    # per-page noise from 1e-3 to 1 (log-uniform) on top of the low-rank keys
    g = torch.Generator(device="cuda").manual_seed(5)
    sigma = torch.exp(torch.empty(n, device="cuda").uniform_(np.log(1e-3), 0.0, generator=g))
    noise = torch.randn(n, 2, 16, 128, device="cuda", generator=g) * sigma[:, None, None, None]
    d["k_cache"][bt] = (d["k_cache"][bt].float() + noise).to(torch.bfloat16)
    run = Run(w, data=d)
    assert run.status == 0
    for h in range(2):
        rec = run.records(0, h)
        tail = O.decode_records(rec)["tail"]
        K = run.pages_f64(d["k_cache"], 0, h, np.arange(n))
        qg = run.q_group(0, h)
        err = np.abs(run.gpu_scores(0, h) - O.exact_page_lse(qg, K)).mean(axis=1)
        # Spearman rank correlation; below a noise of a few 1e-2 the int4/int8
        # quantisation error, which the tail energy does not see, sets a floor
        rho = np.corrcoef(_ranks(tail), _ranks(err))[0, 1]
        lo, hi = np.argsort(tail)[: n // 10], np.argsort(tail)[-(n // 10):]
        ratio = err[hi].mean() / err[lo].mean()
        msg = f"head {h}: rank correlation {rho:.2f}, top/bottom decile error ratio {ratio:.1f}"
        assert rho > 0.3, msg
        assert ratio > 4.0, msg
