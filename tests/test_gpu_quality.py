"""Selection quality of the CUDA path, reported (the pages' claim, not a
parity bar): "LOCKS: Page-Local Compact Key Summaries for Efficient
Long-Context Decoding", abstract and technical summary §2 -- the summaries
should pick the pages that carry the attention mass.

Per unit (request, KV head) of a workload, after one locks_decode_step:
  * recall: the share of the k pages with the largest exact page masses
    (every key read, fp64, grouped the same way) that the GPU selected;
  * carrier retention: the share of the planted carrier pages (one key along
    the group's mean query, in pages the low-rank background would not rank)
    that the GPU selected, next to the share exact selection keeps.
The figures are printed; the bounds only catch a broken path (they sit well
below the measured values)."""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run

pytestmark = pytest.mark.gpu


def _unit_quality(run: Run, b: int, h: int) -> dict:
    n = run.lens[b] // 16
    k = run.w.budget_pages
    K = run.pages_f64(run.d["k_cache"], b, h, range(n))          # [n, 16, 128], logical order
    exact, _ = O.select_pages(O.exact_page_lse(run.q_group(b, h), K), k)
    got = set(run.step["selected"][b, h, :int(run.step["n_selected"][b, h])].cpu().tolist())
    car = {j for (bb, hh, j, s) in run.d["carriers"] if bb == b and hh == h}
    res = {"recall": len(got & set(exact.tolist())) / max(1, min(k, n))}
    if car:
        res["carriers"] = len(car)
        res["kept_gpu"] = len(car & got)
        res["kept_exact"] = len(car & set(exact.tolist()))
    return res


@pytest.mark.parametrize("name,units", [
    ("llama8b_128k", [(0, h) for h in range(8)]),
    ("batch16_32k", [(0, 0), (5, 3), (11, 6), (15, 7)]),
])
def test_selection_recall_and_carrier_retention(name, units):
    run = Run(W.CONFIGS[name], step=True)
    assert run.status == 0
    rows = [(b, h, _unit_quality(run, b, h)) for b, h in units]
    for b, h, r in rows:
        print(f"{name} b={b} h={h}: recall {r['recall']:.3f}, carriers kept "
              f"{r.get('kept_gpu', 0)}/{r.get('carriers', 0)} (exact selection {r.get('kept_exact', 0)})")
    recall = np.mean([r["recall"] for _, _, r in rows])
    print(f"{name}: mean recall {recall:.3f}")
    assert recall >= 0.8, recall
    for b, h, r in rows:
        assert r["recall"] >= 0.7, (b, h, r)
        if "carriers" in r:
            # the summaries keep what reading every key keeps, within one carrier
            assert r["kept_gpu"] >= r["kept_exact"] - 1, (b, h, r)
