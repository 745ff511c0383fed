"""Decode steps over a spread of shapes the named workloads do not cover:
KV-head counts 4 and 16 (16 splits a scoring CTA's heads into two groups),
one to five requests of ragged lengths with every tail length class (0, 1,
15 and in between), budgets below and above a request's page count, and
NaN in the unwritten tail slots.  Each shape runs the separate path (score
+ select, split-K attention), the fused select + attention kernel on the
same scores, and locks_decode_step; every unit is checked against the
oracle (scores on the GPU-built records, selection from the GPU scores,
attention over the GPU selection), and the other two paths against it
("LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
Decoding", technical summary §2)."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run, check_attention, check_selection, check_unit

pytestmark = pytest.mark.gpu

# (batch, context N, upper N for ragged batches, KV heads, budget pages, seed);
# a request holds L = N + 1 tokens (its current token appended)
SHAPES = [
    (1, 16 * 700 + 9, None, 16, 40, 101),
    (1, 16 * 900 - 1, None, 4, 64, 102),        # tail 0: the current token completed the page
    (1, 16 * 1000 + 14, None, 16, 128, 103),    # tail 15
    (1, 16 * 33 + 1, None, 16, 40, 104),        # fewer pages than the budget
    (3, 16 * 300, 16 * 900 + 15, 16, 64, 105),
    (2, 16 * 1200 + 1, 16 * 2500, 4, 128, 106),
    (5, 16 * 20 + 3, 16 * 400, 4, 24, 107),
    (4, 16 * 2000, 16 * 2600 + 7, 8, 100, 108),
    (2, 16 * 50, 16 * 70 + 1, 16, 128, 109),    # budget above every request's page count
]


def _check_path(run, b, h, f):
    """Another path's selection and output for unit (b, h): the selection
    from the separate path's GPU scores, the output against the oracle over
    that path's own selection."""
    got = f["selected"][b, h, :int(f["n_selected"][b, h])].cpu().numpy().astype(np.int64)
    check_selection(got, run.gpu_scores(b, h), run.w.budget_pages)
    kc, vc, bt_row = run.unit_cache(b, h, got)
    ref = O.sparse_attend_unit(run.q_group(b, h), kc, vc, bt_row, 0, run.lens[b], got, 1 / math.sqrt(128))
    G = run.w.group
    check_attention(f["out"][b, h * G:(h + 1) * G].double().cpu().numpy(), ref)


@pytest.mark.parametrize("batch,ctx,ctx_hi,H,k,seed", SHAPES)
def test_shapes_all_paths_against_the_oracle(batch, ctx, ctx_hi, H, k, seed):
    w = W.Workload(f"shape{seed}", batch=batch, context=ctx, context_hi=ctx_hi, num_kv_heads=H, group=4,
                   budget_tokens=16 * k, carriers_per_head=2, seed=seed)
    run = Run(w, tail_fill="nan", fused=True, step=True)
    assert run.status == 0
    for b in range(batch):
        for h in range(H):
            check_unit(run, b, h)
            _check_path(run, b, h, run.fused)
            _check_path(run, b, h, run.step)
    assert torch.isfinite(run.step["out"]).all() and torch.isfinite(run.fused["out"]).all()
    print(f"shape {seed}: lengths {run.lens}, tails {sorted({L % 16 for L in run.lens})}")
