"""End-to-end selection overlap between summaries the oracle builds and the
summaries the GPU builds, on the headline workload (one request, 128K tokens,
8 KV heads, 2,048-token budget).

The GPU builder runs fp32 Jacobi and the oracle fp64 LAPACK, so a record's
codes may differ by one at a rounding edge, and a page near the selection
boundary may swap.  Both pipelines are otherwise independent: the oracle
builds, scores and selects from the bf16 keys on the CPU; the GPU builds,
scores and selects through the C ABI.  The overlap |S_gpu & S_oracle| / k is
reported per KV head (the parity bar is per stage and lives in the other
tests; this is the whole-path agreement)."""

import numpy as np
import pytest

import oracle as O
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run

pytestmark = pytest.mark.gpu


def test_selection_overlap_oracle_built_vs_gpu_built_records():
    w = W.CONFIGS["llama8b_128k"]
    run = Run(w, step=True)
    assert run.status == 0
    n = run.lens[0] // 16
    k = w.budget_pages
    overlaps = []
    for h in range(w.num_kv_heads):
        K = run.pages_f64(run.d["k_cache"], 0, h, range(n))           # [n, 16, 128], logical order
        dq = O.dequantize(O.decode_records(O.build_records(K)))
        s_or = O.page_scores(run.q_group(0, h), dq["mu"], dq["V"], dq["C"])
        sel_or, _ = O.select_pages(s_or, k)
        sel_gpu = run.step["selected"][0, h, :int(run.step["n_selected"][0, h])].cpu().numpy()
        ov = len(set(sel_or.tolist()) & set(sel_gpu.tolist())) / k
        overlaps.append(ov)
        print(f"llama8b_128k h={h}: selection overlap oracle-built vs GPU-built records {ov:.4f}")
    print(f"llama8b_128k: mean overlap {np.mean(overlaps):.4f}, min {np.min(overlaps):.4f}")
    assert np.mean(overlaps) >= 0.95 and np.min(overlaps) >= 0.9, overlaps
