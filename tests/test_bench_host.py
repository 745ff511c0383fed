"""bench.py's host-side clock record (CPU only): the nvidia-smi lines it
parses and the summary that goes into the JSON line (median SM clock under
load, the maximum clock, and every throttle reason seen active)."""

import io
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(sm, mx, power, util=100, hw="Not Active", hw_th="Not Active", sw_th="Not Active",
          sw_pw="Not Active"):
    # --query-gpu=timestamp,index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,active,
    #             hw,hw_thermal,sw_thermal,sw_power   (--format=csv,noheader,nounits)
    return f"2026/12/03 01:00:00.000, 0, {sm}, {mx}, {power}, {util}, 0x0, {hw}, {hw_th}, {sw_th}, {sw_pw}\n"


def _parse(lines):
    s = bench.ClockSampler(0)
    s.proc = type("P", (), {"stdout": io.StringIO("".join(lines))})()
    s._read()
    return s.rows


def test_rows_parsed_and_malformed_lines_skipped():
    rows = _parse([_line(2070, 2070, 900.5), "garbage\n", _line("[N/A]", 2070, 10.0), _line(1980, 2070, 1200)])
    assert [r["sm"] for r in rows] == [2070.0, 1980.0]
    assert rows[1]["power"] == 1200.0 and rows[0]["max"] == 2070.0 and rows[0]["util"] == 100.0


def test_summary_median_max_and_active_reasons():
    rows = _parse([_line(2070, 2070, 800), _line(1800, 2070, 1300, sw_pw="Active"),
                   _line(2070, 2070, 900, util=97), _line(1500, 2100, 1400, hw_th="Active"),
                   _line(345, 2070, 120.0, util=0),            # idle samples: not under load
                   _line(1000, 2070, 300.0, util=12, sw_th="Active")])
    s = bench.ClockSampler.summary(rows)
    assert s["samples"] == 6 and s["samples_under_load"] == 4
    assert s["sm_mhz"] == 2070.0          # upper median of 1500, 1800, 2070, 2070
    assert s["sm_max_mhz"] == 2100.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]   # the idle sample's is left out


def test_summary_with_no_sample_under_load_uses_all():
    rows = _parse([_line(345, 2070, 120.0, util=0), _line(400, 2070, 130.0, util=3)])
    s = bench.ClockSampler.summary(rows)
    assert s["samples"] == 2 and s["samples_under_load"] == 0
    assert s["sm_mhz"] == 400.0


def test_summary_without_samples_says_so():
    s = bench.ClockSampler.summary([])
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == ["no samples"]
    assert s["samples_under_load"] == 0


def test_cpu_baseline_unit_runs_the_whole_oracle_path(tmp_path):
    """The timed CPU baseline's unit of work is the oracle's score, select and
    attend of one (request, KV head), on the host copies bench.py writes."""
    import numpy as np
    import torch

    import oracle as O
    from sparse_long_context_locks_gb300 import workload as W

    w = W.Workload("tiny", batch=2, context=700, context_hi=900, num_kv_heads=2, group=4,
                   budget_tokens=16 * 6, carriers_per_head=2, seed=5)
    d = W.generate(w, device="cpu")
    kc = d["k_cache"].float().numpy()
    summ = torch.from_numpy(O.build_records(kc.astype(np.float64)))
    bench.oracle_host_copy(d, summ, str(tmp_path))
    want = O.decode_step(d["q"].float().numpy(), kc, d["v_cache"].float().numpy(),
                         d["block_table"].numpy().astype(np.int64), d["seq_lens"].numpy(),
                         summ.numpy(), w.num_kv_heads, w.group, w.budget_pages)
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            secs, abs_sum = bench._oracle_unit((str(tmp_path), b, h, w.group, w.budget_pages))
            assert secs > 0
            assert abs_sum == float(np.abs(want[(b, h)]["out"]).sum())


def test_selection_quality_against_the_oracles_exact_selection():
    """bench.py's reported selection quality (torch, every key read) on a
    tiny CPU workload: the oracle's exact-mass selection scores recall 1 and
    keeps what it keeps; selecting the lowest pages instead scores the recall
    of that set against the oracle's."""
    import numpy as np
    import torch
    import oracle as O
    from sparse_long_context_locks_gb300 import workload as W
    w = W.Workload("q", batch=2, context=16 * 40 + 3, context_hi=16 * 60, num_kv_heads=2, group=4,
                   budget_tokens=16 * 8, carriers_per_head=3, seed=4)
    d = W.generate(w, device="cpu")
    H, G, k = w.num_kv_heads, w.group, w.budget_pages
    sel = torch.full((w.batch, H, k), -1, dtype=torch.int32)
    nsel = torch.zeros(w.batch, H, dtype=torch.int32)
    low = torch.full_like(sel, -1)
    exact_sets = {}
    for b in range(w.batch):
        n = int(d["seq_lens"][b]) // 16
        blocks = d["block_table"][b, :n].long()
        for h in range(H):
            K = d["k_cache"][blocks, h].double().numpy()
            q = d["q"][b, h * G:(h + 1) * G].double().numpy()
            ex, _ = O.select_pages(O.exact_page_lse(q, K), k)
            exact_sets[(b, h)] = set(ex.tolist())
            sel[b, h, :len(ex)] = torch.from_numpy(ex.astype(np.int32))
            nsel[b, h] = len(ex)
            low[b, h, :len(ex)] = torch.arange(len(ex), dtype=torch.int32)
    q1 = bench.selection_quality(w, d, sel, nsel)
    assert q1["recall_vs_exact_mass"] == 1.0 and q1["min_recall"] == 1.0
    assert q1["carriers_kept"] == q1["carriers_kept_by_exact"] and q1["carriers"] == w.batch * H * 3
    q2 = bench.selection_quality(w, d, low, nsel)
    want = np.mean([len(exact_sets[(b, h)] & set(range(k))) / k for b in range(w.batch) for h in range(H)])
    assert abs(q2["recall_vs_exact_mass"] - want) < 1e-12
