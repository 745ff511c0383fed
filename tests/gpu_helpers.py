"""Shared pieces of the GPU parity tests: run the CUDA path through the C
ABI, move what it saw to the host, and compare with the fp64 oracle.

Tolerances (written here once, used by every GPU test):
  * selected page indices: bit-exact, except pages whose oracle table entry
    lies within REL_BAND (relative) of the k-th value may swap (both choices
    are correct up to fp32 vs fp64 rounding); every such page is counted;
  * page scores s_j: |gpu - oracle| <= SCORE_RTOL * max(1, |oracle|);
  * attention outputs: max |gpu - oracle| <= ATTN_ATOL (fp64 oracle on the
    same bf16 K/V);
  * summaries: integer codes equal to the oracle's (after aligning the sign of
    each basis direction) except within CODE_EDGE of a rounding boundary,
    where +-1 is allowed; reconstruction quality no worse than the oracle's.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

SCORE_RTOL = 1e-3
ATTN_ATOL = 1e-2
REL_BAND = 1e-5
CODE_EDGE = 0.02


class Run:
    """One decode step of a workload on the GPU, with every intermediate kept."""

    def __init__(self, w: W.Workload, tail_fill="zero", build=True, dense=False, data=None, fused=False,
                 step=False, summ=None):
        self.w = w
        self.d = data if data is not None else W.generate(w, device="cuda", tail_fill=tail_fill)
        d = self.d
        H = w.num_kv_heads
        self.H = H
        self.summ = summ if summ is not None else torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8,
                                                              device="cuda")
        self.bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
        if build and summ is None:
            blocks = W.full_page_blocks(d).cuda()
            L.locks_build_summaries(H, d["k_cache"], blocks, self.summ, self.bufs.workspace)
        L.locks_score_select(H, d["q"], self.summ, d["block_table"], d["seq_lens"], w.budget_pages,
                             self.bufs.selected, self.bufs.n_selected, self.bufs.workspace,
                             scores=self.bufs.scores)
        L.locks_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                              self.bufs.selected, self.bufs.n_selected, w.budget_pages, self.bufs.out,
                              self.bufs.workspace)
        self.dense_out = None
        if dense:
            self.dense_out = torch.empty_like(self.bufs.out)
            L.locks_dense_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                 d["seq_lens"], self.dense_out, self.bufs.workspace)
        self.fused = None
        if fused:
            # the fused cluster kernel itself, on the scores locks_score wrote
            f = {"selected": torch.full_like(self.bufs.selected, -1),
                 "n_selected": torch.full_like(self.bufs.n_selected, -1),
                 "out": torch.full_like(self.bufs.out, float("nan"))}
            L.locks_select_sparse_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                         d["seq_lens"], w.budget_pages, f["selected"], f["n_selected"],
                                         f["out"], self.bufs.workspace, scores=self.bufs.scores)
            self.fused = f
        self.step = None
        if step:
            # the whole step through locks_decode_step (either path)
            f = {"selected": torch.full_like(self.bufs.selected, -1),
                 "n_selected": torch.full_like(self.bufs.n_selected, -1),
                 "out": torch.full_like(self.bufs.out, float("nan"))}
            L.locks_decode_step(H, d["q"], self.summ, d["k_cache"], d["v_cache"], d["block_table"],
                                d["seq_lens"], w.budget_pages, f["selected"], f["n_selected"],
                                f["out"], self.bufs.workspace)
            self.step = f
        torch.cuda.synchronize()
        self.status = L.locks_read_status(self.bufs.workspace)
        self.lens = d["seq_lens"].cpu().tolist()
        self.bt = d["block_table"].cpu().numpy()
        self.q = d["q"].double().cpu().numpy()

    # ---- host copies of what one unit needs
    def q_group(self, b, h):
        G = self.w.group
        return self.q[b, h * G:(h + 1) * G]

    def records(self, b, h):
        n = self.lens[b] // 16
        blocks = torch.from_numpy(self.bt[b, :n].astype(np.int64)).cuda()
        return self.summ[blocks, h].cpu().numpy()

    def pages_f64(self, cache, b, h, pages):
        blocks = torch.from_numpy(self.bt[b, np.asarray(pages, dtype=np.int64)].astype(np.int64)).cuda()
        return cache[blocks, h].double().cpu().numpy()

    def unit_cache(self, b, h, pages):
        """Host float64 copies of the listed pages (+ the tail page) of unit (b, h),
        packed as a small cache with its own block table."""
        L_b = self.lens[b]
        n, t = divmod(L_b, 16)
        pages = list(pages)
        plist = pages + ([n] if t else [])
        k = self.pages_f64(self.d["k_cache"], b, h, plist)[:, None]
        v = self.pages_f64(self.d["v_cache"], b, h, plist)[:, None]
        bt_row = np.zeros(n + 1, dtype=np.int64)
        for i, j in enumerate(plist):
            bt_row[j] = i
        return k, v, bt_row

    def gpu_scores(self, b, h):
        n = self.lens[b] // 16
        return self.bufs.scores[b, h, :n].double().cpu().numpy()

    def gpu_selected(self, b, h):
        ns = int(self.bufs.n_selected[b, h])
        return self.bufs.selected[b, h, :ns].cpu().numpy().astype(np.int64)

    def gpu_out(self, b, h, dense=False):
        G = self.w.group
        o = self.dense_out if dense else self.bufs.out
        return o[b, h * G:(h + 1) * G].double().cpu().numpy()


# ------------------------------------------------------------------ comparisons
def check_scores(gpu: np.ndarray, ref: np.ndarray) -> float:
    assert gpu.shape == ref.shape
    err = np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= SCORE_RTOL, f"score rel err {worst}"
    return worst


def check_selection(sel_gpu: np.ndarray, s_hat_gpu: np.ndarray, k: int) -> int:
    """Selection from the GPU's own scores, decided by the oracle in fp64.
    Returns the number of pages inside the tie band (allowed to swap)."""
    sel_or, avg = O.select_pages(s_hat_gpu, k)
    n = s_hat_gpu.shape[0]
    kk = min(k, n)
    assert sel_gpu.size == kk, (sel_gpu.size, kk)
    assert np.all(np.diff(sel_gpu) > 0), "selection not strictly ascending"
    if kk == n or kk == 0:
        assert sel_gpu.tolist() == list(range(n))[:kk]
        return 0
    thr = np.sort(avg)[::-1][kk - 1]
    band = np.abs(avg - thr) <= REL_BAND * thr
    must = set(np.nonzero((avg > thr) & ~band)[0].tolist())
    never = set(np.nonzero((avg < thr) & ~band)[0].tolist())
    got = set(sel_gpu.tolist())
    assert must <= got, f"missing clear winners {sorted(must - got)[:10]}"
    assert not (got & never), f"selected clear losers {sorted(got & never)[:10]}"
    n_band = int(band.sum())
    if n_band <= 1:
        assert sel_gpu.tolist() == sel_or.tolist()
    return n_band


def check_attention(gpu: np.ndarray, ref: np.ndarray) -> float:
    err = float(np.abs(gpu - ref).max())
    assert np.isfinite(gpu).all(), "non-finite attention output"
    assert err <= ATTN_ATOL, f"attention max-abs err {err}"
    return err


def check_unit(run: Run, b: int, h: int, check_scores_too=True):
    """Score, selection and sparse attention of one unit against the oracle."""
    L_b = run.lens[b]
    qg = run.q_group(b, h)
    s_gpu = run.gpu_scores(b, h)
    res = {}
    if check_scores_too and L_b // 16 > 0:
        rec = run.records(b, h)
        d = O.dequantize(O.decode_records(rec))
        s_ref = O.page_scores(qg, d["mu"], d["V"], d["C"])
        res["score_err"] = check_scores(s_gpu, s_ref)
    sel = run.gpu_selected(b, h)
    res["band"] = check_selection(sel, s_gpu, run.w.budget_pages)
    kc, vc, bt_row = run.unit_cache(b, h, sel)
    out_ref = O.sparse_attend_unit(qg, kc, vc, bt_row, 0, L_b, sel, 1 / math.sqrt(128))
    res["attn_err"] = check_attention(run.gpu_out(b, h), out_ref)
    return res


def check_records(gpu_rec: np.ndarray, K_pages: np.ndarray) -> dict:
    """GPU-built records vs the oracle's build of the same bf16 keys."""
    P = K_pages.shape[0]
    summ = O.page_summary(K_pages)
    qo = O.quantize_summary(summ)
    g = O.decode_records(gpu_rec)
    lam = summ["lam"]
    scale = np.maximum(lam[:, :1], 1e-30)
    gaps = -np.diff(lam[:, :9], axis=1) / scale           # gaps among the top 9
    well = np.all(gaps > 1e-3, axis=1) & (lam[:, 7] > 1e-3 * lam[:, 0])
    # scales: the centroid's always, the basis/coefficient ones where the top-9
    # spectrum is well separated (elsewhere individual directions are not unique)
    np.testing.assert_allclose(g["smu"], qo["smu"], rtol=2e-6, atol=1e-30, err_msg="smu")
    for key in ("sV", "sC"):
        np.testing.assert_allclose(g[key][well], qo[key][well], rtol=2e-4, atol=1e-30, err_msg=key)
    np.testing.assert_allclose(g["tail"], summ["tail"], rtol=2e-3, atol=1e-4 * float(lam[:, 0].max()))

    def code_ok(gc, oc_val, s):
        ok = gc == np.rint(oc_val)
        frac = np.abs(np.abs(oc_val - np.floor(oc_val)) - 0.5)
        near = frac < CODE_EDGE
        return ok | (near & (np.abs(gc - oc_val) <= 1.0))

    # centroid codes
    mu_val = summ["mu"] / np.where(qo["smu"] > 0, qo["smu"], 1)[:, None]
    assert np.all(code_ok(g["muq"].astype(np.float64), mu_val, qo["smu"])), "centroid codes"
    # basis / coefficient codes on well-conditioned pages, per-direction sign aligned
    n_well = int(well.sum())
    bad = 0
    for p in np.nonzero(well)[0]:
        Vg = g["Vq"][p].astype(np.float64)
        Cg = g["Cq"][p].astype(np.float64)
        v_val = summ["V"][p] / (qo["sV"][p] if qo["sV"][p] > 0 else 1)
        c_val = summ["C"][p] / (qo["sC"][p] if qo["sC"][p] > 0 else 1)
        for k in range(O.RANK):
            sgn = 1.0 if np.dot(Vg[:, k], v_val[:, k]) >= 0 else -1.0
            if not (np.all(code_ok(sgn * Vg[:, k], v_val[:, k], None)) and
                    np.all(code_ok(sgn * Cg[:, k], c_val[:, k], None))):
                bad += 1
    assert bad == 0, f"{bad} basis directions with codes off by more than rounding"
    # reconstruction: GPU summary at least as good as the oracle's (quantised)
    dg = O.dequantize(g)
    do = O.dequantize(qo)
    Kg = dg["mu"][:, None, :] + dg["C"] @ np.swapaxes(dg["V"], -1, -2)
    Ko = do["mu"][:, None, :] + do["C"] @ np.swapaxes(do["V"], -1, -2)
    eg = np.linalg.norm((K_pages - Kg).reshape(P, -1), axis=1)
    eo = np.linalg.norm((K_pages - Ko).reshape(P, -1), axis=1)
    xn = np.linalg.norm((K_pages - summ["mu"][:, None, :]).reshape(P, -1), axis=1)
    assert np.all(eg <= 1.05 * eo + 1e-3 * xn + 1e-6), f"reconstruction worse: {np.max(eg - eo)}"
    return {"pages": P, "well_conditioned": n_well}


def check_fused_unit(run: Run, b: int, h: int, which: str = "fused"):
    """The fused select + attend pass (which="fused") or the whole decode step
    (which="step") selects exactly what locks_select does (same scores, same
    selection) and its output matches the oracle's attention over that
    selection."""
    f = run.fused if which == "fused" else run.step
    ns = int(f["n_selected"][b, h])
    sel_f = f["selected"][b, h, :ns].cpu().numpy().astype(np.int64)
    assert sel_f.tolist() == run.gpu_selected(b, h).tolist()
    L_b = run.lens[b]
    qg = run.q_group(b, h)
    kc, vc, bt_row = run.unit_cache(b, h, sel_f)
    ref = O.sparse_attend_unit(qg, kc, vc, bt_row, 0, L_b, sel_f, 1 / math.sqrt(128))
    G = run.w.group
    out = f["out"][b, h * G:(h + 1) * G].double().cpu().numpy()
    return check_attention(out, ref)
