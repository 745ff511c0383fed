"""Unquantised fp32 summaries (cfg quant = 0, rank r <= 16) through the
library's builder and scorer.

At r = 16 a page's record reproduces its 16 keys exactly (the centred keys
have rank <= 15), so by the score equation of the technical summary §2
("Reconstruction and selection") s_j(q) must equal the exact page
log-sum-exp log sum_i exp(q.k_i / sqrt(d)): a closed form that pins the CUDA
scoring arithmetic (centroid term, V^T q, the coefficients' logits and the
log-sum-exp) without the oracle's scorer.  At r = 8 the fp32 records and
scores match the oracle's unquantised rank-8 summary of the same keys, and a
whole decode step at r = 16 selects the pages the read-every-key masses
select."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import check_attention, check_selection

pytestmark = pytest.mark.gpu


def _build(w, d, rank, q_scale=1.0):
    H = w.num_kv_heads
    if q_scale != 1.0:
        d["q"] = (d["q"].float() * q_scale).to(torch.bfloat16)
    summ = torch.zeros(d["num_blocks"], H, L.record_bytes(0, rank), dtype=torch.uint8, device="cuda")
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ, bufs.workspace, quant=0, rank=rank)
    L.locks_score(H, d["q"], summ, d["block_table"], d["seq_lens"], bufs.workspace, scores=bufs.scores,
                  quant=0, rank=rank)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    return summ, bufs


def _unit_pages(d, b, h):
    n = int(d["seq_lens"][b]) // 16
    blocks = d["block_table"][b, :n].long()
    return blocks, d["k_cache"][blocks, h].double().cpu().numpy()


def _records(summ, blocks, h, rank):
    rec = summ[blocks, h].cpu().numpy().view(np.float32).astype(np.float64)
    mu = rec[:, :128]
    V = rec[:, 128:128 + 128 * rank].reshape(-1, 128, rank)
    C = rec[:, 128 + 128 * rank:128 + 144 * rank].reshape(-1, 16, rank)
    tail = rec[:, 128 + 144 * rank]
    return mu, V, C, tail


@pytest.mark.parametrize("regime,q_scale", [("fullrank", 1.0), ("lowrank", 1.0), ("fullrank", 8.0)])
def test_full_rank_scores_equal_exact_page_lse(regime, q_scale):
    w = W.Workload("fp32_r16", batch=2, context=16 * 300 + 5, context_hi=16 * 340 + 3, num_kv_heads=2, group=4,
                   budget_tokens=16 * 16, carriers_per_head=3, key_regime=regime, seed=61)
    d = W.generate(w, device="cuda")
    summ, bufs = _build(w, d, 16, q_scale)
    worst = 0.0
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            blocks, K = _unit_pages(d, b, h)
            q = d["q"][b, h * 4:(h + 1) * 4].double().cpu().numpy()
            exact = O.exact_page_lse(q, K)
            got = bufs.scores[b, h, :K.shape[0]].double().cpu().numpy()
            err = np.abs(got - exact) / np.maximum(1.0, np.abs(exact))
            worst = max(worst, float(err.max()))
            # the record itself reproduces the keys
            mu, V, C, tail = _records(summ, blocks, h, 16)
            Khat = mu[:, None, :] + np.einsum("pir,pdr->pid", C, V)
            scale = np.abs(K).max()
            assert np.abs(Khat - K).max() <= 1e-4 * scale, "r = 16 records do not reproduce the keys"
            assert np.all(tail == 0.0)   # no eigenvalue lies beyond r = 16
    assert worst <= 1e-4, f"score vs exact page LSE: {worst}"


def test_rank8_fp32_records_match_oracle_unquantised_summary():
    w = W.Workload("fp32_r8", batch=1, context=16 * 500 + 9, num_kv_heads=2, group=4, budget_tokens=16 * 16,
                   carriers_per_head=4, seed=62)
    d = W.generate(w, device="cuda")
    summ, bufs = _build(w, d, 8)
    for h in range(w.num_kv_heads):
        blocks, K = _unit_pages(d, 0, h)
        ref = O.page_summary(K, rank=8)
        mu, V, C, tail = _records(summ, blocks, h, 8)
        np.testing.assert_allclose(mu, ref["mu"], atol=1e-6)
        # the rank-8 projection of each page (sign-free), and the tail energy
        P_gpu = np.einsum("pir,pdr->pid", C, V)
        P_ref = np.einsum("pir,pdr->pid", ref["C"], ref["V"])
        np.testing.assert_allclose(P_gpu, P_ref, atol=2e-3 * np.abs(P_ref).max())
        np.testing.assert_allclose(tail, ref["tail"], rtol=2e-3, atol=1e-4 * ref["lam"][:, 0].max())
        q = d["q"][0, h * 4:(h + 1) * 4].double().cpu().numpy()
        s_ref = O.page_scores(q, ref["mu"], ref["V"], ref["C"])
        got = bufs.scores[0, h, :K.shape[0]].double().cpu().numpy()
        assert np.max(np.abs(got - s_ref) / np.maximum(1.0, np.abs(s_ref))) <= 1e-3


def test_decode_step_at_full_rank_selects_by_exact_page_mass():
    w = W.Workload("fp32_step", batch=2, context=16 * 900 + 7, context_hi=16 * 1000 + 2, num_kv_heads=8, group=4,
                   budget_tokens=16 * 32, carriers_per_head=4, seed=63)
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    summ = torch.zeros(d["num_blocks"], H, L.record_bytes(0, 16), dtype=torch.uint8, device="cuda")
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    # page-crossing builder with a device count, over all full pages
    blocks = W.full_page_blocks(d).cuda()
    n_dev = torch.tensor([blocks.numel()], dtype=torch.int32, device="cuda")
    L.locks_build_pending(H, d["k_cache"], blocks, n_dev, summ, bufs.workspace, quant=0, rank=16)
    L.locks_decode_step(H, d["q"], summ, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                        w.budget_pages, bufs.selected, bufs.n_selected, bufs.out, bufs.workspace,
                        scores=bufs.scores, quant=0, rank=16)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    bt = d["block_table"].cpu().numpy()
    for b in range(w.batch):
        L_b = int(d["seq_lens"][b])
        n = L_b // 16
        for h in (0, 3, 7):
            blocks_u, K = _unit_pages(d, b, h)
            q = d["q"][b, h * 4:(h + 1) * 4].double().cpu().numpy()
            exact = O.exact_page_lse(q, K)
            sel = bufs.selected[b, h, :int(bufs.n_selected[b, h])].cpu().numpy().astype(np.int64)
            # exact against the GPU's own scores ...
            check_selection(sel, bufs.scores[b, h, :n].double().cpu().numpy(), w.budget_pages)
            # ... and, beyond the scores' fp32 rounding, the read-every-key selection
            _, table = O.select_pages(exact, w.budget_pages)
            kth = np.sort(table)[::-1][w.budget_pages - 1]
            got = set(sel.tolist())
            assert set(np.nonzero(table > kth * (1 + 1e-3))[0].tolist()) <= got
            assert not (set(np.nonzero(table < kth * (1 - 1e-3))[0].tolist()) & got)
            pages = list(sel) + ([n] if L_b % 16 else [])
            kc = d["k_cache"][torch.from_numpy(bt[b, pages].astype(np.int64)).cuda(), h].double().cpu().numpy()
            vc = d["v_cache"][torch.from_numpy(bt[b, pages].astype(np.int64)).cuda(), h].double().cpu().numpy()
            row = np.zeros(n + 1, dtype=np.int64)
            for i, j in enumerate(pages):
                row[j] = i
            ref = O.sparse_attend_unit(q, kc[:, None], vc[:, None], row, 0, L_b, sel, 1 / math.sqrt(128))
            check_attention(bufs.out[b, h * 4:(h + 1) * 4].double().cpu().numpy(), ref)
