"""Ablation for "LOCKS: Page-Local Compact Key Summaries for Efficient
Long-Context Decoding", technical summary §3 ("impossibility of shared
projections"): a fixed, query-independent low-rank projection shared by all of
a head's pages cannot see within-page directions outside its span.  On pages
with planted carrier keys (one key per page along the group's mean query), a
selector that scores every page through one shared rank-8 basis (the top
principal directions of all of the head's centred keys) loses the carriers,
while the page-local summaries keep them, as does reading every key.

CPU only: the fp64 oracle for the page-local side, numpy for the ablation."""

import numpy as np
import pytest

import oracle as O
from sparse_long_context_locks_gb300 import workload as W


def _shared_basis_scores(qg: np.ndarray, K: np.ndarray, rho: int) -> np.ndarray:
    """s_j through one basis U for all pages: mu_j + (k_i - mu_j) U U^T."""
    mu = K.mean(axis=1)
    X = K - mu[:, None, :]
    flat = X.reshape(-1, K.shape[-1])
    lam, U = np.linalg.eigh(flat.T @ flat)
    U = U[:, ::-1][:, :rho]                                   # top-rho directions
    C = X @ U                                                 # [P, 16, rho]
    V = np.broadcast_to(U, (K.shape[0],) + U.shape)
    return O.page_scores(qg, mu, V, C)


def _retention(sel: np.ndarray, carrier_pages: set) -> float:
    return len(carrier_pages & set(sel.tolist())) / len(carrier_pages)


@pytest.mark.parametrize("h", [0, 1])
@pytest.mark.parametrize("rho", [8, 32])
def test_shared_basis_loses_the_carriers_page_local_keeps_them(h, rho):
    w = W.Workload(name="ablation", batch=1, context=16 * 256, num_kv_heads=2, group=4,
                   budget_tokens=16 * 16, carriers_per_head=8, seed=23)
    d = W.generate(w, device="cpu")
    n = (w.context + 1) // 16
    bt = d["block_table"][0, :n].numpy()
    K = d["k_cache"][bt, h].double().numpy()                  # [n, 16, 128], logical page order
    qg = d["q"][0, h * 4:(h + 1) * 4].double().numpy()
    carriers = {j for (b, hh, j, s) in d["carriers"] if b == 0 and hh == h}
    k = w.budget_pages

    exact, _ = O.select_pages(O.exact_page_lse(qg, K), k)
    summ = O.dequantize(O.quantize_summary(O.page_summary(K)))
    local, _ = O.select_pages(O.page_scores(qg, summ["mu"], summ["V"], summ["C"]), k)
    shared, _ = O.select_pages(_shared_basis_scores(qg, K, rho=rho), k)

    r_exact, r_local, r_shared = (_retention(s, carriers) for s in (exact, local, shared))
    msg = f"carriers kept: exact {r_exact:.2f}, page-local {r_local:.2f}, shared rank-{rho} {r_shared:.2f}"
    # page-local summaries keep what reading every key keeps (within one
    # carrier of eight); one shared basis, even of rank 32, loses most
    assert r_exact >= 0.75, msg
    assert r_local >= r_exact - 0.125, msg
    assert r_shared <= 0.5 and r_shared <= r_local - 0.4, msg
