"""The shared-projection ablation on the GPU path: "LOCKS: Page-Local Compact
Key Summaries for Efficient Long-Context Decoding", technical summary §3
("impossibility of shared projections").

One rank-rho basis per KV head (the top principal directions of all of the
head's centred keys, computed here with torch in fp64 and passed in as fp32)
scores every page through locks_shared_basis_build / locks_shared_basis_score,
and the library's own selection ranks those scores.  Checks:
  * parity: the GPU scores equal the score equation evaluated in fp64 on the
    same basis (centroid term + log-sum-exp of the coefficients' logits);
  * the selection is exact on those scores (same tie band as elsewhere);
  * carrier retention collapses: of the pages holding a planted key along the
    group's mean query, the shared basis keeps at most half, while the
    library's page-local summaries keep what reading every key keeps."""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import SCORE_RTOL, Run, check_selection

pytestmark = pytest.mark.gpu


def _basis(K_all: np.ndarray, rho: int) -> np.ndarray:
    """Top-rho principal directions of a head's centred keys, [128, rho]."""
    X = K_all - K_all.mean(axis=1, keepdims=True)
    flat = torch.from_numpy(X.reshape(-1, X.shape[-1]))
    lam, U = torch.linalg.eigh(flat.T @ flat)
    return U.flip(-1)[:, :rho].numpy()


@pytest.mark.parametrize("rho", [8, 32])
def test_shared_basis_scores_parity_and_carrier_collapse(rho):
    w = W.Workload(name="ablation_gpu", batch=1, context=16 * 256, num_kv_heads=2, group=4,
                   budget_tokens=16 * 16, carriers_per_head=8, seed=23)
    run = Run(w, step=True)          # the page-local path, for comparison
    d = run.d
    H, k = w.num_kv_heads, w.budget_pages
    n = run.lens[0] // 16
    pages = {h: run.pages_f64(d["k_cache"], 0, h, range(n)) for h in range(H)}   # logical order
    basis = np.ascontiguousarray(np.stack([_basis(pages[h], rho) for h in range(H)]).astype(np.float32))
    basis_t = torch.from_numpy(basis).cuda().contiguous()
    rec = torch.zeros(d["num_blocks"], H, L.shared_basis_record_bytes(rho), dtype=torch.uint8, device="cuda")
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    L.locks_shared_basis_build(H, d["k_cache"], W.full_page_blocks(d).cuda(), basis_t, rec, bufs.workspace)
    L.locks_shared_basis_score(H, d["q"], basis_t, rec, d["block_table"], d["seq_lens"], bufs.workspace,
                               scores=bufs.scores)
    L.locks_select(H, d["seq_lens"], w.max_pages, k, bufs.selected, bufs.n_selected, bufs.workspace,
                   scores=bufs.scores)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    for h in range(H):
        K = pages[h]
        qg = run.q_group(0, h)
        U = basis[h].astype(np.float64)
        mu = K.mean(axis=1)
        C = (K - mu[:, None, :]) @ U
        want = O.page_scores(qg, mu, np.broadcast_to(U, (n,) + U.shape), C)
        got = bufs.scores[0, h, :n].double().cpu().numpy()
        assert np.max(np.abs(got - want) / np.maximum(1.0, np.abs(want))) <= SCORE_RTOL
        sel_shared = bufs.selected[0, h, :int(bufs.n_selected[0, h])].cpu().numpy().astype(np.int64)
        check_selection(sel_shared, got, k)
        carriers = {j for (b, hh, j, s) in d["carriers"] if b == 0 and hh == h}
        exact, _ = O.select_pages(O.exact_page_lse(qg, K), k)
        local = set(run.step["selected"][0, h, :int(run.step["n_selected"][0, h])].cpu().tolist())
        kept = {name: len(carriers & set(s)) / len(carriers) for name, s in
                (("exact", exact.tolist()), ("local", local), ("shared", sel_shared.tolist()))}
        msg = f"h={h} rank-{rho} shared basis: carriers kept {kept}"
        print(msg)
        assert kept["exact"] >= 0.75, msg
        assert kept["local"] >= kept["exact"] - 0.125, msg
        assert kept["shared"] <= 0.5 and kept["shared"] <= kept["local"] - 0.4, msg
