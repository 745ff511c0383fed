"""The selection kernel on long requests, with score tables planted straight
into the table (LOCKS summary §2: per-head normalisation, group mean, top-k,
lower page index first on ties).

Past 2,048 pages a CTA of an 8-CTA cluster (more than 256K tokens a request)
the kernel runs 16-CTA clusters when they are all resident at once, else
8-CTA ones; these cases cover both (batch 1 and 2 take 16, batch 3 takes 8),
with every CTA's slice holding boundary candidates:
  * distinct scores: the oracle's fp64 selection, exact outside the tie band;
  * one row copied to pages all over the request, straddling the budget
    boundary, in a boundary bin small enough to be ranked member by member
    (40 copies) and in one that needs every histogram level (5,000 copies):
    the clear winners plus the lowest-index copies."""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import locks as L

from gpu_helpers import check_selection

pytestmark = pytest.mark.gpu

H = 8
K = 128                         # 2,048-token budget


def _run(tables, lens, max_pages):
    B = len(lens)
    bufs = L.DecodeBuffers(H, B, max_pages, K)
    bufs.scores.fill_(float("nan"))
    for b, t in enumerate(tables):
        n = lens[b] // 16
        bufs.scores[b, :, :n] = torch.from_numpy(t[:, :n]).cuda()
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    sel = torch.full_like(bufs.selected, -1)
    nsel = torch.full_like(bufs.n_selected, -1)
    L.locks_select(H, seq_lens, max_pages, K, sel, nsel, bufs.workspace, scores=bufs.scores)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    return sel.cpu().numpy(), nsel.cpu().numpy()


@pytest.mark.parametrize("batch", [1, 2, 3])
def test_long_request_selection_distinct_scores(batch):
    rng = np.random.default_rng(40 + batch)
    lens = [16 * 18750 + 5, 16 * 17000 + 16, 16 * 18001][:batch]
    max_pages = (max(lens) + 15) // 16
    tables = [(rng.normal(size=(H, max_pages, 4)) * 2.0).astype(np.float32) for _ in lens]
    sel, nsel = _run(tables, lens, max_pages)
    for b in range(batch):
        n = lens[b] // 16
        for h in range(H):
            got = sel[b, h, :nsel[b, h]].astype(np.int64)
            check_selection(got, tables[b][h, :n].astype(np.float64), K)


@pytest.mark.parametrize("batch", [1, 3])
@pytest.mark.parametrize("copies", [40, 5000])
def test_long_request_tied_rows_take_lowest_pages(batch, copies):
    rng = np.random.default_rng(7 * copies + batch)
    lens = [16 * 18750 + 5, 16 * 17000 + 16, 16 * 18001][:batch]
    max_pages = (max(lens) + 15) // 16
    take = 10                   # copies inside the budget
    tables, want = [], []
    for b in range(batch):
        n = lens[b] // 16
        t = (rng.normal(size=(H, max_pages, 4)) * 0.5 - 6.0).astype(np.float32)
        w_b = []
        for h in range(H):
            pages = rng.permutation(n)
            winners = pages[:K - take]
            tied = np.sort(pages[K - take:K - take + copies])
            t[h, winners] = (rng.normal(size=(winners.size, 4)) * 0.1 + 6.0).astype(np.float32)
            t[h, tied] = np.float32([1.0, 1.5, 0.5, 2.0])
            expect = np.sort(np.concatenate([winners, tied[:take]]))
            sel_or, _ = O.select_pages(t[h, :n].astype(np.float64), K)
            assert sel_or.tolist() == expect.tolist()
            w_b.append(expect)
        tables.append(t)
        want.append(w_b)
    sel, nsel = _run(tables, lens, max_pages)
    for b in range(batch):
        for h in range(H):
            got = sel[b, h, :nsel[b, h]]
            assert got.tolist() == want[b][h].tolist(), (b, h)
