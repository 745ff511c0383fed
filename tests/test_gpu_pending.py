"""Page-crossing decode: locks_build_pending builds the pages that became
full at a step (a device-side count, so one captured graph serves every
step), and the step that follows scores them like any other page."""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run, check_records, check_unit

pytestmark = pytest.mark.gpu


def _w(**kw):
    base = dict(name="t", batch=1, context=16 * 200 + 14, num_kv_heads=8, group=4,
                budget_tokens=16 * 24, carriers_per_head=4, seed=3)
    base.update(kw)
    return W.Workload(**base)


def test_build_pending_reads_the_device_count():
    w = _w(batch=3, context=16 * 60, context_hi=16 * 120)
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    blocks = W.full_page_blocks(d).cuda()
    ref = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(H, d["k_cache"], blocks, ref)
    pick = blocks[torch.randperm(blocks.numel(), generator=torch.Generator().manual_seed(0))[:6].cuda()]
    ids = torch.full((8,), 2 ** 30, dtype=torch.int32, device="cuda")   # entries past the count: never read
    ids[:6] = pick.to(torch.int32)
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    summ = torch.zeros_like(ref)
    ws = L.DecodeBuffers(H, 1, 16, 2).workspace
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.locks_build_pending(H, d["k_cache"], ids, n, summ, ws)
    g.replay()
    torch.cuda.synchronize()
    assert int(summ.count_nonzero()) == 0                                # count 0: nothing built
    for k in (2, 6):
        n.fill_(k)
        g.replay()
        torch.cuda.synchronize()
        built = pick[:k].long()
        for h in range(H):   # against the oracle's decomposition of the same keys
            check_records(summ[built, h].cpu().numpy(), d["k_cache"][built, h].double().cpu().numpy())
        rest = torch.ones(d["num_blocks"], dtype=torch.bool, device="cuda")
        rest[built] = False
        assert int(summ[rest].count_nonzero()) == 0
    assert L.locks_read_status(ws) == 0


@pytest.mark.parametrize("heads", [8, 2])
def test_decode_across_a_page_boundary(heads):
    # L = N + 1 = 16 m + 15: the next token fills the tail page
    w = _w(num_kv_heads=heads, seed=heads)
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ)
    L0 = int(d["seq_lens"][0])
    assert L0 % 16 == 15
    tail_blk = int(d["block_table"][0, L0 // 16])
    gen = torch.Generator(device="cuda").manual_seed(11)
    new_k = torch.randn(H, 128, generator=gen, device="cuda").to(torch.bfloat16)
    new_v = torch.randn(H, 128, generator=gen, device="cuda").to(torch.bfloat16)
    d["k_cache"][tail_blk, :, 15] = new_k
    d["v_cache"][tail_blk, :, 15] = new_v
    d["seq_lens"] += 1
    ids = torch.tensor([tail_blk], dtype=torch.int32, device="cuda")
    n = torch.ones(1, dtype=torch.int32, device="cuda")
    L.locks_build_pending(H, d["k_cache"], ids, n, summ)
    run = Run(w, data=d, summ=summ)
    assert run.status == 0
    assert run.lens[0] == L0 + 1 and run.lens[0] % 16 == 0   # no tail page left
    for h in range(H):
        check_unit(run, 0, h)
    page = np.array([L0 // 16])
    for h in range(H):
        check_records(summ[torch.tensor([tail_blk], device="cuda").long(), h].cpu().numpy(),
                      run.pages_f64(d["k_cache"], 0, h, page))


@pytest.mark.parametrize("fused", [True, False])
def test_decode_step_crossing_equals_build_then_step(fused):
    """locks_decode_step_crossing builds the page each request's current token
    completed (overlapped with the scoring of the other pages) and decodes: the
    records, selections and outputs equal those of locks_build_pending over
    the same pages followed by locks_decode_step, bit for bit.  A ragged batch
    mixes requests at a crossing (L % 16 == 0) with requests mid-page; the
    new pages' records start as garbage, so a copy taken before the build
    ended would show."""
    batch = 2 if fused else 40          # 40 x 8 clusters exceed the GPU: separate path
    w = _w(batch=batch, context=16 * 300 + 3, context_hi=16 * 420, seed=17)
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    lens = d["seq_lens"].cpu()
    cross = torch.arange(batch) % 3 != 1               # two requests in three at a crossing
    lens = torch.where(cross, (lens // 16) * 16, lens)
    lens = torch.where(lens % 16 == 0, lens, lens | 1)  # the others keep a tail
    d["seq_lens"].copy_(lens.to(torch.int32))
    full = W.full_page_blocks(d).cuda()
    new_pages = [(b, int(lens[b]) // 16 - 1) for b in range(batch) if int(lens[b]) % 16 == 0]
    new_blocks = torch.tensor([int(d["block_table"][b, j]) for b, j in new_pages], dtype=torch.int32,
                              device="cuda")
    # every other full page is built ahead; the new ones hold garbage
    is_new = torch.zeros(d["num_blocks"], dtype=torch.bool, device="cuda")
    is_new[new_blocks.long()] = True
    old = full[~is_new[full.long()]]
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(H, d["k_cache"], old, summ)
    summ[new_blocks.long()] = 0xA5
    ref_summ = summ.clone()
    L.locks_build_pending(H, d["k_cache"], new_blocks, torch.tensor([len(new_pages)], dtype=torch.int32,
                                                                    device="cuda"), ref_summ)
    a = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    b_ = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    L.locks_decode_step(H, d["q"], ref_summ, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                        w.budget_pages, a.selected, a.n_selected, a.out, a.workspace, scores=a.scores)
    L.locks_decode_step_crossing(H, d["q"], summ, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                 w.budget_pages, b_.selected, b_.n_selected, b_.out, b_.workspace,
                                 scores=b_.scores)
    torch.cuda.synchronize()
    assert L.locks_read_status(a.workspace) == 0 and L.locks_read_status(b_.workspace) == 0
    assert torch.equal(summ, ref_summ)
    assert torch.equal(b_.n_selected, a.n_selected)
    for bb in range(batch):
        for h in range(H):
            k = int(a.n_selected[bb, h])
            assert torch.equal(b_.selected[bb, h, :k], a.selected[bb, h, :k])
            n = int(lens[bb]) // 16
            assert torch.equal(b_.scores[bb, h, :n], a.scores[bb, h, :n])
    assert torch.equal(b_.out, a.out)
    # and the step itself against the oracle, on a few units
    run = Run(w, data=d, summ=summ)
    for bb, h in ((0, 0), (min(2, batch - 1), 5)):
        check_unit(run, bb, h)


def test_decode_step_crossing_in_a_graph_replays():
    """One captured graph of the crossing step serves successive steps."""
    w = _w(batch=2, context=16 * 100 - 1, seed=19)          # L = 1600: at a crossing
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ)
    bulk = summ.clone()
    last = [int(d["block_table"][b, int(d["seq_lens"][b]) // 16 - 1]) for b in range(2)]
    new = torch.tensor(last).long()
    summ[new] = 0
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L.locks_decode_step_crossing(H, d["q"], summ, d["k_cache"], d["v_cache"], d["block_table"],
                                     d["seq_lens"], w.budget_pages, bufs.selected, bufs.n_selected, bufs.out,
                                     bufs.workspace, scores=bufs.scores, stream=s)
        s.synchronize()
        ref = summ.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            L.locks_decode_step_crossing(H, d["q"], summ, d["k_cache"], d["v_cache"], d["block_table"],
                                         d["seq_lens"], w.budget_pages, bufs.selected, bufs.n_selected,
                                         bufs.out, bufs.workspace, scores=bufs.scores, stream=s)
    first = bufs.out.clone()
    rest = torch.ones(d["num_blocks"], dtype=torch.bool, device="cuda")
    rest[new] = False
    assert torch.equal(ref[rest], bulk[rest])                  # only the new pages were written
    for h in range(H):
        check_records(ref[new, h].cpu().numpy(), d["k_cache"][new, h].double().cpu().numpy())
    for _ in range(3):
        summ[new] = 0
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(summ, ref)
        assert torch.equal(bufs.out, first)
    assert L.locks_read_status(bufs.workspace) == 0


def test_build_pending_special_pages_against_the_oracle():
    """Both builders on pages where an eigensolver can go wrong: equal keys,
    exact low rank, a zero page, large and tiny magnitudes, 16 equal and two
    repeated eigenvalues, a large centroid, and random pages.  The page
    builder (Householder, multisection, inverse iteration) and the bulk
    builder (Jacobi) each meet the oracle's records, and on the pages whose
    top directions are unique their codes differ by at most one (a value on
    a rounding edge)."""
    rng = np.random.default_rng(12)
    pages = [np.tile(rng.normal(size=128), (16, 1)),
             rng.integers(-3, 4, 128) + rng.integers(-3, 4, (16, 3)) @ rng.integers(-2, 3, (128, 3)).T,
             np.zeros((16, 128)),
             rng.normal(size=(16, 128)) * 300.0,
             rng.normal(size=(16, 128)) * 1e-3]
    Q, _ = np.linalg.qr(rng.normal(size=(128, 16)))
    pages.append(Q[:, :16].T * 2.0)                                       # 16 equal eigenvalues
    pages.append(np.diag(np.repeat([4.0, 2.0], 8)) @ Q[:, :16].T)        # two repeated eigenvalues
    pages.append(rng.normal(size=(16, 128)) * 3.0 + 5.0)                # a large centroid
    for s in (0.05, 1.0, 30.0):
        pages += [rng.normal(size=(16, 128)) * s for _ in range(8)]
    K = torch.tensor(np.stack(pages), dtype=torch.bfloat16)              # 32 pages
    Kd = K.double().numpy()
    lam = O.page_summary(Kd)["lam"]
    gaps = -np.diff(lam[:, :9], axis=1) / np.maximum(lam[:, :1], 1e-30)
    unique = np.all(gaps > 1e-3, axis=1) & (lam[:, 7] > 1e-3 * lam[:, 0])
    assert unique.sum() >= 24
    for H in (1, 2):
        kc = K.view(-1, H, 16, 128).contiguous().cuda()
        nblk = kc.shape[0]
        ids = torch.arange(nblk, dtype=torch.int32, device="cuda")
        bulk = torch.zeros(nblk, H, 784, dtype=torch.uint8, device="cuda")
        got = torch.zeros_like(bulk)
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        L.locks_build_summaries(H, kc, ids, bulk, ws)
        n = torch.full((1,), nblk, dtype=torch.int32, device="cuda")
        L.locks_build_pending(H, kc, ids, n, got, ws)
        torch.cuda.synchronize()
        assert L.locks_read_status(ws) == 0
        for rec in (got, bulk):
            check_records(rec.view(-1, 784).cpu().numpy(), Kd)
        g = O.decode_records(got.view(-1, 784).cpu().numpy())
        b = O.decode_records(bulk.view(-1, 784).cpu().numpy())
        assert np.array_equal(g["muq"], b["muq"])
        for key in ("Vq", "Cq"):
            diff = np.abs(g[key].astype(np.int64) - b[key].astype(np.int64))[unique]
            assert diff.max() <= 1, key


def _hard_pages(rng):
    """Pages whose spectra stress an eigensolver: every rank from 1 to 16 with
    a little noise, geometric spectra with condition numbers up to 1e6, pairs
    of eigenvalues 1e-2 and 1e-5 apart, at magnitudes from 1e-4 to 1e3."""
    pages = []
    for r in range(1, 17):
        for s in (1e-4, 1.0, 1e3):
            K = rng.normal(size=(16, r)) @ rng.normal(size=(r, 128)) + rng.normal(size=128)
            pages.append(s * (K + 1e-3 * rng.normal(size=(16, 128))))
    for kappa in (1e2, 1e4, 1e6):
        for _ in range(8):
            U, _ = np.linalg.qr(rng.normal(size=(16, 16)))
            Wm, _ = np.linalg.qr(rng.normal(size=(128, 16)))
            sig = kappa ** (-np.arange(16) / 15.0)
            pages.append((U * sig) @ Wm.T * rng.uniform(0.5, 20.0))
    for delta in (1e-2, 1e-5):
        for _ in range(8):
            U, _ = np.linalg.qr(rng.normal(size=(16, 16)))
            Wm, _ = np.linalg.qr(rng.normal(size=(128, 16)))
            base = np.sort(rng.uniform(0.2, 1.0, 8))[::-1]
            sig = np.sqrt(np.repeat(base, 2) * np.tile([1.0, 1.0 + delta], 8))
            pages.append((U * sig) @ Wm.T * 10.0)
    return pages


def test_build_pending_hard_spectra_against_the_oracle():
    """The page builder on pages of hard spectra (and the bulk builder on the
    same pages, for comparison), each against the oracle's records.  Rounding
    the keys to bf16 moves the Gram matrix by about 4e-3 relative, so a pair
    designed 1e-5 apart lands at a random gap near 1e-3: the records checks'
    bar for unique top directions.  Just above that bar an fp32 eigenvector
    is off by up to eps * |G| / gap times the solver's accumulated roundings,
    which meets the scales' 2e-4 tolerance; pages whose smallest top-9 gap
    lies in [1e-3, 3e-3) are therefore left out (a handful of 88)."""
    pages = np.stack(_hard_pages(np.random.default_rng(77)))
    lam = O.page_summary(torch.tensor(pages, dtype=torch.bfloat16).double().numpy())["lam"]
    gap = np.min(-np.diff(lam[:, :9], axis=1), axis=1) / np.maximum(lam[:, 0], 1e-30)
    keep = (gap < 1e-3) | (gap >= 3e-3)
    assert keep.sum() >= 80
    K = torch.tensor(pages[keep], dtype=torch.bfloat16)
    Kd = K.double().numpy()
    nblk = K.shape[0]
    kc = K[:, None].contiguous().cuda()
    ids = torch.arange(nblk, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    got = torch.zeros(nblk, 1, 784, dtype=torch.uint8, device="cuda")
    bulk = torch.zeros_like(got)
    L.locks_build_pending(1, kc, ids, torch.full((1,), nblk, dtype=torch.int32, device="cuda"), got, ws)
    L.locks_build_summaries(1, kc, ids, bulk, ws)
    torch.cuda.synchronize()
    assert L.locks_read_status(ws) == 0
    res = check_records(got[:, 0].cpu().numpy(), Kd)
    check_records(bulk[:, 0].cpu().numpy(), Kd)
    assert res["well_conditioned"] >= 40
