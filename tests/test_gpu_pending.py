"""Page-crossing decode: locks_build_pending builds the pages that became
full at a step (a device-side count, so one captured graph serves every
step), and the step that follows scores them like any other page."""

import numpy as np
import pytest
import torch

from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run, check_records, check_unit

pytestmark = pytest.mark.gpu


def _w(**kw):
    base = dict(name="t", batch=1, context=16 * 200 + 14, num_kv_heads=8, group=4,
                budget_tokens=16 * 24, carriers_per_head=4, seed=3)
    base.update(kw)
    return W.Workload(**base)


def test_build_pending_matches_build_and_reads_the_device_count():
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
        assert torch.equal(summ[built], ref[built])
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
