"""Context-parallel decode through the library's kernels: a request's pages
split over 2 or 3 shards (here all on one GPU, run as threads of one process,
or as two gloo ranks in two processes; the shards exchange through host
memory and no kernel waits on another) must select what the one-GPU decode
step selects and attend like it.

Checks, per (request, KV head):
  * every shard's page scores equal the one-GPU scores bit for bit (same
    records, same query, slot-independent scorer);
  * the union of the shards' selections, as global pages, is the one-GPU
    selection: exact outside the tie band of the fp64 table of the one-GPU
    scores, a valid completion inside it (Z_g is summed in another order);
  * the merged output equals the oracle's attention over that selection
    within the attention tolerance, and the one-GPU output when the selections
    agree."""

import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle as O
from sparse_long_context_locks_gb300 import context_parallel as CP
from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from cp_helpers import run_shards
from gpu_helpers import ATTN_ATOL, check_attention, check_selection

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _setup(seed=21, batch=3):
    w = W.Workload("cp_gpu", batch=batch, context=16 * 2000 + 5, context_hi=16 * 2600 + 11, num_kv_heads=8,
                   group=4, budget_tokens=16 * 64, carriers_per_head=4, seed=seed)
    d = W.generate(w, device="cuda", tail_fill="nan")
    d["seq_lens"][2] = 16 * 40 + 7          # a short request: every full page fits the budget
    H = w.num_kv_heads
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    one = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ, one.workspace)
    L.locks_decode_step(H, d["q"], summ, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                        w.budget_pages, one.selected, one.n_selected, one.out, one.workspace, scores=one.scores)
    torch.cuda.synchronize()
    assert L.locks_read_status(one.workspace) == 0
    return w, d, summ, one


def _cuda_shards(w, d, summ, R):
    shards = []
    for r in range(R):
        bt, lens, off = CP.shard_pages(d["block_table"], d["seq_lens"], R, r)
        shards.append(CP.CudaShard(w.num_kv_heads, d["q"], summ, d["k_cache"], d["v_cache"], bt, lens, off,
                                   w.budget_pages, r))
    return shards


def _check(w, d, one, selected, out, shard_scores=None):
    H, G = w.num_kv_heads, w.group
    lens = d["seq_lens"].cpu().tolist()
    bt = d["block_table"].cpu().numpy()
    q = d["q"].double().cpu().numpy()
    agree = 0
    for b in range(w.batch):
        n = lens[b] // 16
        for h in range(H):
            s_one = one.scores[b, h, :n].double().cpu().numpy()
            if shard_scores is not None:
                np.testing.assert_array_equal(shard_scores[b, h, :n], s_one)
            sel = np.array(sorted(selected[(b, h)]), dtype=np.int64)
            check_selection(sel, s_one, w.budget_pages)
            pages = list(sel) + ([n] if lens[b] % 16 else [])
            blocks = torch.from_numpy(bt[b, pages].astype(np.int64)).cuda()
            kc = d["k_cache"][blocks, h].double().cpu().numpy()[:, None]
            vc = d["v_cache"][blocks, h].double().cpu().numpy()[:, None]
            row = np.zeros(n + 1, dtype=np.int64)
            for i, j in enumerate(pages):
                row[j] = i
            ref = O.sparse_attend_unit(q[b, h * G:(h + 1) * G], kc, vc, row, 0, lens[b], sel, 1 / math.sqrt(128))
            got = out[b, h * G:(h + 1) * G].double().cpu().numpy()
            check_attention(got, ref)
            one_sel = one.selected[b, h, :int(one.n_selected[b, h])].cpu().tolist()
            if one_sel == sel.tolist():
                agree += 1
                assert np.abs(got - one.out[b, h * G:(h + 1) * G].double().cpu().numpy()).max() <= ATTN_ATOL
    assert agree >= w.batch * H - 2, f"only {agree} units select exactly as on one GPU"


@pytest.mark.parametrize("R,batch", [(2, 3), (3, 3), (2, 6)])
def test_cuda_shards_match_one_gpu_step(R, batch):
    """batch 3: 24 units, 12 attention splits a unit (merged through the
    workspace); batch 6: 48 units, 6 splits (merged in a thread-block
    cluster)."""
    w, d, summ, one = _setup(batch=batch)
    shards = _cuda_shards(w, d, summ, R)
    outs = run_shards(CP.decode_step, shards)
    torch.cuda.synchronize()
    for s in shards:
        assert L.locks_read_status(s.bufs.workspace) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "shards disagree on the merged output"
    selected = {}
    scores = np.full((w.batch, w.num_kv_heads, w.max_pages, 4), np.nan)
    lens = d["seq_lens"].cpu().tolist()
    for s in shards:
        for key, pages in s.selected_global().items():
            selected.setdefault(key, []).extend(pages)
        off = s.off.cpu().tolist()
        n_loc = (s.lens.cpu() // 16).tolist()
        sc = s.bufs.scores.double().cpu().numpy()
        for b in range(w.batch):
            scores[b, :, off[b]:off[b] + n_loc[b]] = sc[b, :, :n_loc[b]]
    for b in range(w.batch):
        assert not np.isnan(scores[b, :, :lens[b] // 16]).any()
    _check(w, d, one, selected, outs[0], shard_scores=scores)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, result):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        w, d, summ, _ = _setup(seed=22)
        shard = _cuda_shards(w, d, summ, world)[rank]
        out = CP.decode_step(shard, CP.host_all_gather())
        torch.cuda.synchronize()
        assert L.locks_read_status(shard.bufs.workspace) == 0
        result[rank] = (out.cpu(), shard.selected_global())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_on_one_gpu_match_one_gpu_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        result = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, result)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=600)
            assert p.exitcode == 0
        w, d, summ, one = _setup(seed=22)
        assert torch.equal(result[0][0], result[1][0])
        selected = {}
        for r in range(2):
            for key, pages in result[r][1].items():
                selected.setdefault(key, []).extend(pages)
        _check(w, d, one, selected, result[0][0].cuda())
