"""Context-parallel decode on the CPU: the shard decomposition of the
selection and attention (per-shard (max, sum) pairs -> Z_g; the global top-k
from the shards' local top-k lists; attention states merged by the
online-softmax rule), run through the library's own step sequencing
(context_parallel.decode_step) with float64 oracle shards, must reproduce the
oracle's single-shot decode step.  Shards run as threads of one process and
as two gloo ranks (world size 2)."""

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
from sparse_long_context_locks_gb300 import workload as W

from cp_helpers import OracleShard, run_shards

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCALE = 1.0 / math.sqrt(O.HEAD_DIM)


def _data(seed=11, budget_pages=7):
    w = W.Workload("cp_tiny", batch=2, context=16 * 37 + 5, context_hi=16 * 45 + 9, num_kv_heads=2, group=4,
                   budget_tokens=16 * budget_pages, carriers_per_head=2, seed=seed)
    d = W.generate(w, device="cpu")
    kc = d["k_cache"].double().numpy()
    rec = O.build_records(kc)
    return w, d, kc, d["v_cache"].double().numpy(), rec


def _shards(w, d, kc, vc, rec, R):
    q = d["q"].double().numpy()
    out = []
    for r in range(R):
        bt, lens, off = CP.shard_pages(d["block_table"], d["seq_lens"], R, r)
        out.append(OracleShard(q, rec, kc, vc, bt.numpy().astype(np.int64), lens.numpy(), off.numpy(),
                               w.budget_pages, w.num_kv_heads, w.group, r, SCALE))
    return out


def _check(w, d, kc, vc, rec, outs, selected):
    want = O.decode_step(d["q"].double().numpy(), kc, vc, d["block_table"].numpy().astype(np.int64),
                         d["seq_lens"].numpy(), rec, w.num_kv_heads, w.group, w.budget_pages, scale=SCALE)
    G = w.group
    for (b, h), res in want.items():
        assert selected[(b, h)] == res["selected"].tolist(), (b, h)
        for o in outs:
            np.testing.assert_allclose(np.asarray(o)[b, h * G:(h + 1) * G], res["out"], atol=1e-11, rtol=0)


@pytest.mark.parametrize("R", [1, 2, 3, 5])
def test_oracle_shards_reproduce_single_shot_step(R):
    w, d, kc, vc, rec = _data()
    shards = _shards(w, d, kc, vc, rec, R)
    outs = run_shards(CP.decode_step, shards)
    sel = {}
    for s in shards:
        for key, pages in s.selected_global().items():
            sel.setdefault(key, []).extend(pages)
    sel = {k: sorted(v) for k, v in sel.items()}
    _check(w, d, kc, vc, rec, outs, sel)


def test_oracle_shards_when_every_page_fits_the_budget():
    w, d, kc, vc, rec = _data(seed=12, budget_pages=64)   # n <= k: every page is selected
    shards = _shards(w, d, kc, vc, rec, 3)
    outs = run_shards(CP.decode_step, shards)
    sel = {}
    for s in shards:
        for key, pages in s.selected_global().items():
            sel.setdefault(key, []).extend(pages)
    _check(w, d, kc, vc, rec, outs, {k: sorted(v) for k, v in sel.items()})


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
        w, d, kc, vc, rec = _data(seed=13)
        shard = _shards(w, d, kc, vc, rec, world)[rank]
        out = CP.decode_step(shard, CP.host_all_gather())
        result[rank] = (out.numpy(), shard.selected_global())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_single_shot_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        result = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, result)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        w, d, kc, vc, rec = _data(seed=13)
        sel = {}
        for r in range(2):
            for key, pages in result[r][1].items():
                sel.setdefault(key, []).extend(pages)
        # the two ranks hold different pages, but both end with the same output
        _check(w, d, kc, vc, rec, [result[0][0], result[1][0]], {k: sorted(v) for k, v in sel.items()})
