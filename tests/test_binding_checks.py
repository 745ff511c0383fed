"""The Python binding checks the layouts the C ABI assumes (include/locks.h)
before it passes a pointer: contiguous CUDA tensors of the stated dtype and
shape.  CPU part: host tensors are refused before the library is touched.
GPU part: one wrong argument at a time, each refused, and the right call runs;
`out` in pinned host memory (the kernels store the result straight into it)
gives the bits the device buffer gets, and pageable host memory is refused."""

import pytest
import torch

from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W


def test_host_tensors_are_refused():
    H, B, MP = 8, 1, 4
    q = torch.zeros(B, H * 4, 128, dtype=torch.bfloat16)
    summ = torch.zeros(16, H, 784, dtype=torch.uint8)
    bt = torch.zeros(B, MP, dtype=torch.int32)
    lens = torch.zeros(B, dtype=torch.int32)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.locks_score(H, q, summ, bt, lens, ws)
    kc = torch.zeros(16, H, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        L.locks_build_summaries(H, kc, torch.zeros(2, dtype=torch.int32), summ)


@pytest.mark.gpu
def test_wrong_arguments_are_refused_and_the_right_call_runs():
    w = W.Workload("t", batch=2, context=16 * 40 + 3, num_kv_heads=8, group=4, budget_tokens=16 * 8,
                   carriers_per_head=0, seed=5)
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ, bufs.workspace)
    args = dict(q=d["q"], summaries=summ, k_cache=d["k_cache"], v_cache=d["v_cache"],
                block_table=d["block_table"], seq_lens=d["seq_lens"], selected=bufs.selected,
                n_selected=bufs.n_selected, out=bufs.out, workspace=bufs.workspace)

    def step(**over):
        a = dict(args, **over)
        L.locks_decode_step(H, a["q"], a["summaries"], a["k_cache"], a["v_cache"], a["block_table"],
                            a["seq_lens"], w.budget_pages, a["selected"], a["n_selected"], a["out"],
                            a["workspace"])

    bad = {
        "q": d["q"].float(),                                            # dtype
        "k_cache": d["k_cache"][:, :4].contiguous(),                    # heads
        "v_cache": d["v_cache"][:-1],                                   # differs from k_cache
        "block_table": d["block_table"].t().contiguous().t(),           # not contiguous
        "seq_lens": d["seq_lens"][:1],                                  # batch
        "selected": torch.zeros(w.batch, H, w.budget_pages + 1, dtype=torch.int32, device="cuda"),
        "out": bufs.out.to(torch.bfloat16),                             # dtype
        "summaries": summ[:, :, :700].contiguous(),                     # record width
    }
    for name, value in bad.items():
        with pytest.raises(ValueError, match=name):
            step(**{name: value})
    step()
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    assert torch.isfinite(bufs.out).all()


@pytest.mark.gpu
def test_out_in_pinned_host_memory_matches_the_device_buffer():
    w = W.Workload("t", batch=3, context=16 * 300 + 5, context_hi=16 * 500, num_kv_heads=8, group=4,
                   budget_tokens=16 * 24, carriers_per_head=2, seed=9)
    d = W.generate(w, device="cuda")
    H = w.num_kv_heads
    bufs = L.DecodeBuffers(H, w.batch, w.max_pages, w.budget_pages)
    summ = torch.zeros(d["num_blocks"], H, 784, dtype=torch.uint8, device="cuda")
    L.locks_build_summaries(H, d["k_cache"], W.full_page_blocks(d).cuda(), summ, bufs.workspace)
    pinned = torch.full(bufs.out.shape, float("nan"), dtype=torch.float32).pin_memory()
    assert L.load().locks_device_accessible(pinned.data_ptr()) == 1
    assert L.load().locks_device_accessible(bufs.out.data_ptr()) == 1
    assert L.load().locks_device_accessible(torch.zeros(4).data_ptr()) == 0
    common = (H, d["q"], summ, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], w.budget_pages,
              bufs.selected, bufs.n_selected)
    L.locks_decode_step(*common, bufs.out, bufs.workspace, scores=bufs.scores)
    L.locks_decode_step(*common, pinned, bufs.workspace, scores=bufs.scores)
    torch.cuda.synchronize()
    assert L.locks_read_status(bufs.workspace) == 0
    assert torch.equal(pinned, bufs.out.cpu())
    dense_dev = torch.empty_like(bufs.out)
    dense_host = torch.full(bufs.out.shape, float("nan"), dtype=torch.float32).pin_memory()
    L.locks_dense_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], dense_dev,
                         bufs.workspace)
    L.locks_dense_decode(H, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], dense_host,
                         bufs.workspace)
    torch.cuda.synchronize()
    assert torch.equal(dense_host, dense_dev.cpu())
    with pytest.raises(ValueError, match="pinned"):
        L.locks_decode_step(*common, torch.zeros(bufs.out.shape), bufs.workspace)
