"""A bounded device wait that runs out is reported, and the context stays
usable.

locks_check_bounded_wait runs the library's bounded mbarrier wait (the one
every decode kernel uses) on a barrier that waits for two arrivals and gets
one, with a 1 ms limit, after issuing one bulk copy on a second barrier.  The
wait must give up, flag LOCKS_FLAG_TIMEOUT, wait for its copy and return; the
status read then reports LOCKS_ERR_TIMEOUT with the flag, and a decode step
launched afterwards in the same context is still correct.  No fault, trap or
unbounded wait is involved."""

import pytest
import torch

from sparse_long_context_locks_gb300 import locks as L
from sparse_long_context_locks_gb300 import workload as W

from gpu_helpers import Run, check_unit

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    src = torch.arange(256, dtype=torch.int32, device="cuda").to(torch.uint8)
    words = src.view(torch.int32).cpu().to(torch.int64)
    want_sum = int(words.sum().item()) & 0xFFFFFFFF
    result = torch.zeros(4, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    L.locks_check_bounded_wait(src, result, 1000, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    r = result.cpu().tolist()
    assert r[0] == 1, "the wait did not run out"
    assert r[1] == 1, "the issued copy did not land before exit"
    assert (r[2] & 0xFFFFFFFF) == want_sum, "the copy brought the wrong bytes"
    assert 0.9 <= ms < 500.0, f"the 1 ms wait took {ms:.3f} ms"
    # the status read reports the timeout with its flag, then starts clear
    v = ctypes_read(ws)
    assert v == (L.LOCKS_ERR_TIMEOUT, L.FLAG_TIMEOUT)
    assert ctypes_read(ws) == (L.LOCKS_OK, 0)
    assert L.locks_read_status(ws) == 0


def ctypes_read(ws):
    import ctypes
    v = ctypes.c_uint32(0)
    st = L.load().locks_read_status(ws.data_ptr(), ctypes.byref(v),
                                    torch.cuda.current_stream().cuda_stream)
    return st, int(v.value)


def test_context_usable_after_a_wait_ran_out():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    src = torch.zeros(256, dtype=torch.uint8, device="cuda")
    result = torch.zeros(4, dtype=torch.int32, device="cuda")
    for limit_us in (1, 50):
        L.locks_check_bounded_wait(src, result, limit_us, ws)
        torch.cuda.synchronize()
        assert result[0].item() == 1 and result[1].item() == 1
        assert L.locks_read_status(ws) == L.FLAG_TIMEOUT
    w = W.CONFIGS["pr1_4k"].scaled(context=16 * 60 + 7, budget_tokens=16 * 6, seed=3)
    run = Run(w)
    assert run.status == 0
    check_unit(run, 0, 0)
