"""The seeded input generator: determinism, structure, sizes (CPU only)."""

import math

import pytest
import torch

from sparse_long_context_locks_gb300 import workload as W


def _tiny(**kw):
    base = dict(name="tiny", batch=2, context=16 * 20 + 4, num_kv_heads=2, group=4,
                budget_tokens=16 * 5, carriers_per_head=2, seed=7)
    base.update(kw)
    return W.Workload(**base)


def test_deterministic_and_seed_sensitive():
    a = W.generate(_tiny())
    b = W.generate(_tiny())
    c = W.generate(_tiny(seed=8))
    for key in ("q", "k_cache", "v_cache", "block_table", "seq_lens"):
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["k_cache"], c["k_cache"])


def test_shapes_block_table_and_lengths():
    w = _tiny()
    d = W.generate(w)
    L = w.context + 1
    n_pages = math.ceil(L / 16)
    assert d["q"].shape == (2, 8, 128) and d["q"].dtype == torch.bfloat16
    assert d["k_cache"].shape == (2 * n_pages, 2, 16, 128)
    assert d["seq_lens"].tolist() == [L, L]
    bt = d["block_table"]
    assert bt.shape == (2, w.max_pages)
    used = bt[bt >= 0]
    assert sorted(used.tolist()) == list(range(2 * n_pages))  # a permutation
    assert not torch.equal(used, torch.arange(2 * n_pages, dtype=torch.int32))


def test_ragged_lengths_in_range():
    w = W.CONFIGS["batch16_32k"]
    lens = W.request_lengths(w)
    assert len(lens) == 16 and len(set(lens)) > 1
    assert all(24576 + 1 <= L <= 32768 + 1 for L in lens)
    assert any(L % 16 for L in lens)


def test_carriers_are_planted_and_tail_slots_filled():
    w = _tiny()
    d = W.generate(w, tail_fill="nan")
    q = d["q"].float().view(2, 2, 4, 128).mean(2)
    for b, h, j, s in d["carriers"]:
        blk = int(d["block_table"][b, j])
        qb = q[b, h] / q[b, h].norm()
        assert torch.equal(d["k_cache"][blk, h, s], (6 * qb).to(torch.bfloat16))
        assert j < int(d["seq_lens"][b]) // 16
    L = w.context + 1
    t = L % 16
    blk = int(d["block_table"][0, L // 16])
    assert torch.isnan(d["k_cache"][blk, :, t:].float()).all()
    assert not torch.isnan(d["k_cache"][blk, :, :t].float()).any()


def test_lowrank_pages_have_rank8_structure():
    w = _tiny(noise_std=0.0)
    d = W.generate(w)
    blk = int(d["block_table"][0, 3])
    K = d["k_cache"][blk, 0].double()
    X = K - K.mean(0)
    sv = torch.linalg.svdvals(X)
    # rank 8 up to bf16 rounding of the keys
    assert sv[8] / sv[0] < 2e-2 and sv[7] / sv[0] > 2e-2


def test_fullrank_regime_is_flat():
    d = W.generate(_tiny(key_regime="fullrank"))
    blk = int(d["block_table"][1, 2])
    X = d["k_cache"][blk, 1].double()
    X = X - X.mean(0)
    sv = torch.linalg.svdvals(X)
    assert sv[14] / sv[0] > 0.3


def test_algorithmic_bytes_of_the_named_workloads():
    w = W.CONFIGS["llama8b_128k"]
    lens = W.request_lengths(w)
    by = W.algorithmic_bytes(lens, 8, 4, w.budget_pages)
    assert by["score"] == 8 * 8192 * 784
    assert by["sparse_kv"] == 8 * 128 * 8192 + 8 * 1 * 512
    assert by["dense_kv"] == 8 * 8192 * 8192 + 8 * 512
    w4 = W.CONFIGS["ctx1m"]
    b4 = W.algorithmic_bytes(W.request_lengths(w4), 8, 4, w4.budget_pages)
    assert b4["dense_kv"] / (b4["score"] + b4["sparse_kv"]) >= 9.0
