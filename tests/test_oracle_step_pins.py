"""Pins of the oracle's whole-step functions, unit_scores_from_records and
decode_step, against a paged cache whose expected results are gathered by
hand.

The fixture is built without the oracle's summary builder: every page-head's
record is written from chosen integer codes and power-of-two scales, so the
keys it stands for are known exactly.  By linearity of the score equation of
"LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context Decoding"
(technical summary §2, "Reconstruction and selection"), the score of page j is
the log-sum-exp of q.k_i / sqrt(d) over the 16 keys k_i = mu + V c_i that its
record stands for; those keys are formed here with plain torch arithmetic, the
pages of each request are looked up through its block-table row by explicit
Python loops, and the shares, the group mean (§2 "Group-shared selection
(GQA)") and the top-k order are computed by hand.  Attention is torch softmax
over the tokens gathered page by page, the open tail page included.

Two KV heads with different records, a permuted block table with unused
blocks, two requests with different lengths and partially filled tail pages:
a wrong head slice, a wrong block-table row, a dropped tail or an off-by-one
page count changes the result, and the planted-mistake test checks that each
of those slips fails the pins.
"""

import math

import numpy as np
import pytest
import torch

import oracle as O
import oracle.locks_oracle as OL

D, B, R, G, H = O.HEAD_DIM, O.PAGE_SIZE, O.RANK, 4, 2
SCALE = 1.0 / math.sqrt(D)
LENS = [16 * 7 + 5, 16 * 4 + 11]          # 7 and 4 full pages, tails of 5 and 11 tokens
MAX_PAGES = 8
N_BLOCKS = 19
BUDGET = 3


def _fixture(seed=31):
    rng = np.random.default_rng(seed)
    Vq = rng.integers(-7, 8, size=(N_BLOCKS, H, D, R)).astype(np.int8)
    muq = rng.integers(-127, 128, size=(N_BLOCKS, H, D)).astype(np.int8)
    Cq = rng.integers(-127, 128, size=(N_BLOCKS, H, B, R)).astype(np.int8)
    sV = np.full((N_BLOCKS, H), 2.0 ** -3)
    smu = np.full((N_BLOCKS, H), 2.0 ** -6)
    sC = np.full((N_BLOCKS, H), 2.0 ** -5)
    sC[:, 1] = 2.0 ** -4                 # head 1's pages are spread more widely
    rec = O.encode_records({"Vq": Vq, "muq": muq, "Cq": Cq, "sV": sV, "smu": smu, "sC": sC,
                            "tail": np.zeros((N_BLOCKS, H))})
    kc = rng.normal(size=(N_BLOCKS, H, B, D))
    vc = rng.normal(size=(N_BLOCKS, H, B, D))
    bt = np.full((2, MAX_PAGES), -1, dtype=np.int64)
    perm = rng.permutation(N_BLOCKS)
    bt[0, :8] = perm[:8]                 # request 0: 7 full pages + tail page
    bt[1, :5] = perm[8:13]               # request 1: 4 full pages + tail page
    q = rng.normal(size=(2, H * G, D)) * 1.5
    codes = {"Vq": Vq, "muq": muq, "Cq": Cq, "sV": sV, "smu": smu, "sC": sC}
    return q, kc, vc, bt, np.array(LENS), rec, codes


def _keys_of_record(codes, blk, h):
    """The 16 keys a record stands for, k_i = mu + V c_i, in torch fp64."""
    mu = torch.tensor(codes["muq"][blk, h], dtype=torch.float64) * codes["smu"][blk, h]
    V = torch.tensor(codes["Vq"][blk, h], dtype=torch.float64) * codes["sV"][blk, h]      # [d, r]
    C = torch.tensor(codes["Cq"][blk, h], dtype=torch.float64) * codes["sC"][blk, h]      # [16, r]
    return mu[None, :] + C @ V.T


def _expected_unit(q, kc, vc, bt, lens, codes, b, h, budget):
    L = int(lens[b])
    n, t = L // B, L % B
    qg = torch.tensor(q[b, h * G:(h + 1) * G], dtype=torch.float64)
    scores = torch.zeros(n, G, dtype=torch.float64)
    for j in range(n):
        keys = _keys_of_record(codes, int(bt[b, j]), h)
        scores[j] = torch.logsumexp(qg @ keys.T * SCALE, dim=-1)
    shares = torch.softmax(scores, dim=0)                     # per head, over full pages
    table = [float(sum(shares[j, g] for g in range(G)) / G) for j in range(n)]
    order = sorted(range(n), key=lambda j: (-table[j], j))
    sel = sorted(order[:min(budget, n)])
    toks_k, toks_v = [], []
    for j in sel:
        for i in range(B):
            toks_k.append(kc[int(bt[b, j]), h, i])
            toks_v.append(vc[int(bt[b, j]), h, i])
    for i in range(t):
        toks_k.append(kc[int(bt[b, n]), h, i])
        toks_v.append(vc[int(bt[b, n]), h, i])
    Kt = torch.tensor(np.array(toks_k))
    Vt = torch.tensor(np.array(toks_v))
    out = torch.softmax(qg @ Kt.T * SCALE, dim=-1) @ Vt
    # the fixture keeps every selection decision well away from a tie
    if n > budget:
        srt = sorted(table, reverse=True)
        assert srt[budget - 1] - srt[budget] > 1e-6 * srt[0]
    return scores.numpy(), np.array(table), sel, out.numpy()


def _scores_pin_holds(score_fn) -> bool:
    q, kc, vc, bt, lens, rec, codes = _fixture()
    for b in range(2):
        for h in range(H):
            want, _, _, _ = _expected_unit(q, kc, vc, bt, lens, codes, b, h, BUDGET)
            got = score_fn(q[b, h * G:(h + 1) * G], rec, bt[b], h, int(lens[b]))
            if got.shape != want.shape or not np.allclose(got, want, rtol=0, atol=1e-10):
                return False
    return True


def _step_pin_holds(step_fn, budget=BUDGET) -> bool:
    q, kc, vc, bt, lens, rec, codes = _fixture()
    res = step_fn(q, kc, vc, bt, lens, rec, H, G, budget)
    for b in range(2):
        for h in range(H):
            s, table, sel, out = _expected_unit(q, kc, vc, bt, lens, codes, b, h, budget)
            r = res[(b, h)]
            if r["scores"].shape != s.shape or not np.allclose(r["scores"], s, rtol=0, atol=1e-10):
                return False
            if not np.allclose(r["avg"], table, rtol=1e-12, atol=0):
                return False
            if list(r["selected"]) != sel:
                return False
            if r["out"].shape != out.shape or not np.allclose(r["out"], out, rtol=0, atol=1e-12):
                return False
    return True


def test_unit_scores_from_records_equal_hand_gathered_page_lse():
    assert _scores_pin_holds(O.unit_scores_from_records)


@pytest.mark.parametrize("budget", [BUDGET, 1, 16])
def test_decode_step_equals_hand_gathered_selection_and_attention(budget):
    """budget 3 selects a strict subset of both requests, 1 a single page,
    16 every full page (n <= k)."""
    assert _step_pin_holds(O.decode_step, budget)


def test_decode_step_unit_subset_and_scale():
    q, kc, vc, bt, lens, rec, codes = _fixture()
    res = O.decode_step(q, kc, vc, bt, lens, rec, H, G, BUDGET, units=[(1, 1)])
    assert list(res) == [(1, 1)]
    _, _, _, out = _expected_unit(q, kc, vc, bt, lens, codes, 1, 1, BUDGET)
    np.testing.assert_allclose(res[(1, 1)]["out"], out, atol=1e-12)
    # an explicit scale is used for attention (not for scoring)
    res2 = O.decode_step(q, kc, vc, bt, lens, rec, H, G, BUDGET, scale=SCALE, units=[(1, 1)])
    np.testing.assert_allclose(res2[(1, 1)]["out"], out, atol=1e-12)


def test_planted_step_slips_are_caught(monkeypatch):
    """Slips planted in wrapped copies of the oracle's whole-step functions
    (CPU only); each must fail a pin that the oracle passes."""
    assert _scores_pin_holds(O.unit_scores_from_records)
    assert _step_pin_holds(O.decode_step)

    # ---- unit_scores_from_records
    def other_head(qg, rec, bt_row, h, L):
        return O.unit_scores_from_records(qg, rec, bt_row, 1 - h, L)

    def physical_not_logical(qg, rec, bt_row, h, L):   # block ids 0..n-1 instead of the row
        return O.unit_scores_from_records(qg, rec, np.arange(len(bt_row)), h, L)

    def tail_page_scored(qg, rec, bt_row, h, L):       # counts the open page as full
        return O.unit_scores_from_records(qg, rec, bt_row, h, L + B - L % B)

    for bad in (other_head, physical_not_logical, tail_page_scored):
        assert not _scores_pin_holds(bad), bad.__name__

    # ---- decode_step
    def wrong_head_slice(q, kc, vc, bt, lens, rec, Hk, Gq, budget, **kw):
        return O.decode_step(np.roll(q, Gq, axis=1), kc, vc, bt, lens, rec, Hk, Gq, budget, **kw)

    def wrong_table_row(q, kc, vc, bt, lens, rec, Hk, Gq, budget, **kw):
        res = O.decode_step(q, kc, vc, bt[::-1].copy(), lens[::-1].copy(), rec, Hk, Gq, budget, **kw)
        return {(1 - b, h): v for (b, h), v in res.items()}

    def no_group_mean(q, kc, vc, bt, lens, rec, Hk, Gq, budget, **kw):   # first head's shares only
        qq = q.copy()
        for h in range(Hk):
            qq[:, h * Gq:(h + 1) * Gq] = q[:, h * Gq:h * Gq + 1]
        res = O.decode_step(qq, kc, vc, bt, lens, rec, Hk, Gq, budget, **kw)
        full = O.decode_step(q, kc, vc, bt, lens, rec, Hk, Gq, budget, **kw)
        for key in res:
            res[key]["scores"] = full[key]["scores"]
        return res

    for bad in (wrong_head_slice, wrong_table_row, no_group_mean):
        assert not _step_pin_holds(bad), bad.__name__

    # a dropped tail page, planted in the oracle's gather step itself
    real_gather = OL.gather_unit

    def gather_without_tail(cache, bt_row, h, pages, L):
        return real_gather(cache, bt_row, h, pages, L - L % B)

    monkeypatch.setattr(OL, "gather_unit", gather_without_tail)
    assert not _step_pin_holds(O.decode_step)
    monkeypatch.setattr(OL, "gather_unit", real_gather)

    # selection ranked by the raw scores summed over heads instead of the
    # normalised shares (a missing Z_g), planted in the oracle's select step
    real_select = OL.select_pages

    def select_unnormalised(s_hat, k):
        sel, avg = real_select(s_hat, k)
        raw = np.exp(s_hat).sum(axis=1)
        order = np.lexsort((np.arange(len(raw)), -raw))
        return np.sort(order[:min(k, len(raw))]), avg

    monkeypatch.setattr(OL, "select_pages", select_unnormalised)
    assert not _step_pin_holds(O.decode_step)
