"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test names the property it checks.  Together they are chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a missing normalisation) fails at least one of them; the
planted-mistake tests at the end demonstrate this for a few such slips.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
D = O.HEAD_DIM
B = O.PAGE_SIZE


def _rng(seed=0):
    return np.random.default_rng(seed)


def _lowrank_page(rng, rank, noise=0.0, integer=False):
    if integer:
        mu = rng.integers(-3, 4, size=D).astype(np.float64)
        U = rng.integers(-2, 3, size=(D, rank)).astype(np.float64)
        C = rng.integers(-3, 4, size=(B, rank)).astype(np.float64)
        return mu + C @ U.T
    mu = rng.normal(0, 0.5, size=D)
    U, _ = np.linalg.qr(rng.normal(size=(D, rank)))
    C = rng.normal(size=(B, rank)) * np.array([4, 3, 2, 1.5, 1, 0.8, 0.6, 0.5])[:rank]
    return mu + C @ U.T + noise * rng.normal(size=(B, D))


# ---------------------------------------------------------------- a1 build
def test_lowrank_integer_pages_reconstruct_exactly():
    """Keys with page rank <= r (integer valued, exact in bf16) come back exactly."""
    rng = _rng(1)
    for rank in (1, 3, 8):
        K = _lowrank_page(rng, rank, integer=True)
        assert np.abs(K).max() < 256  # exactly representable in bf16
        s = O.page_summary(K)
        Khat = s["mu"] + s["C"] @ s["V"].T
        np.testing.assert_allclose(Khat, K, atol=1e-10, rtol=0)


def test_eckart_young_tail_energy_and_residual_optimality():
    """||X - C V^T||_F^2 equals the spectral tail energy, and no random
    orthonormal rank-r basis does better (residual optimality, Thm. 1)."""
    rng = _rng(2)
    K = rng.normal(size=(B, D))
    s = O.page_summary(K)
    X = K - s["mu"]
    resid = np.sum((X - s["C"] @ s["V"].T) ** 2)
    np.testing.assert_allclose(resid, s["tail"], rtol=1e-10)
    np.testing.assert_allclose(s["tail"], s["lam"][O.RANK:].sum(), rtol=1e-12)
    for _ in range(20):
        Q, _ = np.linalg.qr(rng.normal(size=(D, O.RANK)))
        assert np.sum((X - X @ Q @ Q.T) ** 2) >= resid - 1e-9


def test_basis_orthonormal_and_coefficients_are_projections():
    rng = _rng(3)
    for noise in (0.05, 0.1):
        K = _lowrank_page(rng, 8, noise=noise)
        s = O.page_summary(K)
        np.testing.assert_allclose(s["V"].T @ s["V"], np.eye(O.RANK), atol=1e-10)
        np.testing.assert_allclose((K - s["mu"]) @ s["V"], s["C"], atol=1e-9)


def test_eigenvalues_match_independent_svd_and_centroid_is_mean():
    rng = _rng(4)
    K = rng.normal(size=(5, B, D))
    s = O.page_summary(K)
    X = K - K.mean(axis=1, keepdims=True)
    sv = np.linalg.svd(X, compute_uv=False)  # gesdd, a different LAPACK path
    np.testing.assert_allclose(s["lam"][:, :B], np.sort(sv ** 2, axis=-1)[:, ::-1], atol=1e-9)
    np.testing.assert_allclose(s["mu"], K.sum(axis=1) / B, atol=1e-13)
    assert np.all(np.diff(s["lam"], axis=-1) <= 1e-12)


def test_sign_convention_largest_coefficient_positive():
    rng = _rng(5)
    s = O.page_summary(rng.normal(size=(8, B, D)))
    C = s["C"]
    idx = np.argmax(np.abs(C), axis=-2)
    top = np.take_along_axis(C, idx[:, None, :], axis=-2)
    assert np.all(top > 0)


def test_degenerate_pages():
    rng = _rng(6)
    # cache values are bf16: 16 equal bf16 keys have an exact fp64 mean
    k = torch.from_numpy(rng.normal(size=D)).to(torch.bfloat16).double().numpy()
    s = O.page_summary(np.tile(k, (B, 1)))        # all keys equal
    np.testing.assert_allclose(s["mu"], k, atol=1e-14)
    assert np.all(s["V"] == 0) and np.all(s["C"] == 0) and s["tail"] == 0
    K = _lowrank_page(rng, 3, integer=True)       # rank 3 < r
    s = O.page_summary(K)
    assert np.all(s["V"][:, 3:] == 0) and np.all(s["C"][:, 3:] == 0)
    np.testing.assert_allclose(np.linalg.norm(s["V"][:, :3], axis=0), 1.0, atol=1e-12)


def test_full_rank_reconstruction_is_exact():
    """r = B (the full-rank reading of 'r = d') reproduces every key."""
    rng = _rng(7)
    K = rng.normal(size=(B, D))
    s = O.page_summary(K, rank=B)
    np.testing.assert_allclose(s["mu"] + s["C"] @ s["V"].T, K, atol=1e-10)


# ---------------------------------------------------------------- a2 quantise
def test_quantize_round_half_even_and_bounds():
    x = np.array([7.0, 0.5, 1.5, 2.5, -2.5, -0.5, 3.49, -7.0])
    codes, s = O.quantize_sym(x, 7, axes=(-1,))
    assert s.item() == 1.0
    assert codes.tolist() == [7, 0, 2, 2, -2, 0, 3, -7]
    rng = _rng(8)
    y = rng.normal(size=(4, 100))
    for qmax in (7, 127):
        c, s = O.quantize_sym(y, qmax, axes=(-1,))
        assert np.abs(c).max() <= qmax
        assert np.all(np.abs(c).max(axis=-1) == qmax)
        assert np.all(np.abs(y - s * c) <= s / 2 * (1 + 1e-6))
        assert s.dtype == np.float64 and np.all(s == s.astype(np.float32))
    c, s = O.quantize_sym(np.zeros(5), 127, axes=(-1,))
    assert s.item() == 0 and np.all(c == 0)


def test_record_size_is_about_a_tenth_of_page_kv():
    kv_bytes = 2 * B * D * 2          # K and V, bf16
    assert O.RECORD_BYTES == 512 + 128 + 128 + 16
    assert 0.09 <= O.RECORD_BYTES / kv_bytes <= 0.11


def test_record_layout_golden_positions():
    g = json.load(open(os.path.join(GOLD, "record_layout_positions.json")))
    for e in g["vq"]:
        assert O.vq_position(e["k"], e["dim"]) == (e["byte"], e["high"])
    for e in g["mu"]:
        assert O.mu_position(e["dim"]) == e["byte"]
    for e in g["c"]:
        assert O.c_position(e["i"], e["k"]) == e["byte"]
    # every byte of the quantised planes is used exactly once (nibbles: twice)
    vb = [O.vq_position(k, dd) for k in range(8) for dd in range(D)]
    assert len(set(vb)) == 1024 and {b for b, _ in vb} == set(range(512))
    assert sorted(O.mu_position(dd) for dd in range(D)) == list(range(512, 640))
    assert sorted(O.c_position(i, k) for i in range(B) for k in range(8)) == list(range(640, 768))


def test_record_roundtrip():
    rng = _rng(9)
    q = O.quantize_summary(O.page_summary(rng.normal(size=(3, 2, B, D))))
    rec = O.encode_records(q)
    assert rec.shape == (3, 2, 784) and rec.dtype == np.uint8
    back = O.decode_records(rec)
    for key in ("Vq", "muq", "Cq"):
        np.testing.assert_array_equal(back[key], q[key])
    for key in ("sV", "smu", "sC", "tail"):
        np.testing.assert_array_equal(back[key], q[key].astype(np.float32))


# ---------------------------------------------------------------- a3 score
def test_score_closed_form_unquantised_full_rank():
    """With r = B and no quantisation, s_j(q) is the exact page LSE."""
    rng = _rng(10)
    K = rng.normal(size=(6, B, D))
    q = rng.normal(size=(4, D))
    s = O.page_summary(K, rank=B)
    got = O.page_scores(q, s["mu"], s["V"], s["C"])
    exact = np.array([[math.log(sum(math.exp(float(q[g] @ K[p, i]) / math.sqrt(D))
                                    for i in range(B))) for g in range(4)] for p in range(6)])
    np.testing.assert_allclose(got, exact, atol=1e-11)
    np.testing.assert_allclose(O.exact_page_lse(q, K), exact, atol=1e-12)


def test_score_lowrank_page_exact_at_rank_8():
    rng = _rng(11)
    K = np.stack([_lowrank_page(rng, 8, integer=True) for _ in range(3)])
    q = rng.normal(size=(2, D))
    s = O.page_summary(K)
    np.testing.assert_allclose(O.page_scores(q, s["mu"], s["V"], s["C"]),
                               O.exact_page_lse(q, K), atol=1e-9)


def _two_level_page():
    K = np.zeros((B, D))
    K[1::2, 0] = math.sqrt(2.0)
    q = np.zeros((2, D))
    q[0, 0], q[1, 0] = 8.0, -8.0
    return K, q


def test_score_worked_example_golden_exact_and_quantised():
    g = json.load(open(os.path.join(GOLD, "score_two_level_page.json")))
    K, q = _two_level_page()
    s = O.page_summary(K)
    got = O.page_scores(q, s["mu"][None], s["V"][None], s["C"][None])[0]
    np.testing.assert_allclose(got, g["expected_s_hat"], atol=g["tolerance_exact"])
    # through quantisation and the byte record
    rec = O.build_records(K[None])
    dq = O.dequantize(O.decode_records(rec))
    qd = O.decode_records(rec)
    assert qd["muq"][0, 0] == 127 and abs(int(qd["Vq"][0, 0, 0])) == 7
    assert sorted(set(qd["Cq"][0, :, 0].tolist())) == [-127, 127]
    # odd tokens sit at +sqrt(2)/2 along e_0 whatever sign the basis takes
    assert np.all(qd["Vq"][0, 0, 0] * qd["Cq"][0, 1::2, 0] > 0)
    got_q = O.page_scores(q, dq["mu"], dq["V"], dq["C"])[0]
    np.testing.assert_allclose(got_q, g["expected_s_hat"], atol=g["tolerance_quantised"])


def _quantised_generic_pages():
    rng = _rng(13)
    K = np.stack([_lowrank_page(rng, 8, noise=0.05) for _ in range(5)] +
                 [rng.normal(size=(B, D)) for _ in range(3)])
    q = rng.normal(size=(4, D)) * 2.0
    return K, q, O.dequantize(O.decode_records(O.build_records(K)))


def _reconstruction_pin_holds(score_fn) -> bool:
    """The factored score q.mu + (V^T q).c_i equals, by linearity, attention
    to the 16 keys the summary reconstructs, k_i = mu + V c_i: those keys are
    formed explicitly and their log-sum-exp taken by torch (fp64, CPU)."""
    K, q, dq = _quantised_generic_pages()
    got = score_fn(q, dq["mu"], dq["V"], dq["C"])
    keys = dq["mu"][:, None, :] + np.einsum("pdr,pir->pid", dq["V"], dq["C"])   # [page, token, dim]
    logits = torch.from_numpy(np.einsum("gd,pid->pgi", q, keys) / math.sqrt(D))
    want = torch.logsumexp(logits, dim=-1).numpy()
    return bool(np.allclose(got, want, rtol=0, atol=1e-10))


def test_score_quantised_generic_pages_are_the_lse_of_their_reconstructed_keys():
    """Generic pages at rank 8 (five low-rank with noise, three iid), through
    quantisation and the byte record."""
    assert _reconstruction_pin_holds(O.page_scores)
    # the quantised summary really is a different page from the original:
    # the check is not the unquantised identity in disguise
    K, q, dq = _quantised_generic_pages()
    assert np.max(np.abs(O.page_scores(q, dq["mu"], dq["V"], dq["C"]) - O.exact_page_lse(q, K))) > 1e-4


def test_score_heads_are_independent_and_equivariant():
    rng = _rng(12)
    K = rng.normal(size=(4, B, D))
    q = rng.normal(size=(4, D))
    s = O.page_summary(K)
    full = O.page_scores(q, s["mu"], s["V"], s["C"])
    perm = [2, 0, 3, 1]
    np.testing.assert_allclose(O.page_scores(q[perm], s["mu"], s["V"], s["C"]), full[:, perm])
    np.testing.assert_allclose(O.page_scores(q[:1], s["mu"], s["V"], s["C"]), full[:, :1])


# ---------------------------------------------------------------- a4/a5 select
def test_select_golden_gqa_tables():
    g = json.load(open(os.path.join(GOLD, "gqa_select_tables.json")))
    for case in g["cases"]:
        m = np.array(case["masses"], dtype=np.float64)      # [G, n]
        s_hat = np.log(m).T                                 # [n, G]
        for k, want in case["select"].items():
            sel, avg = O.select_pages(s_hat, int(k))
            assert sel.tolist() == want, case["name"]
            np.testing.assert_allclose(avg, case["avg"], rtol=1e-14)


def test_select_brute_force_tiny():
    rng = _rng(13)
    for trial in range(200):
        n = int(rng.integers(1, 8))
        G = int(rng.choice([1, 2, 4]))
        k = int(rng.integers(1, 9))
        s_hat = rng.normal(size=(n, G)) * 2
        if trial % 5 == 0:  # plant exact ties
            s_hat[rng.integers(0, n)] = s_hat[0]
        sel, avg = O.select_pages(s_hat, k)
        shares = np.exp(s_hat) / np.exp(s_hat).sum(axis=0, keepdims=True)
        table = shares.mean(axis=1)
        kk = min(k, n)
        best = None
        for sub in itertools.combinations(range(n), kk):
            key = (-sum(sorted(table[list(sub)])), sub)   # max mass, then lexicographic
            # ties: the rule "lower index wins" == lexicographically smallest
            # among subsets whose sorted values are all maximal
            vals = sorted(table[list(sub)], reverse=True)
            cand = (tuple(-v for v in vals), sub)
            if best is None or cand < best:
                best = cand
        assert tuple(sel.tolist()) == best[1]
        np.testing.assert_allclose(avg, table, rtol=1e-12)


def test_select_single_head_is_topk_of_scores():
    rng = _rng(14)
    s_hat = rng.normal(size=(50, 1))
    sel, _ = O.select_pages(s_hat, 7)
    assert sel.tolist() == sorted(np.argsort(-s_hat[:, 0], kind="stable")[:7].tolist())


def test_select_all_when_few_pages_and_empty():
    sel, _ = O.select_pages(np.zeros((3, 4)), 16)
    assert sel.tolist() == [0, 1, 2]
    sel, avg = O.select_pages(np.zeros((0, 4)), 16)
    assert sel.size == 0 and avg.size == 0


# ---------------------------------------------------------------- a6/a7 attention
def test_attention_matches_library_sdpa_fp64():
    rng = _rng(15)
    q = rng.normal(size=(4, D))
    K = rng.normal(size=(37, D))
    V = rng.normal(size=(37, D))
    sc = 1 / math.sqrt(D)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K)[None, None].expand(1, 4, 37, D),
        torch.from_numpy(V)[None, None].expand(1, 4, 37, D), scale=sc)[0, :, 0].numpy()
    np.testing.assert_allclose(O.attention(q, K, V, sc), ref, atol=1e-12)


def test_attention_closed_forms():
    rng = _rng(16)
    q = rng.normal(size=(2, D))
    V = rng.normal(size=(5, D))
    np.testing.assert_allclose(O.attention(q, rng.normal(size=(1, D)), V[:1], 0.1), np.tile(V[0], (2, 1)))
    K = np.tile(rng.normal(size=D), (5, 1))
    np.testing.assert_allclose(O.attention(q, K, V, 0.1), np.tile(V.mean(0), (2, 1)), atol=1e-13)
    assert np.all(O.attention(q, np.zeros((0, D)), np.zeros((0, D)), 0.1) == 0)


def _tiny_cache(rng, L, H=2, extra=3):
    n_pages = -(-L // B)
    nblk = n_pages + extra
    kc = rng.normal(size=(nblk, H, B, D))
    vc = rng.normal(size=(nblk, H, B, D))
    bt = rng.permutation(nblk)[:n_pages]
    return kc, vc, bt


@pytest.mark.parametrize("L", [16 * 9, 16 * 9 + 1, 16 * 9 + 15, 5])
def test_sparse_with_all_pages_equals_dense_and_gathers_by_block_table(L):
    rng = _rng(17)
    kc, vc, bt = _tiny_cache(rng, L)
    q = rng.normal(size=(4, D))
    n, t = O.page_split(L)
    for h in range(2):
        dense = O.dense_attend_unit(q, kc, vc, bt, h, L, 0.09)
        sparse = O.sparse_attend_unit(q, kc, vc, bt, h, L, np.arange(n), 0.09)
        np.testing.assert_allclose(sparse, dense, atol=1e-14)
        toks = [kc[bt[j], h, i] for j in range(n) for i in range(B)]
        toks += [kc[bt[n], h, i] for i in range(t)]
        vals = [vc[bt[j], h, i] for j in range(n) for i in range(B)]
        vals += [vc[bt[n], h, i] for i in range(t)]
        ref = O.attention(q, np.array(toks).reshape(-1, D), np.array(vals).reshape(-1, D), 0.09)
        np.testing.assert_allclose(dense, ref, atol=1e-13)


def test_decode_step_full_rank_unquantised_matches_exact_selection():
    """Using exact page LSEs as scores (what r = B, no quantisation gives),
    LOCKS's selection is the read-every-key selection."""
    rng = _rng(18)
    L = 16 * 12 + 3
    kc, vc, bt = _tiny_cache(rng, L, H=1)
    q = rng.normal(size=(4, D))
    n, _ = O.page_split(L)
    pages = kc[bt[:n], 0]
    s = O.page_summary(pages, rank=B)
    via_summary = O.page_scores(q, s["mu"], s["V"], s["C"])
    exact = O.exact_page_lse(q, pages)
    np.testing.assert_allclose(via_summary, exact, atol=1e-10)
    assert O.select_pages(via_summary, 5)[0].tolist() == O.select_pages(exact, 5)[0].tolist()


# ---------------------------------------------------------------- planted mistakes
def _build_pins_hold(summary_fn) -> bool:
    rng = _rng(20)
    K = _lowrank_page(rng, 5, integer=True)
    s = summary_fn(K)
    if not np.allclose(s["mu"] + s["C"] @ s["V"].T, K, atol=1e-9):
        return False
    Kr = rng.normal(size=(B, D))
    s = summary_fn(Kr)
    if not np.allclose(s["V"].T @ s["V"], np.eye(O.RANK), atol=1e-9):
        return False
    resid = np.sum((Kr - s["mu"] - s["C"] @ s["V"].T) ** 2)
    return bool(np.isclose(resid, s["tail"], rtol=1e-9))


def _score_pin_holds(score_fn) -> bool:
    g = json.load(open(os.path.join(GOLD, "score_two_level_page.json")))
    K, q = _two_level_page()
    s = O.page_summary(K)
    got = score_fn(q, s["mu"][None], s["V"][None], s["C"][None])[0]
    return bool(np.allclose(got, g["expected_s_hat"], atol=1e-9))


def _select_pins_hold(select_fn) -> bool:
    g = json.load(open(os.path.join(GOLD, "gqa_select_tables.json")))
    for case in g["cases"]:
        s_hat = np.log(np.array(case["masses"], dtype=np.float64)).T
        for k, want in case["select"].items():
            if list(select_fn(s_hat, int(k))[0]) != want:
                return False
    return True


def test_planted_mistakes_are_caught():
    """Plant plausible slips in wrapped copies of the oracle's steps (CPU
    only) and check that the pins reject every one while accepting the oracle."""
    assert _build_pins_hold(O.page_summary)
    assert _score_pin_holds(O.page_scores)
    assert _select_pins_hold(O.select_pages)

    def no_centroid(K, rank=O.RANK):
        s = O.page_summary(K, rank)
        return dict(s, mu=0 * s["mu"])

    def flipped_coefficients(K, rank=O.RANK):
        s = O.page_summary(K, rank)
        return dict(s, C=-s["C"])

    def unnormalised_basis(K, rank=O.RANK):   # Lambda^{+1/2} lift
        s = O.page_summary(K, rank)
        lam = np.sqrt(np.clip(s["lam"][:rank], 0, None))
        return dict(s, V=s["V"] * lam, C=s["C"] / np.where(lam > 0, lam, 1))

    def smallest_eigenpairs(K, rank=O.RANK):
        s = O.page_summary(K, rank=B)
        return dict(s, V=s["V"][:, B - 1 - rank:B - 1], C=s["C"][:, B - 1 - rank:B - 1])

    for bad in (no_centroid, flipped_coefficients, unnormalised_basis, smallest_eigenpairs):
        assert not _build_pins_hold(bad), bad.__name__

    def score_no_centroid(q, mu, V, C):
        return O.page_scores(q, 0 * mu, V, C)

    def score_no_sqrt_d(q, mu, V, C):
        return O.page_scores(q, mu * math.sqrt(D), V * math.sqrt(D), C)

    def score_mean_not_lse(q, mu, V, C):
        qmu = mu @ q.T
        dev = np.einsum("pir,pgr->pgi", C, np.einsum("pdr,gd->pgr", V, q))
        return ((qmu[:, :, None] + dev) / math.sqrt(D)).mean(-1)

    for bad in (score_no_centroid, score_no_sqrt_d, score_mean_not_lse):
        assert not _score_pin_holds(bad), bad.__name__

    # slips a one-page golden cannot see: another page's coefficients, and
    # basis directions paired with the wrong coefficient columns
    def score_neighbour_coefficients(q, mu, V, C):
        return O.page_scores(q, mu, V, np.roll(C, 1, axis=0))

    def score_reversed_directions(q, mu, V, C):
        return O.page_scores(q, mu, V, C[:, :, ::-1])

    assert _reconstruction_pin_holds(O.page_scores)
    for bad in (score_no_centroid, score_no_sqrt_d, score_mean_not_lse, score_neighbour_coefficients,
                score_reversed_directions):
        assert not _reconstruction_pin_holds(bad), bad.__name__
    assert _score_pin_holds(score_neighbour_coefficients)   # invisible to the one-page golden

    def select_unnormalised(s_hat, k):
        return O.select_pages(s_hat - s_hat.max(), k) if s_hat.shape[1] == 1 else \
            (np.sort(np.lexsort((np.arange(len(s_hat)), -np.exp(s_hat).sum(1)))[:min(k, len(s_hat))]), None)

    def select_ties_to_higher_index(s_hat, k):
        _, avg = O.select_pages(s_hat, k)
        n = len(avg)
        order = np.lexsort((-np.arange(n), -avg))
        return np.sort(order[:min(k, n)]), avg

    def select_unsorted(s_hat, k):
        _, avg = O.select_pages(s_hat, k)
        return np.lexsort((np.arange(len(avg)), -avg))[:min(k, len(avg))], avg

    for bad in (select_unnormalised, select_ties_to_higher_index, select_unsorted):
        assert not _select_pins_hold(bad), bad.__name__
