"""LOCKS decode hot path, restated step by step in float64 on the CPU.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (CPU baseline / reference arm)
may import this module.  It shares no code with the CUDA library.

Citations use the title of the source page and its section:
  [LOCKS §2]      "LOCKS: Page-Local Compact Key Summaries for Efficient
                  Long-Context Decoding", technical summary, §2 "Method: LOCKS"
                  (page-local spectral decomposition, quantisation,
                  reconstruction and selection, group-shared selection (GQA)).
  [LOCKS eq. s]   the same section's single equation, the within-page logit
                  reconstruction  s_j(q) = log sum_{i in P_j}
                  exp((q^T mu_j + (V_j^T q)^T c_i) / sqrt(d)).
  [LOCKS §3]      the same summary, §3 "Main contributions" (Thm. 1: error
                  controlled by the spectral tail energy; page-local basis is
                  residual-optimal among orthogonal rank-r reconstructions).
  [LOCKS abstract] the arXiv abstract: each page's attention mass is
                  estimated from its summary by a log-sum-exp, only the
                  highest-ranked pages are attended, and ranking them reads no
                  cached key or value.

Readings of points the pages leave open:
  * eigendecomposition of the 16x16 Gram matrix of the centred keys (same
    non-zero spectrum as the d x d covariance); eigenvalues <= 1e-6 * lambda_1
    give a zero basis column;
  * sign convention: for each basis direction k the token coefficient c_ik of
    largest magnitude is positive (lowest token index on exact ties);
  * quantisation: symmetric, one fp32 scale per tensor per page
    (s = max|x| / qmax), round half to even, V in int4 [-7, 7], mu and c in
    int8 [-127, 127]; a zero tensor has scale 0 and codes 0; c is quantised
    from the unquantised coefficients;
  * 1/sqrt(d) multiplies the whole logit; per-head shares are a softmax over
    the *full* pages only; the GQA table is the arithmetic mean of the shares;
    ties go to the lower page index; n <= k selects every full page;
  * the token budget counts full pages only; the partially filled tail page
    (no summary yet) is always attended.

Parity pins (tests/test_oracle_pins.py, tests/test_oracle_step_pins.py): every
public function below is pinned against closed forms, hand-derived fixtures
under tests/golden/, brute force, an independent library routine, or (for the
whole-step functions unit_scores_from_records and decode_step) a paged cache
whose scores, selection and attention are gathered by hand.  The quantised
rank-8 score of a generic page has no printed value on the pages: it is
pinned to the log-sum-exp of the keys its summary reconstructs (linearity of the score equation, evaluated by
torch), to the exact-quantisation worked example
(tests/golden/score_two_level_page.json) and to the closed form of the
unquantised full-rank path.
"""

from __future__ import annotations

import numpy as np

PAGE_SIZE = 16          # B, tokens per page                      [LOCKS §2]
HEAD_DIM = 128          # d
RANK = 8                # r                                       [LOCKS §2]
RECORD_BYTES = 784      # one quantised page-head summary (layout in include/locks.h)
V_QMAX = 7              # int4 basis                              [LOCKS §2]
MU_QMAX = 127           # int8 centroid                           [LOCKS §2]
C_QMAX = 127            # int8 coefficients                       [LOCKS §2]
EIG_REL_FLOOR = 1e-6


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def logsumexp(x: np.ndarray, axis: int) -> np.ndarray:
    """log(sum(exp(x))) along ``axis`` with the usual max shift."""
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=axis, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore"):
        out = m + np.log(np.sum(np.exp(x - m), axis=axis, keepdims=True))
    return np.squeeze(out, axis=axis)


# --------------------------------------------------------------------------
# a1: page-local spectral summary                                  [LOCKS §2]
# --------------------------------------------------------------------------
def page_summary(K: np.ndarray, rank: int = RANK) -> dict:
    """Summary of full pages of keys.

    K: [..., 16, d] keys of finalised pages (float64 copies of the bf16 cache).
    Steps, in the order of [LOCKS §2] "page-local spectral decomposition":
      1. centroid mu_j = mean of the page's keys;
      2. deviations X = K - mu_j (centred keys);
      3. small eigendecomposition: Gram matrix X X^T (16 x 16), eigenpairs
         sorted by decreasing eigenvalue (numpy.linalg.eigh is the library
         step);
      4. keep the top ``rank`` eigenvectors W_r; key-space basis
         V_j = X^T W_r Lambda_r^{-1/2} (orthonormal columns) and per-token
         coefficients C = W_r Lambda_r^{1/2} (= X V_j).
    Returns dict(mu [...,d], V [...,d,r], C [...,16,r], lam [...,16] descending,
    tail [...] = sum of the eigenvalues beyond rank r, the spectral tail
    energy of [LOCKS §3] Thm. 1).
    """
    K = np.asarray(K, dtype=np.float64)
    mu = K.mean(axis=-2)
    X = K - mu[..., None, :]
    G = X @ np.swapaxes(X, -1, -2)
    lam, W = np.linalg.eigh(G)
    lam = lam[..., ::-1]
    W = W[..., :, ::-1]
    big = np.argmax(np.abs(W), axis=-2)
    sgn = np.sign(np.take_along_axis(W, big[..., None, :], axis=-2))
    sgn = np.where(sgn == 0, 1.0, sgn)
    W = W * sgn
    lam_r = lam[..., :rank]
    keep = (lam_r > EIG_REL_FLOOR * lam[..., :1]) & (lam_r > 0)
    sig = np.sqrt(np.where(keep, lam_r, 1.0))
    W_r = W[..., :, :rank]
    V = (np.swapaxes(X, -1, -2) @ W_r) / sig[..., None, :] * keep[..., None, :]
    C = W_r * sig[..., None, :] * keep[..., None, :]
    tail = np.clip(lam[..., rank:], 0.0, None).sum(axis=-1)
    return {"mu": mu, "V": V, "C": C, "lam": lam, "tail": tail}


# --------------------------------------------------------------------------
# a2: quantisation                                                 [LOCKS §2]
# --------------------------------------------------------------------------
def quantize_sym(x: np.ndarray, qmax: int, axes) -> tuple[np.ndarray, np.ndarray]:
    """Symmetric quantisation with one fp32 scale over ``axes``.

    s = fp32(max|x| / qmax); code = round_half_even(x / s) clipped to
    [-qmax, qmax]; a zero tensor gets s = 0 and codes 0.
    Returns (codes int8, s float64 holding the fp32 value, keepdims).
    """
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=axes, keepdims=True)
    s = (amax / qmax).astype(np.float32).astype(np.float64)
    safe = np.where(s > 0, s, 1.0)
    codes = np.where(s > 0, np.rint(x / safe), 0.0)
    codes = np.clip(codes, -qmax, qmax).astype(np.int8)
    return codes, s


def quantize_summary(summ: dict) -> dict:
    """int4 basis, int8 centroid and coefficients, one scale each per page."""
    Vq, sV = quantize_sym(summ["V"], V_QMAX, axes=(-2, -1))
    Mq, sM = quantize_sym(summ["mu"], MU_QMAX, axes=(-1,))
    Cq, sC = quantize_sym(summ["C"], C_QMAX, axes=(-2, -1))
    return {
        "Vq": Vq, "sV": sV[..., 0, 0],
        "muq": Mq, "smu": sM[..., 0],
        "Cq": Cq, "sC": sC[..., 0, 0],
        "tail": np.asarray(summ["tail"], dtype=np.float64),
    }


def dequantize(q: dict) -> dict:
    """mu_hat = s_mu mu_q, V_hat = s_V V_q, C_hat = s_c c_q."""
    return {
        "mu": q["smu"][..., None] * q["muq"].astype(np.float64),
        "V": q["sV"][..., None, None] * q["Vq"].astype(np.float64),
        "C": q["sC"][..., None, None] * q["Cq"].astype(np.float64),
    }


# --------------------------------------------------------------------------
# the 784-byte record (layout documented in include/locks.h)
# --------------------------------------------------------------------------
def vq_position(k: int, dim: int) -> tuple[int, int]:
    """(byte offset, 1 if high nibble) of basis code V[dim, k] in a record."""
    s, w = divmod(dim, 16)
    hh, w8 = divmod(w, 8)
    t, e = divmod(w8, 2)
    p, sp = divmod(s, 2)
    m = 2 * sp + hh + 4 * e
    return k * 64 + t * 16 + p * 4 + m // 2, m % 2


def mu_position(dim: int) -> int:
    """byte offset of centroid code mu[dim] in a record."""
    s, w = divmod(dim, 16)
    hh, w8 = divmod(w, 8)
    t, e = divmod(w8, 2)
    return 512 + t * 32 + s * 4 + hh * 2 + e


def c_position(i: int, k: int) -> int:
    """byte offset of coefficient code c[i, k] (token i, direction k)."""
    nt, gid = divmod(i, 8)
    t, e = divmod(k, 2)
    return 640 + (gid * 4 + t) * 4 + nt * 2 + e


def _index_tables():
    vb = np.zeros((HEAD_DIM, RANK), dtype=np.int64)
    vh = np.zeros((HEAD_DIM, RANK), dtype=np.int64)
    for dim in range(HEAD_DIM):
        for k in range(RANK):
            vb[dim, k], vh[dim, k] = vq_position(k, dim)
    mb = np.array([mu_position(dim) for dim in range(HEAD_DIM)], dtype=np.int64)
    cb = np.array([[c_position(i, k) for k in range(RANK)] for i in range(PAGE_SIZE)],
                  dtype=np.int64)
    return vb, vh, mb, cb


_VB, _VH, _MB, _CB = _index_tables()


def encode_records(q: dict) -> np.ndarray:
    """Quantised summaries [..., *] -> uint8 records [..., 784]."""
    Vq = np.asarray(q["Vq"], dtype=np.int64)
    lead = Vq.shape[:-2]
    P = int(np.prod(lead)) if lead else 1
    Vq = Vq.reshape(P, HEAD_DIM, RANK)
    Mq = np.asarray(q["muq"], dtype=np.int64).reshape(P, HEAD_DIM)
    Cq = np.asarray(q["Cq"], dtype=np.int64).reshape(P, PAGE_SIZE, RANK)
    rec = np.zeros((P, RECORD_BYTES), dtype=np.int64)
    nib = (Vq & 0xF) << (4 * _VH[None])
    rows = np.arange(P)[:, None, None]
    np.add.at(rec, (np.broadcast_to(rows, nib.shape), np.broadcast_to(_VB[None], nib.shape)), nib)
    rec[:, _MB] = Mq & 0xFF
    rec[:, _CB] = Cq & 0xFF
    scales = np.stack([
        np.asarray(q["sV"], dtype=np.float64).reshape(P),
        np.asarray(q["smu"], dtype=np.float64).reshape(P),
        np.asarray(q["sC"], dtype=np.float64).reshape(P),
        np.asarray(q["tail"], dtype=np.float64).reshape(P),
    ], axis=-1).astype("<f4")
    out = rec.astype(np.uint8)
    out[:, 768:784] = scales.view(np.uint8).reshape(P, 16)
    return out.reshape(*lead, RECORD_BYTES)


def decode_records(rec: np.ndarray) -> dict:
    """uint8 records [..., 784] -> dict(Vq, muq, Cq int8; sV, smu, sC, tail)."""
    rec = np.asarray(rec, dtype=np.uint8)
    lead = rec.shape[:-1]
    R = rec.reshape(-1, RECORD_BYTES)
    P = R.shape[0]
    nib = (R[:, _VB].astype(np.int64) >> (4 * _VH[None])) & 0xF
    Vq = np.where(nib >= 8, nib - 16, nib).astype(np.int8)
    Mq = R[:, _MB].view(np.int8).copy()
    Cq = R[:, _CB].view(np.int8).copy()
    sc = np.ascontiguousarray(R[:, 768:784]).view("<f4").reshape(P, 4).astype(np.float64)
    return {
        "Vq": Vq.reshape(*lead, HEAD_DIM, RANK),
        "muq": Mq.reshape(*lead, HEAD_DIM),
        "Cq": Cq.reshape(*lead, PAGE_SIZE, RANK),
        "sV": sc[:, 0].reshape(lead), "smu": sc[:, 1].reshape(lead),
        "sC": sc[:, 2].reshape(lead), "tail": sc[:, 3].reshape(lead),
    }


def build_records(K_pages: np.ndarray) -> np.ndarray:
    """a1 + a2 for pages [..., 16, d] -> records [..., 784]."""
    return encode_records(quantize_summary(page_summary(K_pages)))


# --------------------------------------------------------------------------
# a3: within-page logit reconstruction                         [LOCKS eq. s]
# --------------------------------------------------------------------------
def page_scores(q: np.ndarray, mu: np.ndarray, V: np.ndarray, C: np.ndarray,
                head_dim: int = HEAD_DIM) -> np.ndarray:
    """s_j(q) for every page j and every query row of q.

    q: [G, d]; mu: [P, d]; V: [P, d, r]; C: [P, 16, r]  ->  [P, G]
    s_j(q) = log sum_i exp((q . mu_j + (V_j^T q) . c_i) / sqrt(d)): the log of
    page j's (unnormalised) attention mass estimated from the summary alone.
    """
    q = np.asarray(q, dtype=np.float64)
    qmu = np.asarray(mu, dtype=np.float64) @ q.T                       # [P, G]
    u = np.einsum("pdr,gd->pgr", np.asarray(V, dtype=np.float64), q)   # V_j^T q
    dev = np.einsum("pir,pgr->pgi", np.asarray(C, dtype=np.float64), u)
    logits = (qmu[:, :, None] + dev) / np.sqrt(head_dim)
    return logsumexp(logits, axis=-1)


# --------------------------------------------------------------------------
# a4 + a5: per-head shares, GQA average, top-k          [LOCKS §2, abstract]
# --------------------------------------------------------------------------
def select_pages(s_hat: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Pages of one (request, KV head) to attend.

    s_hat: [n, G] estimated log page masses of the n full pages for the G
    query heads of the group.  Per head, Z_g = logsumexp_j s_hat[j, g] and
    share = exp(s_hat - Z_g); the shared table is the mean over the group's
    heads; the k' = min(k, n) largest entries are selected (lower page index
    wins ties) and returned in ascending page order, with the table.
    """
    s_hat = np.asarray(s_hat, dtype=np.float64)
    n = s_hat.shape[0]
    if n == 0:
        return np.zeros(0, dtype=np.int64), np.zeros(0)
    Z = logsumexp(s_hat, axis=0)
    share = np.exp(s_hat - Z[None, :])
    avg = share.mean(axis=1)
    kk = min(int(k), n)
    order = np.lexsort((np.arange(n), -avg))
    return np.sort(order[:kk]).astype(np.int64), avg


# --------------------------------------------------------------------------
# a6 / a7: softmax attention over gathered tokens
# --------------------------------------------------------------------------
def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q K^T * scale) V for q [G, d], K/V [T, d] -> [G, d] (zeros if T=0)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[-1]))
    logits = (q @ K.T) * scale
    m = logits.max(axis=-1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ V


def page_split(L: int) -> tuple[int, int]:
    """(full pages n, tail tokens t) of a sequence of L cached tokens."""
    return L // PAGE_SIZE, L % PAGE_SIZE


def gather_unit(cache: np.ndarray, bt_row: np.ndarray, h: int, pages, L: int) -> np.ndarray:
    """Tokens of the listed full logical pages, then the tail page's t tokens."""
    n, t = page_split(L)
    parts = [cache[int(bt_row[int(j)]), h] for j in pages]
    if t > 0:
        parts.append(cache[int(bt_row[n]), h, :t])
    if not parts:
        return np.zeros((0, cache.shape[-1]))
    return np.concatenate(parts, axis=0).astype(np.float64)


def sparse_attend_unit(q_grp, k_cache, v_cache, bt_row, h, L, selected, scale):
    """a6: attention of the group's G queries over the selected full pages
    plus the open tail page."""
    K = gather_unit(k_cache, bt_row, h, selected, L)
    V = gather_unit(v_cache, bt_row, h, selected, L)
    return attention(q_grp, K, V, scale)


def dense_attend_unit(q_grp, k_cache, v_cache, bt_row, h, L, scale):
    """a7: attention over every cached token of the unit."""
    n, _ = page_split(L)
    return sparse_attend_unit(q_grp, k_cache, v_cache, bt_row, h, L, range(n), scale)


# --------------------------------------------------------------------------
# O7: the read-every-key selection (quality reference)    [LOCKS abstract]
# --------------------------------------------------------------------------
def exact_page_lse(q: np.ndarray, K_pages: np.ndarray, head_dim: int = HEAD_DIM) -> np.ndarray:
    """Exact log page mass log sum_i exp(q . k_i / sqrt(d)); K_pages [P,16,d] -> [P,G]."""
    q = np.asarray(q, dtype=np.float64)
    logits = np.einsum("pid,gd->pgi", np.asarray(K_pages, dtype=np.float64), q)
    return logsumexp(logits / np.sqrt(head_dim), axis=-1)


# --------------------------------------------------------------------------
# whole decode step over a paged cache (unit = one request x one KV head)
# --------------------------------------------------------------------------
def unit_scores_from_records(q_grp, records, bt_row, h, L):
    """s_hat [n, G] of the unit's full pages, read from the stored records."""
    n, _ = page_split(L)
    if n == 0:
        return np.zeros((0, q_grp.shape[0]))
    blocks = np.asarray(bt_row[:n], dtype=np.int64)
    d = dequantize(decode_records(records[blocks, h]))
    return page_scores(q_grp, d["mu"], d["V"], d["C"])


def decode_step(q, k_cache, v_cache, block_table, seq_lens, records, num_kv_heads,
                group, budget_pages, scale=None, units=None):
    """Score, select and attend for the listed (b, h) units (default: all).

    q: [batch, Hkv*G, d]; caches [nblk, Hkv, 16, d]; block_table [batch, max_pages];
    seq_lens [batch]; records [nblk, Hkv, 784].
    Returns dict keyed by (b, h): scores [n, G], avg [n], selected, out [G, d].
    """
    if scale is None:
        scale = 1.0 / np.sqrt(HEAD_DIM)
    batch = q.shape[0]
    if units is None:
        units = [(b, h) for b in range(batch) for h in range(num_kv_heads)]
    res = {}
    for b, h in units:
        L = int(seq_lens[b])
        qg = np.asarray(q[b, h * group:(h + 1) * group], dtype=np.float64)
        s_hat = unit_scores_from_records(qg, records, block_table[b], h, L)
        sel, avg = select_pages(s_hat, budget_pages)
        out = sparse_attend_unit(qg, k_cache, v_cache, block_table[b], h, L, sel, scale)
        res[(b, h)] = {"scores": s_hat, "avg": avg, "selected": sel, "out": out}
    return res
