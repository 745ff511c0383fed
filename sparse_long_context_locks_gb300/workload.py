"""Seeded synthetic decode workloads (inputs only -- no LOCKS arithmetic).

This module is the one piece both the CUDA path's tests/bench and the fp64
oracle consume: it draws queries, a paged bf16 K/V cache, a block table and
sequence lengths.  It computes nothing of the method itself.

Key generator (per page j and KV head h), following the workload description
that accompanies the LOCKS study of page-local low-rank keys:
    K = mu_j + C U_j^T + eps,   mu_j ~ N(0, 0.5^2) per coordinate,
    U_j = orthonormal d x 8 basis (Gram-Schmidt of a Gaussian matrix),
    C[:, k] ~ N(0, sigma_k^2), sigma = (4, 3, 2, 1.5, 1, 0.8, 0.6, 0.5),
    eps ~ N(0, noise^2);   or K ~ N(0, 1) iid in the "fullrank" regime.
Values and queries ~ N(0, 1).  Everything is rounded to bf16.
Carrier tokens: per KV head, ``carriers_per_head`` distinct full pages get one
key (random slot) equal to 6 * qbar / |qbar|, qbar = mean of the group's
queries.  Physical blocks are a seeded permutation, so kernels must go through
the block table.  A request's context N excludes the token being decoded; the
cache holds L = N + 1 tokens (the current token's K/V already appended).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

PAGE = 16
HEAD_DIM = 128
SIGMAS = (4.0, 3.0, 2.0, 1.5, 1.0, 0.8, 0.6, 0.5)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    context: int                      # N, or lower bound when context_hi is set
    num_kv_heads: int
    group: int                        # G query heads per KV head
    budget_tokens: int
    carriers_per_head: int
    noise_std: float = 0.05
    key_regime: str = "lowrank"       # "lowrank" | "fullrank"
    context_hi: Optional[int] = None  # per-request N ~ U{context..context_hi}
    seed: int = 1234
    head_dim: int = HEAD_DIM

    @property
    def budget_pages(self) -> int:
        return self.budget_tokens // PAGE

    @property
    def max_context(self) -> int:
        return self.context_hi if self.context_hi is not None else self.context

    @property
    def max_pages(self) -> int:
        return -(-(self.max_context + 1) // PAGE)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the study's decode path is characterised on.
CONFIGS = {
    "pr1_4k": Workload("pr1_4k", batch=1, context=4096, num_kv_heads=1, group=4,
                       budget_tokens=256, carriers_per_head=4),
    "llama8b_128k": Workload("llama8b_128k", batch=1, context=131072, num_kv_heads=8,
                             group=4, budget_tokens=2048, carriers_per_head=16),
    "batch16_32k": Workload("batch16_32k", batch=16, context=24576, context_hi=32768,
                            num_kv_heads=8, group=4, budget_tokens=2048,
                            carriers_per_head=8),
    "ctx1m": Workload("ctx1m", batch=1, context=1048576, num_kv_heads=8, group=4,
                      budget_tokens=2048, carriers_per_head=16, noise_std=0.1),
    "batch64_256k_lowrank": Workload("batch64_256k_lowrank", batch=64, context=262144,
                                     num_kv_heads=8, group=4, budget_tokens=2048,
                                     carriers_per_head=8),
    "batch64_256k_fullrank": Workload("batch64_256k_fullrank", batch=64, context=262144,
                                      num_kv_heads=8, group=4, budget_tokens=2048,
                                      carriers_per_head=8, key_regime="fullrank"),
    # the batch-64 attention and selection shapes (512 units, 128 selected
    # pages each: 537 MB of K/V a step) on a cache small enough (2.1 GB of K
    # and V) for counter captures of single kernels
    "batch64_8k": Workload("batch64_8k", batch=64, context=8192, num_kv_heads=8, group=4,
                           budget_tokens=2048, carriers_per_head=4),
}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1000003 + stream * 7919 + 17) % (2 ** 63 - 1))
    return g


def request_lengths(w: Workload) -> list[int]:
    """Cached tokens L_b = N_b + 1 per request (seeded)."""
    if w.context_hi is None:
        return [w.context + 1] * w.batch
    g = _gen(w.seed, 999_999, "cpu")
    n = torch.randint(w.context, w.context_hi + 1, (w.batch,), generator=g)
    return [int(x) + 1 for x in n]


def _orthonormal_columns(A: torch.Tensor) -> torch.Tensor:
    """Modified Gram-Schmidt on the last two dims of A [..., d, r]."""
    cols = []
    for k in range(A.shape[-1]):
        v = A[..., k]
        for u in cols:
            v = v - (v * u).sum(-1, keepdim=True) * u
        v = v / v.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        cols.append(v)
    return torch.stack(cols, dim=-1)


def _draw_keys(npages: int, H: int, d: int, w: Workload, g: torch.Generator,
               device) -> torch.Tensor:
    if w.key_regime == "fullrank":
        return torch.randn(npages, H, PAGE, d, generator=g, device=device)
    mu = torch.randn(npages, H, 1, d, generator=g, device=device) * 0.5
    U = _orthonormal_columns(torch.randn(npages, H, d, 8, generator=g, device=device))
    sig = torch.tensor(SIGMAS, device=device)
    C = torch.randn(npages, H, PAGE, 8, generator=g, device=device) * sig
    eps = torch.randn(npages, H, PAGE, d, generator=g, device=device) * w.noise_std
    return mu + C @ U.transpose(-1, -2) + eps


def generate(w: Workload, device="cpu", chunk_pages: int = 4096,
             tail_fill: str = "zero", extra_blocks: int = 0) -> dict:
    """Draw one decode step's inputs.

    Returns dict with q [batch, Hkv*G, d] bf16, k_cache / v_cache
    [num_blocks, Hkv, 16, d] bf16, block_table [batch, max_pages] int32 (-1 =
    unused), seq_lens [batch] int32, carriers: list of (b, h, page, slot),
    plus the workload.  ``tail_fill`` chooses what the unwritten slots of each
    tail page hold: "zero", "nan" or "huge" (kernels must never use them).
    """
    device = torch.device(device)
    H, G, d = w.num_kv_heads, w.group, w.head_dim
    lens = request_lengths(w)
    pages_per_req = [-(-L // PAGE) for L in lens]
    total = sum(pages_per_req) + extra_blocks
    perm = torch.randperm(total, generator=_gen(w.seed, 888_888, "cpu"))
    k_cache = torch.empty(total, H, PAGE, d, dtype=torch.bfloat16, device=device)
    v_cache = torch.empty_like(k_cache)
    if extra_blocks:
        k_cache.zero_()
        v_cache.zero_()
    max_pages = w.max_pages
    block_table = torch.full((w.batch, max_pages), -1, dtype=torch.int32)
    q_all = torch.empty(w.batch, H * G, d, dtype=torch.bfloat16, device=device)
    carriers = []
    off = 0
    for b in range(w.batch):
        L, npg = lens[b], pages_per_req[b]
        g = _gen(w.seed, b, device)
        q = torch.randn(H * G, d, generator=g, device=device).to(torch.bfloat16)
        q_all[b] = q
        blocks = perm[off:off + npg]
        off += npg
        block_table[b, :npg] = blocks.to(torch.int32)
        blocks_dev = blocks.to(device)
        for p0 in range(0, npg, chunk_pages):
            p1 = min(npg, p0 + chunk_pages)
            K = _draw_keys(p1 - p0, H, d, w, g, device)
            V = torch.randn(p1 - p0, H, PAGE, d, generator=g, device=device)
            k_cache[blocks_dev[p0:p1]] = K.to(torch.bfloat16)
            v_cache[blocks_dev[p0:p1]] = V.to(torch.bfloat16)
        # planted carriers: one key per chosen full page, per KV head
        n_full = L // PAGE
        gc = _gen(w.seed, 500_000 + b, "cpu")
        qf = q.float().view(H, G, d).mean(dim=1)
        qf = qf / qf.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        for h in range(H):
            m = min(w.carriers_per_head, n_full)
            if m == 0:
                continue
            pages = torch.randperm(n_full, generator=gc)[:m]
            slots = torch.randint(0, PAGE, (m,), generator=gc)
            for j, s in zip(pages.tolist(), slots.tolist()):
                blk = int(block_table[b, j])
                k_cache[blk, h, s] = (6.0 * qf[h]).to(torch.bfloat16)
                carriers.append((b, h, j, s))
        # unwritten slots of the open tail page
        t = L % PAGE
        if t:
            blk = int(block_table[b, L // PAGE])
            fill = {"zero": 0.0, "nan": float("nan"), "huge": 3.0e38}[tail_fill]
            k_cache[blk, :, t:] = fill
            v_cache[blk, :, t:] = fill
    return {
        "workload": w,
        "q": q_all,
        "k_cache": k_cache,
        "v_cache": v_cache,
        "block_table": block_table.to(device),
        "seq_lens": torch.tensor(lens, dtype=torch.int32, device=device),
        "carriers": carriers,
        "num_blocks": total,
    }


def full_page_blocks(data: dict) -> torch.Tensor:
    """Physical blocks of every full (finalised) page, request-major order."""
    bt = data["block_table"].cpu()
    lens = data["seq_lens"].cpu().tolist()
    out = [bt[b, :L // PAGE] for b, L in enumerate(lens)]
    return torch.cat(out).to(torch.int32) if out else torch.zeros(0, dtype=torch.int32)


def algorithmic_bytes(lens: Sequence[int], num_kv_heads: int, group: int,
                      budget_pages: int, record_bytes: int = 784,
                      head_dim: int = HEAD_DIM) -> dict:
    """Bytes a decode step must move at minimum (per layer).

    score/select: every full page's record per KV head; sparse attention: the
    selected pages' K and V plus the tail tokens; dense: every cached token.
    q (bf16) and out (fp32) are counted once each.
    """
    kv_page = 2 * PAGE * head_dim * 2
    kv_tok = 2 * head_dim * 2
    score = sparse = dense = 0
    for L in lens:
        n, t = L // PAGE, L % PAGE
        score += num_kv_heads * n * record_bytes
        sparse += num_kv_heads * (min(budget_pages, n) * kv_page + t * kv_tok)
        dense += num_kv_heads * (n * kv_page + t * kv_tok)
    io = len(lens) * num_kv_heads * group * head_dim * (2 + 4)
    return {"score": score, "sparse_kv": sparse, "dense_kv": dense,
            "step": score + sparse + io, "dense_step": dense + io}
