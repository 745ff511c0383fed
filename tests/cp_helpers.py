"""Test harness for context-parallel shards: run several shards' decode_step
in one process (one thread per shard, gathers through a barrier), and an
oracle-backed shard that restates each shard's part in float64 on the CPU."""

from __future__ import annotations

import math
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle as O

LOG2E = 1.0 / math.log(2.0)


class ThreadGather:
    """all_gather between n shards running in n threads of one process."""

    def __init__(self, n: int, timeout: float = 300.0):
        self.n = n
        self.barrier = threading.Barrier(n, timeout=timeout)
        self.slots = [None] * n

    def for_shard(self, r: int):
        def gather(t):
            self.slots[r] = t
            self.barrier.wait()
            out = torch.stack([s.to(t.device) for s in self.slots])
            self.barrier.wait()
            return out
        return gather


def run_shards(step, shards, gather_cls=ThreadGather):
    """step(shard, all_gather) on every shard concurrently; results in shard order."""
    g = gather_cls(len(shards))
    with ThreadPoolExecutor(len(shards)) as ex:
        futs = [ex.submit(step, s, g.for_shard(r)) for r, s in enumerate(shards)]
        return [f.result() for f in futs]


class OracleShard:
    """One shard's part of the decode step, in float64 on the CPU: the same
    five calls as the library's CudaShard, written from the decomposition of
    the selection and attention over the shards' pages (shares normalised by
    Z_g = LSE over every shard's pages; the global top-k taken from the
    shards' local top-k lists; attention states merged by the online-softmax
    rule).  Scores come from the oracle's own records of the shard's pages."""

    def __init__(self, q, records, k_cache, v_cache, block_table, shard_lens, page_offset, budget, H, G,
                 shard, scale):
        self.q, self.rec, self.kc, self.vc = q, records, k_cache, v_cache
        self.bt, self.lens, self.off = block_table, shard_lens, page_offset
        self.budget, self.H, self.G, self.shard, self.scale = budget, H, G, shard, scale
        self.B = len(shard_lens)

    def _units(self):
        return [(b, h) for b in range(self.B) for h in range(self.H)]

    def score_pairs(self):
        self.x = {}
        pairs = torch.zeros(self.B, self.H, self.G, 2, dtype=torch.float64)
        for b, h in self._units():
            qg = self.q[b, h * self.G:(h + 1) * self.G]
            s_hat = O.unit_scores_from_records(qg, self.rec, self.bt[b], h, int(self.lens[b]))
            x = s_hat * LOG2E
            self.x[(b, h)] = x
            for g in range(self.G):
                if x.shape[0]:
                    m = x[:, g].max()
                    pairs[b, h, g, 0] = m
                    pairs[b, h, g, 1] = np.sum(np.exp2(x[:, g] - m))
                else:
                    pairs[b, h, g, 0] = -math.inf
        return pairs

    def select_local(self, pairs_all):
        pa = pairs_all.numpy()
        kb = max(1, self.budget)
        pages = torch.full((self.B, self.H, kb), -1, dtype=torch.int64)
        keys = torch.zeros(self.B, self.H, kb, dtype=torch.float64)
        counts = torch.zeros(self.B, self.H, dtype=torch.int64)
        self.avg = {}
        for b, h in self._units():
            z = np.zeros(self.G)
            for g in range(self.G):
                m = pa[:, b, h, g, 0]
                M = np.max(m)
                z[g] = M + np.log2(np.sum(pa[:, b, h, g, 1] * np.exp2(np.where(np.isfinite(m), m - M, -np.inf))))
            x = self.x[(b, h)]
            avg = np.exp2(x - z[None, :]).mean(axis=1) if x.shape[0] else np.zeros(0)
            n = avg.shape[0]
            kk = min(self.budget, n)
            order = sorted(range(n), key=lambda j: (-avg[j], j))[:kk]
            sel = sorted(order)
            counts[b, h] = kk
            for i, j in enumerate(sel):
                pages[b, h, i] = j + int(self.off[b])
                keys[b, h, i] = avg[j]
        return pages, keys, counts

    def merge_select(self, pages_all, keys_all, counts_all):
        self.sel = {}
        R = counts_all.shape[0]
        for b, h in self._units():
            cands = []
            for r in range(R):
                for i in range(int(counts_all[r, b, h])):
                    cands.append((-float(keys_all[r, b, h, i]), int(pages_all[r, b, h, i])))
            kk = min(self.budget, len(cands))
            top = sorted(cands)[:kk]
            mine = sorted(p - int(self.off[b]) for _, p in top
                          if 0 <= p - int(self.off[b]) < int(self.lens[b]) // O.PAGE_SIZE)
            self.sel[(b, h)] = mine

    def attend_partial(self):
        states = torch.zeros(self.B, self.H * self.G, 2 + O.HEAD_DIM, dtype=torch.float64)
        for b, h in self._units():
            K = O.gather_unit(self.kc, self.bt[b], h, self.sel[(b, h)], int(self.lens[b]))
            V = O.gather_unit(self.vc, self.bt[b], h, self.sel[(b, h)], int(self.lens[b]))
            qg = self.q[b, h * self.G:(h + 1) * self.G]
            for g in range(self.G):
                row = states[b, h * self.G + g]
                if K.shape[0] == 0:
                    row[0] = -math.inf
                    continue
                x = (K @ qg[g]) * self.scale * LOG2E
                m = x.max()
                p = np.exp2(x - m)
                row[0] = m
                row[1] = p.sum()
                row[2:] = torch.from_numpy(p @ V)
        return states

    def merge_attention(self, states_all):
        st = states_all.numpy()
        M = st[:, :, :, 0].max(axis=0)
        f = np.exp2(np.where(np.isfinite(st[:, :, :, 0]), st[:, :, :, 0] - M[None], -np.inf))
        Ls = (st[:, :, :, 1] * f).sum(axis=0)
        Os = (st[:, :, :, 2:] * f[..., None]).sum(axis=0)
        return torch.from_numpy(Os / np.where(Ls > 0, Ls, 1.0)[..., None])

    def selected_global(self):
        return {(b, h): [j + int(self.off[b]) for j in self.sel[(b, h)]] for b, h in self._units()}
