"""Context-parallel LOCKS decode step: one request's full pages split over
several GPUs (shards), each holding a contiguous range of logical pages in its
own K/V cache, summaries and block table.

The selection of "LOCKS: Page-Local Compact Key Summaries for Efficient
Long-Context Decoding" (technical summary §2, "Reconstruction and selection",
"Group-shared selection (GQA)") normalises every query head's page scores over
all of the request's pages and keeps the k largest group-mean shares, so a
sharded request needs three gathers of small per-shard results (see
include/locks.h): the (max, sum) pairs that make Z_g, each shard's local top-k
candidates, and the unnormalised attention states.  Everything computed runs
in the library's kernels; this module only sequences the calls and moves the
gathered tensors, through whatever all-gather the caller provides.

  shard = CudaShard(...)                      # one per GPU
  out = decode_step(shard, host_all_gather())  # same call on every shard
"""

from __future__ import annotations

from typing import Callable

import torch

from . import locks as L


class CudaShard:
    """One shard's inputs and device buffers, and its five library calls."""

    def __init__(self, num_kv_heads: int, q, summaries, k_cache, v_cache, block_table, shard_lens,
                 page_offset, budget_pages: int, shard: int, sm_scale=None, stream=None):
        self.H = num_kv_heads
        self.q, self.summ, self.k, self.v = q, summaries, k_cache, v_cache
        self.bt, self.lens, self.off = block_table, shard_lens, page_offset
        self.budget, self.shard, self.scale, self.stream = budget_pages, shard, sm_scale, stream
        B, MP = block_table.shape
        self.B, self.MP = B, MP
        dev = q.device
        self.bufs = L.DecodeBuffers(num_kv_heads, B, MP, budget_pages, device=dev)
        kb = max(1, budget_pages)
        self.pairs = torch.empty(B, num_kv_heads, L.GROUP, 2, dtype=torch.float32, device=dev)
        self.cand_pages = torch.full((B, num_kv_heads, kb), -1, dtype=torch.int32, device=dev)
        self.cand_keys = torch.zeros(B, num_kv_heads, kb, dtype=torch.int32, device=dev)
        self.cand_counts = torch.zeros(B, num_kv_heads, dtype=torch.int32, device=dev)
        self.states = torch.empty(B, num_kv_heads * L.GROUP, 2 + L.HEAD_DIM, dtype=torch.float32, device=dev)
        self.out = torch.empty(B, num_kv_heads * L.GROUP, L.HEAD_DIM, dtype=torch.float32, device=dev)

    def score_pairs(self):
        b = self.bufs
        L.locks_score(self.H, self.q, self.summ, self.bt, self.lens, b.workspace, scores=b.scores,
                      stream=self.stream)
        L.locks_cp_score_pairs(self.H, self.lens, self.MP, self.pairs, b.workspace, scores=b.scores,
                               stream=self.stream)
        return self.pairs

    def select_local(self, pairs_all):
        b = self.bufs
        L.locks_cp_select_local(self.H, self.lens, self.off, self.MP, self.budget, pairs_all, self.cand_pages,
                                self.cand_keys, self.cand_counts, b.workspace, scores=b.scores,
                                stream=self.stream)
        return self.cand_pages, self.cand_keys, self.cand_counts

    def merge_select(self, cand_pages_all, cand_keys_all, cand_counts_all):
        b = self.bufs
        L.locks_cp_merge_select(self.H, self.off, self.budget, self.shard, cand_pages_all, cand_keys_all,
                                cand_counts_all, b.selected, b.n_selected, stream=self.stream)

    def attend_partial(self):
        b = self.bufs
        L.locks_cp_sparse_decode_partial(self.H, self.q, self.k, self.v, self.bt, self.lens, b.selected,
                                         b.n_selected, self.budget, self.states, b.workspace,
                                         sm_scale=self.scale, stream=self.stream)
        return self.states

    def merge_attention(self, states_all):
        L.locks_cp_merge_attention(self.H, states_all, self.out, stream=self.stream)
        return self.out

    def selected_global(self):
        """This shard's selected pages as global indices, per (request, KV head)."""
        b = self.bufs
        sel = b.selected.cpu()
        cnt = b.n_selected.cpu()
        off = self.off.cpu()
        return {(i, h): (sel[i, h, :int(cnt[i, h])] + int(off[i])).tolist()
                for i in range(self.B) for h in range(self.H)}


def decode_step(shard, all_gather: Callable):
    """Run one shard's part of the decode step.  all_gather(t) must return
    every shard's t stacked on a new leading axis, in shard order, on t's
    device; every shard calls decode_step with the same sequence of gathers."""
    pairs_all = all_gather(shard.score_pairs())
    cands = shard.select_local(pairs_all)
    cands_all = [all_gather(x) for x in cands]
    shard.merge_select(*cands_all)
    states_all = all_gather(shard.attend_partial())
    return shard.merge_attention(states_all)


def host_all_gather(group=None) -> Callable:
    """An all_gather over a torch.distributed group through host memory (for
    a gloo group): the tensor is copied to the host, gathered, stacked and
    copied back to its device."""
    import torch.distributed as dist

    def gather(t):
        host = t.detach().cpu().contiguous()
        parts = [torch.empty_like(host) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, host, group=group)
        return torch.stack(parts).to(t.device)

    return gather


def shard_pages(block_table, seq_lens, n_shards: int, shard: int):
    """Contiguous split of every request's full pages over n_shards: shard r
    takes full pages [n r / R, n (r + 1) / R) of a request with n full pages,
    and the last shard also its open tail page.  Returns this shard's block
    table (its pages first, -1 after), token counts and first global page, as
    int32 tensors on the block table's device (index arithmetic only)."""
    bt = block_table.cpu()
    lens = seq_lens.cpu().tolist()
    B, MP = bt.shape
    rows, shard_lens, offsets = [], [], []
    for b, L_b in enumerate(lens):
        n, t = divmod(int(L_b), L.PAGE_SIZE)
        p0 = n * shard // n_shards
        p1 = n * (shard + 1) // n_shards
        pages = list(range(p0, p1))
        tokens = (p1 - p0) * L.PAGE_SIZE
        if shard == n_shards - 1 and t > 0:
            pages.append(n)
            tokens += t
        row = torch.full((MP,), -1, dtype=torch.int32)
        if pages:
            row[:len(pages)] = bt[b, pages]
        rows.append(row)
        shard_lens.append(tokens)
        offsets.append(p0)
    dev = block_table.device
    return (torch.stack(rows).to(dev), torch.tensor(shard_lens, dtype=torch.int32, device=dev),
            torch.tensor(offsets, dtype=torch.int32, device=dev))
