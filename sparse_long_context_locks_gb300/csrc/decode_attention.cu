// decode_attention.cu -- split-K paged decode attention for LOCKS (a6) and the
// dense comparator (a7).
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", abstract and technical summary §2: after selection only the top
// pages are attended, with all query heads of a GQA group attending the same
// pages (so one K/V read serves the whole group).  The still-open tail page
// (no summary yet) is always attended.  The dense comparator is the same
// kernel over every cached page.
//
// Grid: (split, request x KV head).  Each CTA owns a contiguous slice of the
// unit's item list (selected pages + tail, or all pages + tail); each of its 4
// warps runs its own 3-stage ring: lane 0 issues four 2 KB cp.async.bulk.tensor
// loads per page (K and V, 64-column halves, 128-byte swizzle) onto an
// mbarrier, the warp waits, then
//   S = K q^T   (mma.sync m16n8k16 bf16: 16 tokens x 8 columns (4 heads, padded))
//   online softmax per head (exp2, running max / sum)
//   O^T += V^T P (ldmatrix.trans on the swizzled V tile; P transposed in
//                 registers with movmatrix)
// Warps merge through shared memory; splits merge through per-split partials
// in the workspace, combined by the last CTA of each unit (atomic ticket, no
// spinning).

#include <cstdint>

#include <cooperative_groups.h>

#include "attn_tile.cuh"
#include "common.cuh"
#include "params.h"

namespace locks {

namespace cg = cooperative_groups;


constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnStages = 3;
constexpr int kAttnRing = kAttnWarps * kAttnStages * kStageBytes;
constexpr int kAttnSmem = kAttnRing + 1024 /*align*/ + 256 /*barriers*/;
constexpr int kPartStride = 2 + kHeadDim;

__device__ __forceinline__ void unit_items(const AttnParams& p, int b, int h, int& n, int& t,
                                           int& nsel, int& items) {
  const int L = p.seq_lens[b];
  if (L < 0 || (L + kPage - 1) / kPage > p.max_pages) {
    n = t = nsel = items = 0;
    return;
  }
  n = L / kPage;
  t = L % kPage;
  if (p.dense) {
    nsel = n;
  } else {
    nsel = p.n_selected[b * p.H_kv + h];
    const int cap = min(p.budget, n);
    if (nsel < 0 || nsel > cap) nsel = max(0, min(nsel, cap));
  }
  items = nsel + (t > 0 ? 1 : 0);
}

// Entry i of the unit's selection list, read before the list's length is
// known (entries past the length are never used); -1 past the budget.
__device__ __forceinline__ int sel_entry(const AttnParams& p, int b, int h, int i) {
  return (!p.dense && i >= 0 && i < p.budget) ? p.selected[((int64_t)b * p.H_kv + h) * p.budget + i] : -1;
}

// Resolve item i of the unit: physical block (or -1 to skip) and valid tokens.
// sel_i: the unit's selection entry i (sel_entry), for i < nsel.
__device__ __forceinline__ void item_block(const AttnParams& p, int b, int h, int i, int n, int t,
                                           int nsel, int sel_i, int64_t& blk, int& valid) {
  int page;
  if (i < nsel) {
    page = p.dense ? i : sel_i;
    valid = kPage;
    if (page < 0 || page >= n) {
      flag_status(p.status, LOCKS_FLAG_BAD_SELECT);
      blk = -1;
      valid = 0;
      return;
    }
  } else {
    page = n;
    valid = t;
  }
  blk = p.block_table[(int64_t)b * p.max_pages + page];
  if (blk < 0 || blk >= p.num_blocks) {
    flag_status(p.status, LOCKS_FLAG_BAD_BLOCK);
    blk = -1;
    valid = 0;
  }
}

// kClusterMerge: the unit's p.splits CTAs (at most 8) form a thread-block
// cluster and merge their states through distributed shared memory, with no
// partials in the workspace, fence or ticket; otherwise the last CTA of the
// unit to finish merges the partials it finds in the workspace.
template <bool kClusterMerge>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kAttnRing);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.y, split = blockIdx.x;
  const int b = unit / p.H_kv, h = unit % p.H_kv;

  uint64_t* mybar = bars + warp * kAttnStages;
  const uint32_t ring = smem_u32(smem) + warp * kAttnStages * kStageBytes;
  uint8_t* ring_ptr = smem + warp * kAttnStages * kStageBytes;
  if (lane == 0) {
    for (int s = 0; s < kAttnStages; ++s) mbar_init(&mybar[s], 1);
    fence_mbar_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  __syncwarp();
  // The request's length and block-table row are inputs, not the selection's
  // results: the row's lines this split may touch are pulled into L2 before
  // the wait, so the block lookup after it is an L2 hit.  (A sparse split's
  // pages are anywhere in the row; each of the unit's CTAs prefetches its
  // share of the row's lines.)
  {
    const int L0 = p.seq_lens[b];
    if (L0 > 0 && (L0 + kPage - 1) / kPage <= p.max_pages) {
      const int npg = (L0 + kPage - 1) / kPage;
      const int32_t* row = p.block_table + (int64_t)b * p.max_pages;
      const int lines = (npg + 31) / 32;   // 32 entries a line
      const int per = (lines + p.splits - 1) / p.splits;
      const int l0 = p.dense ? (int)((int64_t)split * p.items_per_split / 32) : split * per;
      const int l1 = p.dense ? min(lines, (int)(((int64_t)(split + 1) * p.items_per_split + 31) / 32))
                             : min(lines, l0 + per);
      for (int l = l0 + threadIdx.x; l < l1; l += blockDim.x) prefetch_l2(row + 32 * l);
    }
  }
  // launched as a programmatic dependent of the selection: its lists are
  // visible from here on
  griddep_wait();

  // The first two windows' selection entries are requested together with the
  // request's length and the list's length: one dependent round trip fewer
  // before the first block lookup.  (A split's items start at
  // split * items_per_split whatever the unit's item count.)
  const int spec0 = split * p.items_per_split + warp + lane * kAttnWarps;
  const int sel0 = sel_entry(p, b, h, spec0), sel1 = sel_entry(p, b, h, spec0 + 32 * kAttnWarps);
  int n, tail, nsel, items;
  unit_items(p, b, h, n, tail, nsel, items);
  const int r0 = min(items, split * p.items_per_split);
  const int r1 = min(items, r0 + p.items_per_split);
  // this warp's items: r0 + warp, r0 + warp + 4, ...
  const int my_first = r0 + warp;
  const int my_count = my_first < r1 ? (r1 - my_first + kAttnWarps - 1) / kAttnWarps : 0;

  // Item metadata windows: lane l of `cur` describes issue index base + l,
  // `nxt` the 32 after it (loaded one window ahead so refills never wait).
  __shared__ int stage_valid[kAttnWarps][kAttnStages];
  int64_t cur_blk = -1, nxt_blk = -1;
  int cur_valid = 0, nxt_valid = 0;
  if (lane < my_count)
    item_block(p, b, h, my_first + lane * kAttnWarps, n, tail, nsel, sel0, cur_blk, cur_valid);
  if (32 + lane < my_count)
    item_block(p, b, h, my_first + (32 + lane) * kAttnWarps, n, tail, nsel, sel1, nxt_blk, nxt_valid);

  auto issue = [&](int64_t blk, int stage) {
    attn_issue_page(&tmk, &tmv, ring_ptr + stage * kStageBytes, &mybar[stage], blk, p.H_kv, h);
  };

  // prologue: lane k issues item k into stage k
  if (lane < min(kAttnStages, my_count)) {
    stage_valid[warp][lane] = cur_valid;
    issue(cur_blk, lane);
  }

  uint32_t qb[8][2];
  attn_load_q(qb, p.q + ((int64_t)b * p.H_kv * kGroup + (int64_t)h * kGroup) * kHeadDim, lane);
  __syncwarp();

  PageAttnState st;
  attn_init(st);
  bool ok = true;

  for (int k = 0; k < my_count; ++k) {
    const int stage = k % kAttnStages;
    if (ok) ok = mbar_wait(&mybar[stage], (k / kAttnStages) & 1, p.status);
    const int valid = stage_valid[warp][stage];
    if (ok && valid > 0)
      attn_page(st, ring + stage * kStageBytes, ring_ptr + stage * kStageBytes + kTileBytes, valid, qb,
                p.scale_log2, lane);
    // order this warp's generic smem accesses before the next async write
    fence_proxy_async_smem();
    __syncwarp();
    // refill this stage with item k + S
    const int kn = k + kAttnStages;
    if (kn < my_count) {
      if ((kn & 31) == 0) {
        cur_blk = nxt_blk;
        cur_valid = nxt_valid;
        nxt_blk = -1;
        nxt_valid = 0;
        if (kn + 32 + lane < my_count) {
          const int i = my_first + (kn + 32 + lane) * kAttnWarps;
          item_block(p, b, h, i, n, tail, nsel, sel_entry(p, b, h, i), nxt_blk, nxt_valid);
        }
      }
      const int64_t blk = __shfl_sync(0xffffffffu, cur_blk, kn & 31);
      const int v = __shfl_sync(0xffffffffu, cur_valid, kn & 31);
      if (lane == 0) {
        stage_valid[warp][stage] = v;
        issue(blk, stage);
      }
    }
    __syncwarp();
  }

  attn_finish(st);

  // ---- merge the 4 warps through shared memory (ring no longer in use)
  __syncthreads();
  float* wO = reinterpret_cast<float*>(smem);                       // [warp][G][128]
  float* wM = wO + kAttnWarps * kGroup * kHeadDim;                  // [warp][G]
  float* wL = wM + kAttnWarps * kGroup;                             // [warp][G]
  attn_store_warp(st, wO + warp * kGroup * kHeadDim, wM + warp * kGroup, wL + warp * kGroup, lane);
  __syncthreads();

  const int d = threadIdx.x;   // 128 threads = 128 dims
  float Mg[kGroup], Lg[kGroup], Og[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wM[w * kGroup + g]);
    float Ls = 0.f, Os = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = fast_exp2(wM[w * kGroup + g] - M);
        Ls += wL[w * kGroup + g] * f;
        Os += wO[(w * kGroup + g) * kHeadDim + d] * f;
      }
    }
    Mg[g] = M;
    Lg[g] = Ls;
    Og[g] = Os;
  }

  float* orow = p.out + ((int64_t)b * p.H_kv * kGroup + (int64_t)h * kGroup) * kHeadDim;
  // context-parallel shards export the unnormalised state instead
  float* srow = p.state_out ? p.state_out + ((int64_t)b * p.H_kv * kGroup + (int64_t)h * kGroup) * kPartStride
                            : nullptr;
  if (p.splits == 1) {
    if (srow) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        srow[g * kPartStride + 2 + d] = Og[g];
        if (d == 0) {
          srow[g * kPartStride] = Mg[g];
          srow[g * kPartStride + 1] = Lg[g];
        }
      }
      return;
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) orow[g * kHeadDim + d] = Lg[g] > 0.f ? Og[g] / Lg[g] : 0.f;
    return;
  }

  if constexpr (kClusterMerge) {
    // publish this CTA's state; CTA r then finishes dims r, r + S, r + 2S, ...
    cg::cluster_group cluster = cg::this_cluster();
    float* pub = reinterpret_cast<float*>(smem + 12288);   // [G][2 + 128], past the warp states
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      pub[g * kPartStride + 2 + d] = Og[g];
      if (d == 0) {
        pub[g * kPartStride] = Mg[g];
        pub[g * kPartStride + 1] = Lg[g];
      }
    }
    cluster.sync();   // every split's state is published
    const int S = p.splits;
    const int per = (kHeadDim + S - 1) / S;
    for (int idx = threadIdx.x; idx < kGroup * per; idx += blockDim.x) {
      const int g = idx / per, dd = split + S * (idx % per);
      if (dd < kHeadDim) {
        float mr[8], lr[8], orr[8], M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 8; ++r) {   // every remote load first
          if (r < S) {
            const float* rp = cluster.map_shared_rank(&pub[g * kPartStride], r);
            mr[r] = rp[0];
            lr[r] = rp[1];
            orr[r] = rp[2 + dd];
          }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < S) M = fmaxf(M, mr[r]);
        float Ls = 0.f, Os = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            if (r < S) {
              const float f = fast_exp2(mr[r] - M);
              Ls += lr[r] * f;
              Os += orr[r] * f;
            }
          }
        }
        if (srow) {
          srow[g * kPartStride + 2 + dd] = Os;
          if (dd == split) {
            srow[g * kPartStride] = M;
            srow[g * kPartStride + 1] = Ls;
          }
        } else {
          orow[g * kHeadDim + dd] = Ls > 0.f ? Os / Ls : 0.f;
        }
      }
    }
    cluster.sync();   // keep shared memory alive until every CTA has read it
    return;
  }

  float* mypart = p.part + ((int64_t)unit * p.splits + split) * kGroup * kPartStride;
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    mypart[g * kPartStride + 2 + d] = Og[g];
    if (d == 0) {
      mypart[g * kPartStride] = Mg[g];
      mypart[g * kPartStride + 1] = Lg[g];
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ uint32_t sh_last;
  if (threadIdx.x == 0) {
    const uint32_t ticket = atomicAdd(&p.tickets[unit], 1u);
    sh_last = (ticket == (uint32_t)p.splits - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  // last CTA of the unit: combine all splits.  Max and weights are computed
  // cooperatively (split sp -> thread sp mod 128), then every thread (one
  // output dim) sums the splits' partial outputs with many loads in flight.
  const float* up = p.part + (int64_t)unit * p.splits * kGroup * kPartStride;
  const int S = p.splits;
  float* red = reinterpret_cast<float*>(smem + 12288);   // [warp][G] reductions
  float* wsm = reinterpret_cast<float*>(smem + 16384);   // [S][G] split weights
  float mloc[kGroup], lloc[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    mloc[g] = -INFINITY;
    lloc[g] = 0.f;
  }
  for (int sp = threadIdx.x; sp < S; sp += blockDim.x)
#pragma unroll
    for (int g = 0; g < kGroup; ++g) mloc[g] = fmaxf(mloc[g], __ldcg(up + (sp * kGroup + g) * kPartStride));
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc[g] = fmaxf(mloc[g], __shfl_xor_sync(0xffffffffu, mloc[g], o));
    if (lane == 0) red[warp * kGroup + g] = mloc[g];
  }
  __syncthreads();
  float Mall[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    Mall[g] = red[g];
    for (int w = 1; w < kAttnWarps; ++w) Mall[g] = fmaxf(Mall[g], red[w * kGroup + g]);
  }
  __syncthreads();
  for (int sp = threadIdx.x; sp < S; sp += blockDim.x) {
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const float* q = up + (sp * kGroup + g) * kPartStride;
      const float f = Mall[g] == -INFINITY ? 0.f : fast_exp2(__ldcg(q) - Mall[g]);
      wsm[sp * kGroup + g] = f;
      lloc[g] += __ldcg(q + 1) * f;
    }
  }
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lloc[g] += __shfl_xor_sync(0xffffffffu, lloc[g], o);
    if (lane == 0) red[warp * kGroup + g] = lloc[g];
  }
  __syncthreads();
  float Lall[kGroup], acc_o[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    Lall[g] = 0.f;
    for (int w = 0; w < kAttnWarps; ++w) Lall[g] += red[w * kGroup + g];
    acc_o[g] = 0.f;
  }
#pragma unroll 4
  for (int sp = 0; sp < S; ++sp) {
    const float4 wv = *reinterpret_cast<const float4*>(wsm + sp * kGroup);
    const float* q = up + sp * kGroup * kPartStride + 2 + d;
    acc_o[0] += wv.x * __ldcg(q);
    acc_o[1] += wv.y * __ldcg(q + kPartStride);
    acc_o[2] += wv.z * __ldcg(q + 2 * kPartStride);
    acc_o[3] += wv.w * __ldcg(q + 3 * kPartStride);
  }
  if (srow) {
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      srow[g * kPartStride + 2 + d] = acc_o[g];
      if (d == 0) {
        srow[g * kPartStride] = Mall[g];
        srow[g * kPartStride + 1] = Lall[g];
      }
    }
  } else {
#pragma unroll
    for (int g = 0; g < kGroup; ++g) orow[g * kHeadDim + d] = Lall[g] > 0.f ? acc_o[g] / Lall[g] : 0.f;
  }
  if (threadIdx.x == 0) p.tickets[unit] = 0;   // ready for the next call
}

template <bool kClusterMerge>
cudaError_t launch_attn_t(const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p,
                          cudaStream_t stream) {
  static DynSmemAttr smem_attr;
  const cudaError_t e =
      ensure_dyn_smem(reinterpret_cast<const void*>(attn_kernel<kClusterMerge>), kAttnSmem, smem_attr);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.batch * p.H_kv, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kClusterMerge ? p.splits : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kClusterMerge ? 2 : 1;
  const cudaError_t el = cudaLaunchKernelEx(&cfg, attn_kernel<kClusterMerge>, tmk, tmv, p);
  if (el != cudaSuccess) return el;
  return cudaGetLastError();
}

cudaError_t launch_attn(const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p,
                        cudaStream_t stream) {
  // 2..8 splits a unit: a cluster per unit (portable size)
  if (p.splits >= 2 && p.splits <= 8) return launch_attn_t<true>(tmk, tmv, p, stream);
  return launch_attn_t<false>(tmk, tmv, p, stream);
}

}  // namespace locks
