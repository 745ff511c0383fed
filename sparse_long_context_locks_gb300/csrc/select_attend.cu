// select_attend.cu -- fused LOCKS selection (a4, a5) and sparse paged decode
// attention (a6) for one (request, KV head) unit per thread-block cluster.
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2 ("Reconstruction and selection",
// "Group-shared selection (GQA)", and the implementation note that the whole
// decode step -- scoring, selection and sparse attention -- runs back to back
// without host round trips) and the abstract (attention reads the selected
// pages only).
//
// The cluster's 8 CTAs first run cluster_select (rank 0 ends up holding the
// physical blocks of the selected pages; the block-table entries were fetched
// into shared memory before the wait on the scoring pass).  Then the
// cluster's 64 warps attend the unit's selected pages plus the open tail
// page, item i to warp i mod 64; a warp reads the block of item i from rank
// 0's shared memory (distributed shared memory) and stages K and V with
// cp.async.bulk.tensor.  Warp states merge in shared
// memory, CTA states across the cluster through distributed shared memory, so
// no split partials, tickets or second launch are needed.  The kernel is
// launched as a programmatic dependent of the scoring pass: barrier set-up,
// tensor-map prefetch and the query fragments overlap the scorer's tail.

#include <cstdint>

#include "attn_tile.cuh"
#include "cluster_select.cuh"
#include "common.cuh"
#include "params.h"

namespace locks {

constexpr int kFusedWarps = kSelThreads / 32;                  // 8
constexpr int kFusedStages = 2;
constexpr int kFusedRing = kFusedWarps * kFusedStages * kStageBytes;   // 128 KB
// Warps 0 and 1 own a third stage (after the ring), so a unit of up to 130
// items (128 selected pages and the tail) is read in one round of copies.
constexpr int kFusedExtraWarps = 2;
constexpr int kFusedMaxStages = kFusedStages + 1;
constexpr int kFusedExtra = kFusedExtraWarps * kStageBytes;             // 16 KB


// Dynamic shared memory: [ring (keys and block ids of the slice during the
// selection)] [selected blocks (rank 0)] [barriers]
__host__ __device__ inline size_t fused_list_bytes(int budget) { return (4 * (size_t)budget + 15) / 16 * 16; }
size_t fused_smem_bytes(int max_pages, int budget) {
  (void)max_pages;   // the slice's keys and block ids live in the ring (host limits their size)
  return 1024 + kFusedRing + kFusedExtra + fused_list_bytes(budget) + kFusedWarps * kFusedMaxStages * 8;
}

__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads, 1)
    select_attend_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const FusedParams p) {
  extern __shared__ uint8_t fused_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fused_raw) + 1023) & ~uintptr_t(1023));
  const int slice_cap = (p.sel.max_pages + kSelCluster - 1) / kSelCluster;
  int* list = reinterpret_cast<int*>(smem + kFusedRing + kFusedExtra);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFusedRing + kFusedExtra + fused_list_bytes(p.sel.budget));
  __shared__ int stage_valid[kFusedWarps][kFusedMaxStages];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.y;
  const int b = unit / p.sel.H_kv, h = unit % p.sel.H_kv;
  uint64_t* mybar = bars + warp * kFusedMaxStages;
  const int nst = warp < kFusedExtraWarps ? kFusedMaxStages : kFusedStages;   // this warp's stages
  auto stage_ptr = [&](int st) -> uint8_t* {
    return st < kFusedStages ? smem + (warp * kFusedStages + st) * kStageBytes
                             : smem + kFusedRing + warp * kStageBytes;
  };

  // ---- prologue: independent of the scoring pass's results
  if (lane == 0) {
    for (int s = 0; s < nst; ++s) mbar_init(&mybar[s], 1);
    fence_mbar_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  uint32_t qb[8][2];
  attn_load_q(qb, p.q + ((int64_t)b * p.sel.H_kv * kGroup + (int64_t)h * kGroup) * kHeadDim, lane);
  // block ids of this CTA's slice of the page range (the same split as the
  // selection's), and of the tail page: inputs, so fetched before the wait
  int* bt_slice = reinterpret_cast<int*>(smem) + slice_cap;   // after the keys, inside the ring
  __shared__ int tail_blk;
  {
    const int L = p.sel.seq_lens[b];
    const bool okL = L >= 0 && (L + kPage - 1) / kPage <= p.sel.max_pages;
    const int n = okL ? L / kPage : 0;
    const int j0 = (int)(((long long)n * rank) / kSelCluster);
    const int j1 = (int)(((long long)n * (rank + 1)) / kSelCluster);
    const int32_t* bt_row = p.block_table + (int64_t)b * p.sel.max_pages;
    for (int i = threadIdx.x; i < j1 - j0; i += blockDim.x) bt_slice[i] = bt_row[j0 + i];
    if (threadIdx.x == 0) tail_blk = (okL && L % kPage) ? bt_row[n] : -1;
  }
  __syncthreads();

  griddep_wait();   // the scoring pass's scores are now visible

  // ---- selection (the ring holds this CTA's keys and block ids meanwhile)
  SelScratch sc;
  sc.keys_s = reinterpret_cast<uint32_t*>(smem);
  sc.bt_slice = bt_slice;
  sc.out_blk = list;
  sc.stage = nullptr;
  const ClusterSel cs = cluster_select<kSelCluster, false>(p.sel, sc);
  fence_proxy_async_smem();   // generic writes to the ring before the tensor copies reuse it
  __syncthreads();

  // ---- sparse attention over the selected pages and the tail page
  const int items = cs.kk + (cs.tail > 0 ? 1 : 0);
  const int gw = rank * kFusedWarps + warp;
  constexpr int kWarpsPerUnit = kSelCluster * kFusedWarps;   // 64
  const int my_count = items > gw ? (items - gw + kWarpsPerUnit - 1) / kWarpsPerUnit : 0;
  // lane k resolves this warp's item k (host limits a unit to 32 items per warp)
  int64_t blk = -1;
  int valid = 0;
  if (lane < my_count) {
    const int i = gw + lane * kWarpsPerUnit;
    if (i < cs.kk) {
      blk = *cluster.map_shared_rank(&sc.out_blk[i], 0);   // physical block, from rank 0
      valid = kPage;
    } else {
      blk = tail_blk;
      valid = cs.tail;
    }
    if (blk < 0 || blk >= p.num_blocks) {
      flag_status(p.sel.status, LOCKS_FLAG_BAD_BLOCK);
      blk = -1;
      valid = 0;
    }
  }
  if (lane < min(nst, my_count)) {
    stage_valid[warp][lane] = valid;
    attn_issue_page(&tmk, &tmv, stage_ptr(lane), &mybar[lane], blk, p.sel.H_kv, h);
  }
  __syncwarp();

  PageAttnState st;
  attn_init(st);
  bool ok = true;
  for (int k = 0; k < my_count; ++k) {
    const int stage = k % nst;
    if (ok) ok = mbar_wait(&mybar[stage], (k / nst) & 1, p.sel.status);
    const int v = stage_valid[warp][stage];
    uint8_t* sp = stage_ptr(stage);
    if (ok && v > 0) attn_page(st, smem_u32(sp), sp + kTileBytes, v, qb, p.scale_log2, lane);
    fence_proxy_async_smem();
    __syncwarp();
    const int kn = k + nst;
    if (kn < my_count) {
      const int64_t nb = __shfl_sync(0xffffffffu, blk, kn);
      const int nv = __shfl_sync(0xffffffffu, valid, kn);
      if (lane == 0) {
        stage_valid[warp][stage] = nv;
        attn_issue_page(&tmk, &tmv, sp, &mybar[stage], nb, p.sel.H_kv, h);
      }
    }
    __syncwarp();
  }
  attn_finish(st);

  // ---- merge the CTA's 8 warps in shared memory
  __syncthreads();   // ring no longer in use
  float* wO = reinterpret_cast<float*>(smem);                        // [warp][G][128]
  float* wM = wO + kFusedWarps * kGroup * kHeadDim;                  // [warp][G]
  float* wL = wM + kFusedWarps * kGroup;                             // [warp][G]
  float* pub = reinterpret_cast<float*>(smem + 32768);               // [G][2 + 128] published
  attn_store_warp(st, wO + warp * kGroup * kHeadDim, wM + warp * kGroup, wL + warp * kGroup, lane);
  __syncthreads();
  // warp 0, lane 4w + g: the factor exp2(m_{w,g} - M_g) of warp w's state for
  // head g, M_g and the merged sum l_g; then every thread forms two of the
  // CTA's G x 128 outputs from the 8 warps' states
  __shared__ float fw[kFusedWarps][kGroup];
  if (warp == 0) {
    const int w = lane >> 2, g = lane & 3;
    const float m = wM[w * kGroup + g];
    float M = m;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = M == -INFINITY ? 0.f : fast_exp2(m - M);
    fw[w][g] = f;
    float l = wL[w * kGroup + g] * f;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (w == 0) {
      pub[g * (2 + kHeadDim)] = M;
      pub[g * (2 + kHeadDim) + 1] = l;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kGroup * kHeadDim; i += blockDim.x) {
    const int g = i / kHeadDim, d = i % kHeadDim;
    float Os = 0.f;
#pragma unroll
    for (int w = 0; w < kFusedWarps; ++w) Os += wO[(w * kGroup + g) * kHeadDim + d] * fw[w][g];
    pub[g * (2 + kHeadDim) + 2 + d] = Os;
  }
  cluster.sync();   // every CTA's state is published

  // ---- merge the cluster: CTA `rank` finishes output dims [16 rank, 16 rank + 16)
  if (threadIdx.x < kGroup * 16) {
    const int g = threadIdx.x >> 4, d = 16 * rank + (threadIdx.x & 15);
    // every remote load is issued before any of them is used
    float mr[kSelCluster], lr[kSelCluster], orr[kSelCluster], M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) {
      const float* rp = cluster.map_shared_rank(&pub[g * (2 + kHeadDim)], r);
      mr[r] = rp[0];
      lr[r] = rp[1];
      orr[r] = rp[2 + d];
    }
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) M = fmaxf(M, mr[r]);
    float Ls = 0.f, Os = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int r = 0; r < kSelCluster; ++r) {
        const float f = fast_exp2(mr[r] - M);
        Ls += lr[r] * f;
        Os += orr[r] * f;
      }
    }
    p.out[((int64_t)b * p.sel.H_kv * kGroup + (int64_t)h * kGroup + g) * kHeadDim + d] = Ls > 0.f ? Os / Ls : 0.f;
  }
  cluster.sync();   // keep shared memory alive until every CTA has read it
}

cudaError_t launch_select_attend(const CUtensorMap& tmk, const CUtensorMap& tmv, const FusedParams& p,
                                 int units, cudaStream_t stream) {
  const size_t dyn = fused_smem_bytes(p.sel.max_pages, p.sel.budget);
  static DynSmemAttr smem_attr;
  const cudaError_t ea = ensure_dyn_smem(reinterpret_cast<const void*>(select_attend_kernel), dyn, smem_attr);
  if (ea != cudaSuccess) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSelCluster, units, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, select_attend_kernel, tmk, tmv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace locks
