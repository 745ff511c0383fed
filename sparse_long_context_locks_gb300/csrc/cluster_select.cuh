// cluster_select.cuh -- LOCKS group-shared top-k selection (a4, a5) inside a
// thread-block cluster, shared by the selection kernel and the fused
// select + sparse-attention kernel.
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2, "Reconstruction and selection" and
// "Group-shared selection (GQA)": per-head page-mass shares exp(s_j - Z_g),
// Z_g = log sum_j exp(s_j,g) over the full pages, averaged over the group's
// query heads into one table; the k largest entries (lower page index on
// ties) are attended.
//
// One cluster of C CTAs per (request, KV head) (C a power of two, at most 16);
// CTA r owns pages [n r / C, n (r + 1) / C).
//   1. Z_g: each CTA folds its slice's scores into a (max, sum) pair per head
//      and publishes it in shared memory; after a cluster barrier every CTA
//      combines the C pairs, read through distributed shared memory.
//   2. Keys: the fp32 bits of the table entries (non-negative floats order
//      like unsigned ints).
//   3. Exact cluster-wide select.  Level 0: every CTA histograms its keys by
//      bits 30-20 (exponent and 3 mantissa bits) and publishes its highest
//      occupied bin; after a cluster barrier every CTA walks the C
//      histograms top-down from the highest bin, 32 bins (one remote count
//      per thread) at a time, to the bin holding the k-th largest key, and
//      takes from the per-CTA counts above it its own number of selected keys
//      and the number selected by lower-ranked CTAs (its output offset).  The
//      boundary bin's members (typically tens to a few hundred) then go to
//      rank 0 as (key, page), and every CTA ranks all of them exactly (key
//      descending, lower page first), a thread per member.  When the bin holds more
//      than kMemberCap keys, levels over bits 19-10 and 9-0 follow instead,
//      each a full histogram exchange; after the last one the boundary keys
//      are equal and the lowest pages go first.
//   4. Each CTA writes its selected pages, ascending, from its offset on, and
//      their physical blocks into rank 0's shared memory; a final cluster
//      barrier publishes that list.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "params.h"

namespace locks {

namespace cg = cooperative_groups;

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelMaxChunks = kFusedMaxKeysPerCta / 32;   // 32-key chunks of one slice
constexpr int kMemberCap = 512;   // boundary-bin members ranked pairwise after level 0

// Merge of two (max, sum) log-sum-exp partials (log2 units).
__device__ __forceinline__ void lse2_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * fast_exp2(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * fast_exp2(m2 - m);
  }
}

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_buf, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_buf[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  total = warp_buf[nw - 1];
  const int before = (warp > 0 ? warp_buf[warp - 1] : 0) + x - v;
  __syncthreads();
  return before;
}

// Block-wide sums of two ints (every thread gets both); ends with a barrier.
__device__ __forceinline__ void block_sum2(int& a, int& b, int* warp_buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (lane == 0) {
    warp_buf[2 * warp] = a;
    warp_buf[2 * warp + 1] = b;
  }
  __syncthreads();
  a = 0;
  b = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    a += warp_buf[2 * w];
    b += warp_buf[2 * w + 1];
  }
  __syncthreads();
}

// Radix levels over the 31 value bits of a non-negative float's pattern.
__device__ __forceinline__ int lvl_shift(int lvl) { return lvl == 0 ? 20 : (lvl == 1 ? 10 : 0); }
__device__ __forceinline__ int lvl_bits(int lvl) { return lvl == 0 ? 11 : 10; }
__device__ __forceinline__ uint32_t lvl_digit(uint32_t key, int lvl) {
  return (key >> lvl_shift(lvl)) & ((1u << lvl_bits(lvl)) - 1u);
}

// Selection key of one page: the mean over the group's heads of the page's
// mass share exp(s_g - Z_g), computed in log2 units (z = log2 Z_g), as fp32
// bits (non-negative floats order like unsigned ints).  A non-finite or
// negative mean becomes 0.  Every selection path takes its keys from here, so
// keys computed on different GPUs for different pages of one request compare
// exactly as they would on one.
__device__ __forceinline__ uint32_t group_key(const float4& v, float z0, float z1, float z2, float z3) {
  float avg = 0.25f * (fast_exp2(v.x * kLog2e - z0) + fast_exp2(v.y * kLog2e - z1) +
                       fast_exp2(v.z * kLog2e - z2) + fast_exp2(v.w * kLog2e - z3));
  if (!(avg >= 0.f) || isinf(avg)) avg = 0.f;
  return __float_as_uint(avg);
}

// log2 Z_g of unit `unit` and head g from the per-shard (max, sum) pairs of
// the unit's pages held by `n_shards` GPUs: pairs[(shard * units + unit) * 4 + g]
// = (max over the shard's pages of s * log2(e), sum of 2^(s log2(e) - max)).
__device__ __forceinline__ float z_from_shards(const float2* pairs, int n_shards, int units, int unit, int g) {
  float mx = -INFINITY, sv = 0.f;
  for (int r = 0; r < n_shards; ++r) {
    const float2 pr = pairs[((int64_t)r * units + unit) * kGroup + g];
    lse2_merge(mx, sv, pr.x, pr.y);
  }
  return mx + fast_log2(sv);
}

// Result of cluster_select for the calling CTA.
struct ClusterSel {
  int n;        // full pages of the request (0 when its length is invalid)
  int tail;     // tokens of the open tail page
  int kk;       // pages selected for the unit
};

// Shared-memory scratch handed to cluster_select:
//   keys_s   ceil(max_pages / C) <= kFusedMaxKeysPerCta words: this CTA's keys;
//   bt_slice optional block ids of this CTA's pages (nullptr: none);
//   out_blk  budget words, used on rank 0: the selected pages' physical
//            blocks (bt_slice given) or page indices, ascending by page;
//   stage    room for this CTA's slice of scores (used when kStaged; else
//            both passes over the scores read them from global memory).
struct SelScratch {
  uint32_t* keys_s;
  const int* bt_slice;
  int* out_blk;
  float4* stage;
};

// Selects the pages of unit (b, h) = blockIdx.y.  Every thread of every CTA
// of the cluster must call it.  Writes `selected` and `n_selected`; ends with
// a cluster barrier after which rank 0's out_blk[0, kk) may be read through
// distributed shared memory.  kExtZ: Z_g is not formed from this unit's
// scores but taken from p.zpairs (per-shard (max, sum) pairs of a request
// whose pages several GPUs hold); the scores and pages are then this GPU's
// shard of the request.
template <int C, bool kStaged, bool kExtZ = false>
static __device__ ClusterSel cluster_select(const SelectParams& p, const SelScratch& sc) {
  __shared__ __align__(16) int hist0[1 << 11];
  __shared__ __align__(16) int hist1[1 << 10];
  __shared__ __align__(16) int hist2[1 << 10];
  __shared__ int s_hmax;                       // this CTA's highest occupied level-0 bin
  __shared__ __align__(8) float lse_pub[kGroup][2];   // this CTA's (max, sum) per head, log2 units
  __shared__ float red_m[kSelWarps][kGroup], red_s[kSelWarps][kGroup];
  __shared__ float zl[kGroup];
  __shared__ int scan_buf[32];
  __shared__ int bnd_cnt[C];         // per-CTA count in the boundary bin
  __shared__ int s_bin, s_above, s_cutoff, s_cnt;
  __shared__ int chunk_base[kSelMaxChunks];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int unit = blockIdx.y;              // (request, KV head)
  const int b = unit / p.H_kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = p.seq_lens[b];
  int32_t* sel = p.selected + (int64_t)unit * p.budget;
  ClusterSel res{0, 0, 0};
  // every CTA of a cluster takes the same branches below (same unit)
  if (L < 0 || (L + kPage - 1) / kPage > p.max_pages) {
    if (tid == 0 && rank == 0) {
      p.n_selected[unit] = 0;
      if (unit % p.H_kv == 0) flag_status(p.status, LOCKS_FLAG_BAD_SEQLEN);
    }
    cluster.sync();
    return res;
  }
  const int n = L / kPage;
  res.n = n;
  res.tail = L % kPage;
  const int kk = min(p.budget, n);
  res.kk = kk;
  const int j0 = (int)(((long long)n * rank) / C);
  const int j1 = (int)(((long long)n * (rank + 1)) / C);
  const int len = j1 - j0;
  if (n <= p.budget || kk == 0) {   // every full page is selected (or none is)
    if (kk > 0) {
      for (int i = tid; i < len; i += blockDim.x) {
        sel[j0 + i] = j0 + i;
        // rank 0 holds the list: fill its out_blk through distributed shared memory
        *cluster.map_shared_rank(&sc.out_blk[j0 + i], 0) = sc.bt_slice ? sc.bt_slice[i] : j0 + i;
      }
    }
    if (tid == 0 && rank == 0) p.n_selected[unit] = kk;
    cluster.sync();
    return res;
  }

  // ---- 1. this slice's (max, sum) of the scores per head, log2 units
  const float4* srow = reinterpret_cast<const float4*>(p.scores + (int64_t)unit * p.max_pages * kGroup) + j0;
  // Staged: every thread copies the scores it will read (its own indices in
  // both passes) with asynchronous copies, so the whole slice is in flight at
  // once instead of a few loads per thread.
  const float4* src = kStaged ? sc.stage : srow;
  if constexpr (kStaged) {
    for (int i = tid; i < len; i += blockDim.x) cp_async16(&sc.stage[i], &srow[i]);
  }
  constexpr int kPre = 4;   // scores held in registers for both passes
  float4 pre[kPre];
  if constexpr (!kStaged) {
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int i = tid + r * kSelThreads;
      pre[r] = i < len ? srow[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  for (int i = tid; i < (1 << 10); i += blockDim.x) {
    hist1[i] = 0;
    hist2[i] = 0;
  }
  for (int i = tid; i < (1 << 11); i += blockDim.x) hist0[i] = 0;
  if (tid == 0) s_hmax = -1;
  if constexpr (kStaged) {
    cp_async_wait_all();
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int i = tid + r * kSelThreads;
      pre[r] = i < len ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if constexpr (kExtZ) {
    if (tid < kGroup) zl[tid] = z_from_shards(reinterpret_cast<const float2*>(p.zpairs), p.z_shards,
                                              p.batch * p.H_kv, unit, tid);
    __syncthreads();   // zl and the cleared histograms are visible
  } else {
    float m[kGroup] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    float s[kGroup] = {0.f, 0.f, 0.f, 0.f};
    // fold kPre scores (an absent one is -inf) into (m, s): the batch's max
    // per head first, then one rescale of s and kPre independent terms
    auto fold_batch = [&](const float4 (&v)[kPre], int cnt) {
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        float x[kPre];
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
          const float c = g == 0 ? v[k].x : g == 1 ? v[k].y : g == 2 ? v[k].z : v[k].w;
          x[k] = k < cnt ? c * kLog2e : -INFINITY;
        }
        float mn = m[g];
#pragma unroll
        for (int k = 0; k < kPre; ++k) mn = fmaxf(mn, x[k]);
        if (mn != -INFINITY) {
          float acc = s[g] * fast_exp2(m[g] - mn);
#pragma unroll
          for (int k = 0; k < kPre; ++k) acc += fast_exp2(x[k] - mn);
          s[g] = acc;
          m[g] = mn;
        }
      }
    };
    fold_batch(pre, min(kPre, max(0, (len - tid + kSelThreads - 1) / kSelThreads)));
    for (int i0 = tid + kPre * kSelThreads; i0 < len; i0 += kPre * kSelThreads) {
      float4 v[kPre];
#pragma unroll
      for (int k = 0; k < kPre; ++k) {
        const int i = i0 + k * kSelThreads;
        v[k] = i < len ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      fold_batch(v, min(kPre, (len - i0 + kSelThreads - 1) / kSelThreads));
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      float mx = m[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sv = m[g] == -INFINITY ? 0.f : s[g] * fast_exp2(m[g] - mx);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
      if (lane == 0) {
        red_m[warp][g] = mx;
        red_s[warp][g] = sv;
      }
    }
    __syncthreads();
    if (tid < kGroup) {
      float mx = -INFINITY, sv = 0.f;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) lse2_merge(mx, sv, red_m[w][tid], red_s[w][tid]);
      lse_pub[tid][0] = mx;
      lse_pub[tid][1] = sv;
    }
    cluster.sync();   // every CTA's (max, sum) pairs and cleared histograms are visible
    if (tid < kGroup) {
      float2 pr[C];   // issue every remote load before merging
#pragma unroll
      for (int r = 0; r < C; ++r)
        pr[r] = *reinterpret_cast<const float2*>(cluster.map_shared_rank(&lse_pub[tid][0], r));
      float mx = -INFINITY, sv = 0.f;
#pragma unroll
      for (int r = 0; r < C; ++r) lse2_merge(mx, sv, pr[r].x, pr[r].y);
      zl[tid] = mx + fast_log2(sv);   // log2 Z_g
    }
    __syncthreads();
  }

  // ---- 2. keys of this slice: mean over heads of exp(s - Z_g), as fp32 bits
  {
    const float z0 = zl[0], z1 = zl[1], z2 = zl[2], z3 = zl[3];
    uint32_t kmax = 0u;
    bool any = false;
    auto make_key = [&](const float4& v, int i) {
      const uint32_t key = group_key(v, z0, z1, z2, z3);
      sc.keys_s[i] = key;
      atomicAdd(&hist0[lvl_digit(key, 0)], 1);
      kmax = max(kmax, key);
      any = true;
    };
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int i = tid + r * kSelThreads;
      if (i < len) make_key(pre[r], i);
    }
#pragma unroll 4
    for (int i = tid + kPre * kSelThreads; i < len; i += blockDim.x) make_key(src[i], i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    if (__any_sync(0xffffffffu, any) && lane == 0) atomicMax(&s_hmax, (int)lvl_digit(kmax, 0));
  }

  // ---- 3. cluster-wide select
  uint32_t bnd[3] = {0u, 0u, 0u};
  int need = kk;        // keys still to take among those in play
  int mine = 0;         // keys this CTA selects above the boundary so far
  int before = 0;       // keys lower-ranked CTAs select above the boundary so far
  int final_lvl = 2;    // -1: boundary members marked by bit 31 of their key
  cluster.sync();       // level-0 histograms and highest bins are complete

  // level 0: walk the bins top-down from the highest occupied one, 32 bins a
  // round; thread t reads CTA (t % 8)'s count of bin top - t / 8
  {
    if (tid < C) scan_buf[tid] = *cluster.map_shared_rank(&s_hmax, tid);
    __syncthreads();
    int hi = -1;
#pragma unroll
    for (int r = 0; r < C; ++r) hi = max(hi, scan_buf[r]);
    __syncthreads();
    const int r_of = tid % C;
    int add_mine = 0, add_before = 0;
    int carry = 0;   // keys in the bins above this round
    bool found = false;
    if (tid == 0) {
      s_bin = 0;
      s_above = 0;
    }
    for (int top = hi; top >= 0 && !found; top -= kSelThreads / C) {
      const int bin = top - tid / C;
      const int v = bin >= 0 ? *cluster.map_shared_rank(&hist0[bin], r_of) : 0;
      // bin total over the 8 CTAs: lanes 8k..8k+7 hold one bin
      int tot = v;
#pragma unroll
      for (int o = 1; o < C; o <<= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      int round_total;
      const int above = carry + block_exclusive_scan(r_of == 0 ? tot : 0, scan_buf, round_total);
      // `above` on lane r_of == 0 of each bin; share it with the bin's lanes
      const int above_bin = __shfl_sync(0xffffffffu, above, lane & ~(C - 1));
      const bool is_bnd = bin >= 0 && above_bin < need && above_bin + tot >= need;
      if (is_bnd) {
        bnd_cnt[r_of] = v;
        if (r_of == 0) {
          s_bin = bin;
          s_above = above_bin;
        }
      }
      found = __syncthreads_or(is_bnd);
      if (!found) {
        if (r_of == rank) add_mine += v;
        if (r_of < rank) add_before += v;
        carry += round_total;
        continue;
      }
      if (bin > s_bin) {
        if (r_of == rank) add_mine += v;
        if (r_of < rank) add_before += v;
      }
    }
    if (!found && tid == 0) flag_status(p.status, LOCKS_FLAG_BAD_SELECT);   // counts inconsistent: cannot happen
    block_sum2(add_mine, add_before, scan_buf);
    mine += add_mine;
    before += add_before;
    bnd[0] = (uint32_t)s_bin;
    need -= s_above;
  }
  int in_bin = 0, lower = 0;
#pragma unroll
  for (int r = 0; r < C; ++r) {
    in_bin += bnd_cnt[r];
    if (r < rank) lower += bnd_cnt[r];
  }
  if (in_bin == need) {   // the boundary bin is needed whole
    final_lvl = 0;
    before += lower;
    mine += bnd_cnt[rank];
    if (tid == 0) s_cutoff = len;
    __syncthreads();
  } else if (in_bin <= kMemberCap) {
    // The boundary bin's members go to rank 0 as (key, page); every CTA then
    // ranks all of them exactly (key descending, lower page first) and marks
    // its own taken members with bit 31 of their key (free: the keys are
    // non-negative floats).  The level-1 and level-2 histograms are unused
    // on this path: their storage holds the members (rank 0's copy in
    // hist1, a local copy in hist2).
    uint32_t* mkey = reinterpret_cast<uint32_t*>(hist1);
    int* mpage = hist1 + kMemberCap;
    // local copy as one sortable word per member: key above, ~page below, so
    // a larger word ranks first (larger key, then lower page)
    unsigned long long* lword = reinterpret_cast<unsigned long long*>(hist2);
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    uint32_t* rkey = cluster.map_shared_rank(mkey, 0) + lower;
    int* rpage = cluster.map_shared_rank(mpage, 0) + lower;
    for (int i = tid; i < len; i += blockDim.x) {
      const uint32_t key = sc.keys_s[i];
      if (lvl_digit(key, 0) == bnd[0]) {
        const int slot = atomicAdd(&s_cnt, 1);
        rkey[slot] = key;
        rpage[slot] = j0 + i;
      }
    }
    cluster.sync();   // every CTA's members are on rank 0
    {
      const uint32_t* k0 = cluster.map_shared_rank(mkey, 0);
      const int* p0 = cluster.map_shared_rank(mpage, 0);
      for (int x = tid; x < in_bin; x += blockDim.x)
        lword[x] = ((unsigned long long)k0[x] << 32) | (0xFFFFFFFFu - (uint32_t)p0[x]);
    }
    __syncthreads();
    // thread x ranks member x against all members (broadcast reads)
    int own_taken = 0, lower_taken = 0;
    for (int x = tid; x < in_bin; x += blockDim.x) {
      const unsigned long long wx = lword[x];
      int rk = 0;
#pragma unroll 8
      for (int y = 0; y < in_bin; ++y) rk += lword[y] > wx;
      if (rk < need) {
        const int px = (int)(0xFFFFFFFFu - (uint32_t)wx);
        if (px < j0) {
          ++lower_taken;
        } else if (px < j1) {
          ++own_taken;
          sc.keys_s[px - j0] = (uint32_t)(wx >> 32) | 0x80000000u;
        }
      }
    }
    block_sum2(own_taken, lower_taken, scan_buf);
    mine += own_taken;
    before += lower_taken;
    final_lvl = -1;
    if (tid == 0) s_cutoff = len;
    __syncthreads();
  } else {
    // crowded boundary bin: full histogram exchanges over the lower digits
    for (int lvl = 1; lvl < 3; ++lvl) {
      int* hist = lvl == 1 ? hist1 : hist2;
      for (int i = tid; i < len; i += blockDim.x) {
        const uint32_t key = sc.keys_s[i];
        if (lvl_digit(key, 0) == bnd[0] && (lvl < 2 || lvl_digit(key, 1) == bnd[1]))
          atomicAdd(&hist[lvl_digit(key, lvl)], 1);
      }
      cluster.sync();   // every CTA's histogram of this level is complete
      // thread t owns bins [lo_bin, lo_bin + 4), highest first
      constexpr int per = 4;
      const int top = (1 << 10) - 1 - per * tid;
      const int lo_bin = top - per + 1;
      int v[C][per];
#pragma unroll
      for (int r = 0; r < C; ++r) {   // every remote load first
        const int4 q = *reinterpret_cast<const int4*>(cluster.map_shared_rank(hist, r) + lo_bin);
        v[r][0] = q.x;
        v[r][1] = q.y;
        v[r][2] = q.z;
        v[r][3] = q.w;
      }
      int c[per] = {0, 0, 0, 0};
#pragma unroll
      for (int r = 0; r < C; ++r)
#pragma unroll
        for (int i = 0; i < per; ++i) c[i] += v[r][i];
      const int cnt_all = c[0] + c[1] + c[2] + c[3];
      int total;
      const int above = block_exclusive_scan(cnt_all, scan_buf, total);
      const bool holder = above < need && above + cnt_all >= need;
      if (holder) {
        int acc = above, bi = per - 1;
#pragma unroll
        for (int i = per - 1; i >= 0; --i) {
          if (acc + c[i] >= need) {
            bi = i;
            break;
          }
          acc += c[i];
        }
        s_bin = lo_bin + bi;
        s_above = acc;
      }
      __syncthreads();
      const int bin = s_bin;
      int add_mine = 0, add_before = 0;
#pragma unroll
      for (int r = 0; r < C; ++r)
#pragma unroll
        for (int i = 0; i < per; ++i) {
          if (lo_bin + i > bin) {
            if (r == rank) add_mine += v[r][i];
            if (r < rank) add_before += v[r][i];
          }
          if (lo_bin + i == bin) bnd_cnt[r] = v[r][i];
        }
      block_sum2(add_mine, add_before, scan_buf);   // (ends with a barrier: bnd_cnt is visible)
      mine += add_mine;
      before += add_before;
      bnd[lvl] = (uint32_t)bin;
      need -= s_above;
      int inb = 0, low = 0;
#pragma unroll
      for (int r = 0; r < C; ++r) {
        inb += bnd_cnt[r];
        if (r < rank) low += bnd_cnt[r];
      }
      if (inb == need || lvl == 2) {
        // inb == need: the boundary bin is needed whole.  Otherwise (last
        // level) its keys are equal in all 31 bits: lowest pages first, and
        // CTAs hold ascending page ranges.
        final_lvl = lvl;
        const int take = max(0, min(bnd_cnt[rank], need - low));
        before += min(low, need);
        mine += take;
        if (take == bnd_cnt[rank]) {
          if (tid == 0) s_cutoff = len;
        } else if (warp == 0) {
          // index of this CTA's first boundary key that is not taken
          int seen = 0, cut = len;
          for (int base = 0; base < len && cut == len; base += 32) {
            const int i = base + lane;
            bool hit = false;
            if (i < len) {
              const uint32_t key = sc.keys_s[i];
              hit = lvl_digit(key, 0) == bnd[0] && lvl_digit(key, 1) == bnd[1] &&
                    (lvl < 2 || lvl_digit(key, 2) == bnd[2]);
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, hit);
            const int cnt = __popc(bal);
            if (seen + cnt > take) {
              uint32_t x = bal;
              for (int k = 0; k < take - seen; ++k) x &= x - 1u;   // drop the members taken
              cut = base + __ffs(x) - 1;
            }
            seen += cnt;
          }
          if (lane == 0) s_cutoff = cut;
        }
        __syncthreads();
        break;
      }
    }
  }
  const int cutoff = s_cutoff;
  const int off = before;   // this CTA's first output slot

  // ---- 4. this CTA's selected pages, ascending, at slots [off, off + mine)
  {
    auto taken = [&](uint32_t key, int i) -> bool {
      if (final_lvl < 0) return (key >> 31) != 0u || lvl_digit(key, 0) > bnd[0];
      for (int l = 0; l <= final_lvl; ++l) {
        const uint32_t d = lvl_digit(key, l);
        if (d != bnd[l]) return d > bnd[l];
      }
      return i < cutoff;
    };
    const int nchunks = (len + 31) / 32;
    for (int ch = warp; ch < nchunks; ch += kSelWarps) {   // count per 32-key chunk
      const int i = ch * 32 + lane;
      const bool t = i < len && taken(sc.keys_s[i], i);
      const int cnt = __popc(__ballot_sync(0xffffffffu, t));
      if (lane == 0) chunk_base[ch] = cnt;
    }
    __syncthreads();
    {
      // exclusive scan of the chunk counts, two per thread
      const int a = 2 * tid < nchunks ? chunk_base[2 * tid] : 0;
      const int c2 = 2 * tid + 1 < nchunks ? chunk_base[2 * tid + 1] : 0;
      int total;
      const int ex = block_exclusive_scan(a + c2, scan_buf, total);
      if (2 * tid < nchunks) chunk_base[2 * tid] = ex;
      if (2 * tid + 1 < nchunks) chunk_base[2 * tid + 1] = ex + a;
    }
    __syncthreads();
    int* out0 = cluster.map_shared_rank(sc.out_blk, 0);
    for (int ch = warp; ch < nchunks; ch += kSelWarps) {
      const int i = ch * 32 + lane;
      const bool t = i < len && taken(sc.keys_s[i], i);
      const uint32_t bal = __ballot_sync(0xffffffffu, t);
      if (t) {
        const int pos = off + chunk_base[ch] + __popc(bal & ((1u << lane) - 1u));
        if (pos < kk) {
          sel[pos] = j0 + i;
          out0[pos] = sc.bt_slice ? sc.bt_slice[i] : j0 + i;
        }
      }
    }
  }
  if (tid == 0 && rank == 0) p.n_selected[unit] = kk;
  cluster.sync();   // rank 0's out_blk is complete; no CTA reads another's histograms after this
  return res;
}

}  // namespace locks
