// cluster_select.cuh -- LOCKS group-shared top-k selection (a4, a5) inside a
// thread-block cluster, shared by the selection kernel and the fused
// select + sparse-attention kernel.
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2, "Reconstruction and selection" and
// "Group-shared selection (GQA)": per-head page-mass shares exp(s_j - Z_g),
// averaged over the group's query heads into one table; the k largest entries
// (lower page index on ties) are attended.
//
// One cluster of kSelCluster CTAs per (request, KV head).  CTA r owns pages
// [n r / C, n (r + 1) / C).  Every CTA combines the scoring pass's partial
// log-sum-exps into Z_g and forms its slice's keys (the fp32 bits of the
// table entry; non-negative floats order like unsigned ints).  One pass of a
// 1024-bin order-preserving histogram (exponent and 4 mantissa bits) gives the
// bin holding the slice's k-th largest key; every key in or above that bin -- a superset of
// the slice's top k -- goes to rank 0's shared memory through distributed
// shared memory (a crowded bin falls back to an exact radix select).  The
// global top k is inside the union of those sets, so after one cluster
// barrier rank 0 finds the boundary bin of the candidates the same way,
// ranks the few candidates inside it exactly (key, then lower page), and
// writes the result in ascending page order; after a second barrier every CTA
// may read it.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "params.h"

namespace locks {

namespace cg = cooperative_groups;

constexpr int kSelThreads = 256;

// Merge of two (max, sum) log-sum-exp partials (natural-log units).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * fast_exp2((m - m2) * kLog2e) + s2;
    m = m2;
  } else {
    s += s2 * fast_exp2((m2 - m) * kLog2e);
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

// Warp-aggregated shared-memory histogram add: lanes holding the same bin add once.
__device__ __forceinline__ void hist_add(int* hist, uint32_t bin, bool active) {
  const uint32_t act = __ballot_sync(0xffffffffu, active);
  if (active) {
    const uint32_t peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1)) atomicAdd(&hist[bin], (int)__popc(peers));
  }
}

// Selection rule produced by block_radix_select: a key k is selected when
// (k >> shift) > prefix, or when (k >> shift) == prefix and it is among the
// first `take` such keys in index order.
struct RadixCut {
  uint32_t prefix;
  int shift;
  int take;
};

// Block-wide radix select (8-bit digits, MSB first) of the `need`-th largest
// of keys[0, cnt) in shared memory; stops early once the boundary bin holds
// exactly the keys still needed.  Every thread of the block must call it.
static __device__ RadixCut block_radix_select(const uint32_t* keys, int cnt, int need) {
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem, s_shift, s_done;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_prefix = 0;
    s_rem = need;
    s_shift = 0;
    s_done = 0;
  }
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int base = tid & ~31; base < cnt; base += blockDim.x) {
      const int i = base + lane;
      uint32_t k = 0;
      bool match = false;
      if (i < cnt) {
        k = keys[i];
        match = (k & hmask) == (prefix & hmask);
      }
      hist_add(hist, (k >> shift) & 255u, match);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits [8l, 8l+8); find the digit holding the rem-th
      // largest key, scanning from the top
      int c[8], lt = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[8 * lane + i];
        lt += c[i];
      }
      int above = lt;   // inclusive suffix sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, above, o);
        if (lane + o < 32) above += y;
      }
      const int strictly_above = above - lt;
      const int rem = s_rem;
      if (strictly_above < rem && above >= rem) {
        int acc = strictly_above;
        int digit = 8 * lane, dcount = 0;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
          if (acc + c[i] >= rem) {
            digit = 8 * lane + i;
            dcount = c[i];
            break;
          }
          acc += c[i];
        }
        s_prefix = prefix | ((uint32_t)digit << shift);
        s_rem = rem - acc;
        s_shift = shift;
        if (rem - acc == dcount) s_done = 1;   // every key left in the bin is needed
      }
    }
    __syncthreads();
    if (s_done) break;
  }
  RadixCut cut{s_prefix >> s_shift, s_shift, s_rem};
  __syncthreads();
  return cut;
}

// Histogram bin of a key: order-preserving (a larger key never falls in a
// lower bin).  Table entries lie in [0, 1]; exponents 64..127 get 16 bins
// each (4 mantissa bits, 6.25 % wide), everything below 2^-63 shares bin 0.
constexpr int kBins = 1024;
constexpr int kExactCap = 256;     // boundary-bin members ranked pairwise
static_assert(3 * kExactCap <= kBins, "bin members reuse the histogram");
__device__ __forceinline__ int key_bin(uint32_t key) {
  const int b = (int)(key >> 19) - 1024;
  return b < 0 ? 0 : (b > kBins - 1 ? kBins - 1 : b);
}

// Block-wide histogram of key_bin over keys[0, cnt) and the bin holding the
// need-th largest key (1 <= need <= cnt).  Every thread must call it.
struct BinCut {
  int bin;
  int above;   // keys in higher bins
  int count;   // keys in the bin
};
static __device__ BinCut block_bin_cut(const uint32_t* keys, int cnt, int need, int* hist, int* scan_buf) {
  __shared__ BinCut s_cut;
  const int tid = threadIdx.x;
  constexpr int kPer = kBins / kSelThreads;
  for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < cnt; i += blockDim.x) atomicAdd(&hist[key_bin(keys[i])], 1);
  __syncthreads();
  // thread t owns bins top, top - 1, ..., top - kPer + 1, scanned from the top
  const int top = kBins - 1 - kPer * tid;
  int c[kPer], tot = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    c[i] = hist[top - i];
    tot += c[i];
  }
  int all;
  const int above = block_exclusive_scan(tot, scan_buf, all);
  if (above < need && above + tot >= need) {
    int acc = above;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (acc + c[i] >= need) {
        s_cut = BinCut{top - i, acc, c[i]};
        break;
      }
      acc += c[i];
    }
  }
  __syncthreads();
  const BinCut cut = s_cut;
  __syncthreads();
  return cut;
}

// First item of CTA c of the scoring grid, and the CTA holding item x.
__host__ __device__ __forceinline__ long long score_item_begin(long long c, long long n_items, long long grid) {
  return (c * n_items) / grid;
}
__host__ __device__ __forceinline__ int score_cta_of(long long x, long long n_items, long long grid) {
  return (int)(((x + 1) * grid - 1) / n_items);
}

// Result of cluster_select for the calling CTA.
struct ClusterSel {
  int n;        // full pages of the request (0 when its length is invalid)
  int tail;     // tokens of the open tail page
  int kk;       // pages selected for the unit
};

// Scratch layout (shared memory) handed to cluster_select:
//   keys_s   ceil(max_pages / C) words: this CTA's keys;
//   bt_slice optional block ids of this CTA's pages (nullptr: none);
//   cand_*   C * min(budget, ceil(max_pages / C)) entries each, used on rank 0:
//            the local winners of every CTA, then rank 0's selection;
//   out_blk  rank 0: the selected pages' physical blocks (bt_slice given) or
//            page indices, ascending by page.
struct SelScratch {
  uint32_t* keys_s;
  const int* bt_slice;
  uint32_t* cand_key;
  int* cand_page;
  int* cand_blk;
  int cand_stride;      // entries per CTA in the cand arrays
  int* out_blk;
};

// Selects the pages of unit (b, h) = blockIdx.y.  Every thread of every CTA
// of the cluster must call it.  Writes `selected` and `n_selected`; ends with
// a cluster barrier after which rank 0's out_blk[0, kk) may be read through
// distributed shared memory.
static __device__ ClusterSel cluster_select(const SelectParams& p, const SelScratch& sc) {
  __shared__ float red[kSelThreads / 32][kGroup], red2[kSelThreads / 32][kGroup];
  __shared__ int hist_s[kBins];
  __shared__ float zl[kGroup];
  __shared__ int scan_buf[32];
  __shared__ int cand_count[kSelCluster];
  __shared__ int s_ncover;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int unit = blockIdx.y;              // (request, KV head)
  const int b = unit / p.H_kv, h = unit % p.H_kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = p.seq_lens[b];
  int32_t* sel = p.selected + (int64_t)unit * p.budget;
  ClusterSel res{0, 0, 0};
  // every CTA of a cluster takes the same branches below (same unit)
  if (L < 0 || (L + kPage - 1) / kPage > p.max_pages) {
    if (tid == 0 && rank == 0) {
      p.n_selected[unit] = 0;
      if (h == 0) flag_status(p.status, LOCKS_FLAG_BAD_SEQLEN);
    }
    cluster.sync();
    return res;
  }
  const int n = L / kPage;
  res.n = n;
  res.tail = L % kPage;
  const int kk = min(p.budget, n);
  res.kk = kk;
  const int j0 = (int)(((long long)n * rank) / kSelCluster);
  const int j1 = (int)(((long long)n * (rank + 1)) / kSelCluster);
  const int len = j1 - j0;
  if (n <= p.budget) {   // every full page is selected
    for (int i = tid; i < len; i += blockDim.x) {
      sel[j0 + i] = j0 + i;
      // rank 0 holds the list: fill its out_blk through distributed shared memory
      *cluster.map_shared_rank(&sc.out_blk[j0 + i], 0) = sc.bt_slice ? sc.bt_slice[i] : j0 + i;
    }
    if (tid == 0 && rank == 0) p.n_selected[unit] = n;
    cluster.sync();
    return res;
  }

  // ---- this thread's first scores, issued before the partials' loads
  const float4* srow = reinterpret_cast<const float4*>(p.scores + (int64_t)unit * p.max_pages * kGroup);
  constexpr int kPre = 4;
  float4 pre[kPre];
#pragma unroll
  for (int r = 0; r < kPre; ++r) {
    const int i = tid + r * kSelThreads;
    pre[r] = i < len ? srow[j0 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- Z_g from the scoring pass's partials: slots (unit u, covering CTA)
  const int hg = h / p.h_cta, hl = h % p.h_cta;
  const long long u = (long long)b * p.head_groups + hg;
  if (tid == 0) {
    const int cf = score_cta_of(u * p.n_chunks, p.n_items, p.score_grid);
    const int cl = score_cta_of(u * p.n_chunks + p.n_chunks - 1, p.n_items, p.score_grid);
    s_ncover = cl - cf + 1;
  }
  __syncthreads();
  const int nent = s_ncover * p.wph;
  {
    // each warp folds entries warp, warp + 8, ... (lane-strided), then the
    // block merges the 8 warps' (max, sum) per head
    float m[kGroup] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    float sm[kGroup] = {0.f, 0.f, 0.f, 0.f};
    for (int i = tid; i < nent; i += blockDim.x) {
      const int slot = i / p.wph, sub = i % p.wph;
      const float4* part = reinterpret_cast<const float4*>(
          p.partials + ((((int64_t)u * p.seg_slots + slot) * 8 + hl * p.wph + sub) * kGroup * 2));
      const float4 a = part[0], c = part[1];   // (m0 s0 m1 s1) (m2 s2 m3 s3)
      lse_merge(m[0], sm[0], a.x, a.y);
      lse_merge(m[1], sm[1], a.z, a.w);
      lse_merge(m[2], sm[2], c.x, c.y);
      lse_merge(m[3], sm[3], c.z, c.w);
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      float mx = m[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sv = m[g] == -INFINITY ? 0.f : sm[g] * fast_exp2((m[g] - mx) * kLog2e);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
      if (lane == 0) {
        red[warp][g] = mx;
        red2[warp][g] = sv;
      }
    }
    __syncthreads();
    if (tid < kGroup) {
      float mx = -INFINITY, sv = 0.f;
#pragma unroll
      for (int w = 0; w < kSelThreads / 32; ++w) lse_merge(mx, sv, red[w][tid], red2[w][tid]);
      zl[tid] = (mx + logf(sv)) * kLog2e;   // log2 units
    }
    __syncthreads();
  }

  // ---- keys of this slice
  {
    const float z0 = zl[0], z1 = zl[1], z2 = zl[2], z3 = zl[3];
    auto key_of = [&](float4 sv) {
      float avg = 0.25f * (fast_exp2(sv.x * kLog2e - z0) + fast_exp2(sv.y * kLog2e - z1) +
                           fast_exp2(sv.z * kLog2e - z2) + fast_exp2(sv.w * kLog2e - z3));
      if (!(avg >= 0.f) || isinf(avg)) avg = 0.f;
      return __float_as_uint(avg);
    };
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int i = tid + r * kSelThreads;
      if (i < len) sc.keys_s[i] = key_of(pre[r]);
    }
#pragma unroll 4
    for (int i = tid + kPre * kSelThreads; i < len; i += blockDim.x) sc.keys_s[i] = key_of(srow[j0 + i]);
  }
  __syncthreads();

  // ---- this slice's candidates (a superset of its top kk), to rank 0 in
  // ascending page order
  {
    const int lk = min(kk, len);
    // selection rule for this slice: key >> shift > prefix, or == prefix and
    // among the first `take` (index order)
    // (bin rule: every key whose bin is at or above the cut bin)
    RadixCut cut{0u, 31, len};   // len <= kk: every key (bit 31 is clear)
    int min_bin = 0;
    bool by_bin = true;
    if (len > kk) {
      const BinCut bc = block_bin_cut(sc.keys_s, len, lk, hist_s, scan_buf);
      if (bc.above + bc.count <= sc.cand_stride) {
        min_bin = bc.bin;
      } else {
        by_bin = false;
        cut = block_radix_select(sc.keys_s, len, lk);   // crowded bin: exact local top lk
      }
    }
    const int per = (len + blockDim.x - 1) / blockDim.x;
    const int c0 = min(len, tid * per), c1 = min(len, c0 + per);
    int gt = 0, eq = 0;
    for (int i = c0; i < c1; ++i) {
      const uint32_t key = sc.keys_s[i];
      if (by_bin) {
        gt += key_bin(key) >= min_bin;
      } else {
        const uint32_t k = key >> cut.shift;
        gt += k > cut.prefix;
        eq += k == cut.prefix;
      }
    }
    int gt_tot, eq_tot;
    const int gt_before = block_exclusive_scan(gt, scan_buf, gt_tot);
    const int eq_before = block_exclusive_scan(eq, scan_buf, eq_tot);
    const int take = max(0, min(eq, cut.take - eq_before));
    int pos = gt_before + max(0, min(eq_before, cut.take));
    int taken = 0;
    uint32_t* rkey = cluster.map_shared_rank(sc.cand_key, 0) + rank * sc.cand_stride;
    int* rpage = cluster.map_shared_rank(sc.cand_page, 0) + rank * sc.cand_stride;
    int* rblk = cluster.map_shared_rank(sc.cand_blk, 0) + rank * sc.cand_stride;
    for (int i = c0; i < c1; ++i) {
      const uint32_t key = sc.keys_s[i];
      const uint32_t k = key >> cut.shift;
      const bool in_bin = by_bin && key_bin(key) >= min_bin;
      const bool eqk = !by_bin && k == cut.prefix;
      if (in_bin || (!by_bin && k > cut.prefix) || (eqk && taken < take)) {
        if (eqk) ++taken;
        rkey[pos] = key;
        rpage[pos] = j0 + i;
        rblk[pos] = sc.bt_slice ? sc.bt_slice[i] : j0 + i;
        ++pos;
      }
    }
    if (tid == 0) *cluster.map_shared_rank(&cand_count[rank], 0) = gt_tot + min(eq_tot, cut.take);
  }
  cluster.sync();   // every CTA's local winners are on rank 0

  // ---- rank 0: exact top-kk among the candidates, ascending page order
  if (rank == 0) {
    // pack the C segments in rank order (rank r's pages precede rank r+1's)
    __shared__ int seg_base[kSelCluster + 1];
    if (tid == 0) {
      int acc = 0;
      for (int r = 0; r < kSelCluster; ++r) {
        seg_base[r] = acc;
        acc += cand_count[r];
      }
      seg_base[kSelCluster] = acc;
    }
    __syncthreads();
    const int total = seg_base[kSelCluster];
    // compact in place: segment r moves from [r * stride, ...) down to seg_base[r]
    // (seg_base[r] <= r * stride, and segments move in rank order, one
    // segment per pass so no entry is overwritten before it is read)
    for (int r = 1; r < kSelCluster; ++r) {
      const int cnt = cand_count[r], from = r * sc.cand_stride, to = seg_base[r];
      if (to != from) {
        for (int i0 = 0; i0 < cnt; i0 += blockDim.x) {
          const int i = i0 + tid;
          uint32_t k = 0;
          int pg = 0, bk = 0;
          if (i < cnt) {
            k = sc.cand_key[from + i];
            pg = sc.cand_page[from + i];
            bk = sc.cand_blk[from + i];
          }
          __syncthreads();
          if (i < cnt) {
            sc.cand_key[to + i] = k;
            sc.cand_page[to + i] = pg;
            sc.cand_blk[to + i] = bk;
          }
          __syncthreads();
        }
      }
    }
    // boundary bin of the kk-th largest candidate; its members are ranked
    // exactly (key descending, then lower page) when few, else a radix
    // select over all candidates decides
    __shared__ int bin_n;
    const BinCut bc = block_bin_cut(sc.cand_key, total, kk, hist_s, scan_buf);
    // the histogram is free again: it holds the boundary bin's members
    int* bin_idx = hist_s;
    uint32_t* bin_key = reinterpret_cast<uint32_t*>(hist_s + kExactCap);
    int* bin_page = hist_s + 2 * kExactCap;
    const int need = kk - bc.above;
    const bool exact_bin = bc.count <= kExactCap;
    RadixCut fin{0u, 0, 0};
    if (exact_bin) {
      if (tid == 0) bin_n = 0;
      __syncthreads();
      for (int i = tid; i < total; i += blockDim.x) {
        const uint32_t key = sc.cand_key[i];
        if (key_bin(key) == bc.bin) {
          const int slot = atomicAdd(&bin_n, 1);
          bin_idx[slot] = i;
          bin_key[slot] = key;
          bin_page[slot] = sc.cand_page[i];
        }
      }
      __syncthreads();
      // a member is taken when fewer than `need` members precede it
      // (larger key, or equal key and lower page); taken members get bit 31
      // of their candidate key set (free: the keys are non-negative floats)
      const int nb = bin_n;
      for (int a = tid; a < nb; a += blockDim.x) {
        const uint32_t ka = bin_key[a];
        const int pa = bin_page[a];
        int before = 0;
        for (int bb = 0; bb < nb; ++bb) {
          const uint32_t kb = bin_key[bb];
          before += kb > ka || (kb == ka && bin_page[bb] < pa);
        }
        if (before < need) sc.cand_key[bin_idx[a]] = ka | 0x80000000u;
      }
      __syncthreads();
    } else {
      fin = block_radix_select(sc.cand_key, total, kk);
    }
    const int per = (total + blockDim.x - 1) / blockDim.x;
    const int c0 = min(total, tid * per), c1 = min(total, c0 + per);
    auto chosen_exact = [&](uint32_t key) {
      return (key >> 31) != 0u || key_bin(key) > bc.bin;
    };
    int pos;
    if (exact_bin) {
      int cnt = 0;
      for (int i = c0; i < c1; ++i) cnt += chosen_exact(sc.cand_key[i]);
      int all;
      pos = block_exclusive_scan(cnt, scan_buf, all);
      for (int i = c0; i < c1; ++i)
        if (chosen_exact(sc.cand_key[i])) {
          if (pos < kk) {
            sel[pos] = sc.cand_page[i];
            sc.out_blk[pos] = sc.cand_blk[i];
          }
          ++pos;
        }
    } else {
      int gt = 0, eq = 0;
      for (int i = c0; i < c1; ++i) {
        const uint32_t k = sc.cand_key[i] >> fin.shift;
        gt += k > fin.prefix;
        eq += k == fin.prefix;
      }
      int gt_tot, eq_tot;
      const int gt_before = block_exclusive_scan(gt, scan_buf, gt_tot);
      const int eq_before = block_exclusive_scan(eq, scan_buf, eq_tot);
      const int take = max(0, min(eq, fin.take - eq_before));
      pos = gt_before + max(0, min(eq_before, fin.take));
      int taken = 0;
      for (int i = c0; i < c1; ++i) {
        const uint32_t k = sc.cand_key[i] >> fin.shift;
        if (k > fin.prefix || (k == fin.prefix && taken < take)) {
          if (k == fin.prefix) ++taken;
          if (pos < kk) {
            sel[pos] = sc.cand_page[i];
            sc.out_blk[pos] = sc.cand_blk[i];
          }
          ++pos;
        }
      }
    }
    if (tid == 0) p.n_selected[unit] = kk;
  }
  cluster.sync();   // rank 0's out_blk is complete
  return res;
}

}  // namespace locks
