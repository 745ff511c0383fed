// context_parallel.cu -- one request's pages held by several GPUs (shards):
// the kernels of each shard's part of a LOCKS decode step.
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2 ("Reconstruction and selection",
// "Group-shared selection (GQA)") and §4 (long contexts, 1M+ tokens): the
// selection normalises each query head's page scores over ALL of a request's
// pages (Z_g) and keeps the k largest group-mean shares.  With the pages
// split over shards that needs three exchanges, each a gather of small
// per-shard results (the host moves them; no kernel waits on another GPU):
//   1. per (request, KV head, head g): the shard's (max, sum) of its page
//      scores in log2 units -> every shard forms the same Z_g
//      (cp_pairs_kernel, then cluster_select with kExtZ);
//   2. each shard's local top-k pages with their exact selection keys and
//      global page indices (cp_candidates_kernel) -> the global top-k is the
//      top-k of the union of local top-k lists (a page of the global top-k is
//      beaten by fewer than k pages anywhere, so by fewer than k of its own
//      shard); cp_merge_select_kernel keeps this shard's part of it;
//   3. each shard's unnormalised attention state (m, l, o) over its selected
//      pages (and the open tail page, which the last shard holds) ->
//      cp_merge_attn_kernel combines them by the online-softmax rule.
// Keys come from group_key (cluster_select.cuh), so they compare across
// shards exactly as on one GPU; ties go to the lower global page index.

#include <cstdint>

#include "cluster_select.cuh"
#include "common.cuh"
#include "params.h"

namespace locks {

constexpr int kCpThreads = 256;
constexpr int kCpMaxCandidates = 16384;   // n_shards * budget words sorted in shared memory

// Shard pages of request b: n = L / 16 full pages (L = the shard's tokens);
// -1 for an invalid length.
__device__ __forceinline__ int cp_full_pages(const int32_t* lens, int b, int max_pages) {
  const int L = lens[b];
  if (L < 0 || (L + kPage - 1) / kPage > max_pages) return -1;
  return L / kPage;
}

// (max, sum) of 2^(s log2 e) over the shard's full pages, per head.
__global__ void __launch_bounds__(kCpThreads) cp_pairs_kernel(const int32_t* shard_lens, const float* scores,
                                                              float2* pairs, uint32_t* status, int H,
                                                              int max_pages) {
  __shared__ float red_m[kCpThreads / 32][kGroup], red_s[kCpThreads / 32][kGroup];
  const int unit = blockIdx.x, b = unit / H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int n = cp_full_pages(shard_lens, b, max_pages);
  if (n < 0) {
    if (tid == 0 && unit % H == 0) flag_status(status, LOCKS_FLAG_BAD_SEQLEN);
    n = 0;
  }
  const float4* row = reinterpret_cast<const float4*>(scores + (int64_t)unit * max_pages * kGroup);
  float m[kGroup] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float s[kGroup] = {0.f, 0.f, 0.f, 0.f};
  for (int j = tid; j < n; j += kCpThreads) {
    const float4 v = row[j];
    const float x[kGroup] = {v.x * kLog2e, v.y * kLog2e, v.z * kLog2e, v.w * kLog2e};
#pragma unroll
    for (int g = 0; g < kGroup; ++g) lse2_merge(m[g], s[g], x[g], 1.f);
  }
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[g], o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s[g], o);
      lse2_merge(m[g], s[g], m2, s2);
    }
    if (lane == 0) {
      red_m[warp][g] = m[g];
      red_s[warp][g] = s[g];
    }
  }
  __syncthreads();
  if (tid < kGroup) {
    float mx = -INFINITY, sv = 0.f;
    for (int w = 0; w < kCpThreads / 32; ++w) lse2_merge(mx, sv, red_m[w][tid], red_s[w][tid]);
    pairs[(int64_t)unit * kGroup + tid] = make_float2(mx, sv);
  }
}

// The shard's selected pages (local indices, ascending, in `pages`) become
// candidates: global page index and selection key, in place.
__global__ void __launch_bounds__(128) cp_candidates_kernel(const float* scores, const float2* zpairs, int n_shards,
                                                            const int32_t* page_offset, int32_t* pages,
                                                            uint32_t* keys, const int32_t* counts, int H,
                                                            int max_pages, int budget, int units) {
  __shared__ float zl[kGroup];
  const int unit = blockIdx.x, b = unit / H;
  if (threadIdx.x < kGroup) zl[threadIdx.x] = z_from_shards(zpairs, n_shards, units, unit, threadIdx.x);
  __syncthreads();
  const int cnt = counts[unit];
  const int off = page_offset[b];
  const float4* row = reinterpret_cast<const float4*>(scores + (int64_t)unit * max_pages * kGroup);
  for (int i = threadIdx.x; i < cnt && i < budget; i += blockDim.x) {
    const int j = pages[(int64_t)unit * budget + i];
    uint32_t key = 0u;
    if (j >= 0 && j < max_pages) key = group_key(row[j], zl[0], zl[1], zl[2], zl[3]);
    keys[(int64_t)unit * budget + i] = key;
    pages[(int64_t)unit * budget + i] = j + off;
  }
}

// Global top-k of the union of every shard's candidates; this shard keeps its
// own, as local page indices in ascending order.
__global__ void __launch_bounds__(kCpThreads) cp_merge_select_kernel(
    const int32_t* cand_pages, const uint32_t* cand_keys, const int32_t* cand_counts, int n_shards, int shard,
    const int32_t* page_offset, int32_t* selected, int32_t* n_selected, int H, int budget, int units, int n_pow2) {
  extern __shared__ unsigned long long words[];   // n_pow2 words: key << 32 | ~page
  __shared__ int scan_buf[32];
  const int unit = blockIdx.x, b = unit / H, tid = threadIdx.x;
  int total = 0;
  for (int r = 0; r < n_shards; ++r) total += min(budget, max(0, cand_counts[(int64_t)r * units + unit]));
  for (int x = tid; x < n_pow2; x += kCpThreads) {
    const int r = x / max(budget, 1), i = x - r * max(budget, 1);
    unsigned long long w = 0ull;
    if (r < n_shards && i < min(budget, max(0, cand_counts[(int64_t)r * units + unit]))) {
      const int64_t at = ((int64_t)r * units + unit) * budget + i;
      w = ((unsigned long long)cand_keys[at] << 32) | (0xFFFFFFFFu - (uint32_t)cand_pages[at]);
    }
    words[x] = w;
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int x = tid; x < n_pow2; x += kCpThreads) {
        const int y = x ^ stride;
        if (y > x) {
          const bool desc = (x & size) == 0;
          const unsigned long long a = words[x], c = words[y];
          if (desc ? (a < c) : (a > c)) {
            words[x] = c;
            words[y] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const int kk = min(budget, total);
  const unsigned long long thr = kk > 0 ? words[kk - 1] : ~0ull;
  // this shard's candidates at or above the k-th word, in their (ascending) order
  const int mine = min(budget, max(0, cand_counts[(int64_t)shard * units + unit]));
  const int off = page_offset[b];
  int written = 0;
  for (int base = 0; base < mine; base += kCpThreads) {
    const int i = base + tid;
    bool keep = false;
    int local = 0;
    if (i < mine) {
      const int64_t at = ((int64_t)shard * units + unit) * budget + i;
      const unsigned long long w =
          ((unsigned long long)cand_keys[at] << 32) | (0xFFFFFFFFu - (uint32_t)cand_pages[at]);
      keep = kk > 0 && w >= thr;
      local = cand_pages[at] - off;
    }
    int round_total;
    const int pos = written + block_exclusive_scan(keep ? 1 : 0, scan_buf, round_total);
    if (keep && pos < budget) selected[(int64_t)unit * budget + pos] = local;
    written += round_total;
  }
  if (tid == 0) n_selected[unit] = min(written, budget);
}

// out = (sum_r 2^(m_r - M) o_r) / (sum_r 2^(m_r - M) l_r) over the shards'
// states [shard][batch * H * G][2 + 128] (m in log2 units).
__global__ void __launch_bounds__(kHeadDim) cp_merge_attn_kernel(const float* states, int n_shards, int rows,
                                                                  float* out) {
  const int row = blockIdx.x, d = threadIdx.x;
  constexpr int kStride = 2 + kHeadDim;
  float M = -INFINITY;
  for (int r = 0; r < n_shards; ++r) M = fmaxf(M, states[((int64_t)r * rows + row) * kStride]);
  float Ls = 0.f, Os = 0.f;
  if (M != -INFINITY) {
    for (int r = 0; r < n_shards; ++r) {
      const float* st = states + ((int64_t)r * rows + row) * kStride;
      const float f = fast_exp2(st[0] - M);
      Ls += st[1] * f;
      Os += st[2 + d] * f;
    }
  }
  out[(int64_t)row * kHeadDim + d] = Ls > 0.f ? Os / Ls : 0.f;
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_cp_pairs(const int32_t* shard_lens, const float* scores, float* pairs, uint32_t* status,
                            int units, int H, int max_pages, cudaStream_t stream) {
  cp_pairs_kernel<<<units, kCpThreads, 0, stream>>>(shard_lens, scores, reinterpret_cast<float2*>(pairs), status, H,
                                                     max_pages);
  return cudaGetLastError();
}

cudaError_t launch_cp_candidates(const float* scores, const float* zpairs, int n_shards, const int32_t* page_offset,
                                 int32_t* pages, uint32_t* keys, const int32_t* counts, int units, int H,
                                 int max_pages, int budget, cudaStream_t stream) {
  cp_candidates_kernel<<<units, 128, 0, stream>>>(scores, reinterpret_cast<const float2*>(zpairs), n_shards,
                                                  page_offset, pages, keys, counts, H, max_pages, budget, units);
  return cudaGetLastError();
}

int cp_merge_pow2(int n_shards, int budget) {
  int n = 1;
  while (n < n_shards * budget) n <<= 1;
  return n;
}

bool cp_merge_fits(int n_shards, int budget) { return (int64_t)n_shards * budget <= kCpMaxCandidates; }

cudaError_t launch_cp_merge_select(const int32_t* cand_pages, const uint32_t* cand_keys, const int32_t* cand_counts,
                                   int n_shards, int shard, const int32_t* page_offset, int32_t* selected,
                                   int32_t* n_selected, int units, int H, int budget, cudaStream_t stream) {
  const int n_pow2 = cp_merge_pow2(n_shards, budget);
  const size_t smem = (size_t)n_pow2 * sizeof(unsigned long long);
  static DynSmemAttr smem_attr;
  const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(cp_merge_select_kernel), smem, smem_attr);
  if (e != cudaSuccess) return e;
  cp_merge_select_kernel<<<units, kCpThreads, smem, stream>>>(cand_pages, cand_keys, cand_counts, n_shards, shard,
                                                              page_offset, selected, n_selected, H, budget, units,
                                                              n_pow2);
  return cudaGetLastError();
}

cudaError_t launch_cp_merge_attn(const float* states, int n_shards, int rows, float* out, cudaStream_t stream) {
  cp_merge_attn_kernel<<<rows, kHeadDim, 0, stream>>>(states, n_shards, rows, out);
  return cudaGetLastError();
}

}  // namespace locks
