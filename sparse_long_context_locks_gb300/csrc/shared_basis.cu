// shared_basis.cu -- the shared-projection ablation: page scores through one
// rank-rho key basis per KV head instead of each page's own basis.
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §3, "impossibility of shared projections": a
// fixed, query-independent low-rank projection shared by every page of a head
// cannot represent within-page directions outside its span, so a page whose
// mass rests on such a direction (a key along the query) is ranked by its
// centroid alone.  This file builds the comparison selector the paper argues
// against, with the same score equation and selection:
//   record (per page-head, fp32): mu_j [128], c_i = U^T (k_i - mu_j) [16][rho];
//   s_j(q) = log sum_i exp((q.mu_j + (U^T q).c_i) / sqrt(d)),
// with U [128][rho] the caller's basis of the KV head (e.g. the top principal
// directions of all of its centred keys).  The scores go to the same table
// as locks_score's, so locks_select / locks_sparse_decode run on them.

#include <cstdint>

#include "common.cuh"
#include "params.h"

namespace locks {

constexpr int kSbWarps = 8;
constexpr int kSbBuildWarps = 4;   // 32 KB of centred keys a CTA
constexpr int kSbPagesPerCta = 64;

// One warp per page-head: centroid, centred keys, coefficients in the basis.
__global__ void __launch_bounds__(kSbBuildWarps * 32) shared_basis_build_kernel(
    const __nv_bfloat16* k_cache, int64_t num_blocks, const int32_t* block_ids, int n_build, int H,
    const float* basis, int rho, uint8_t* records, uint32_t* status) {
  __shared__ float xs[kSbBuildWarps][kPage][kHeadDim];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ph = (int64_t)blockIdx.x * kSbBuildWarps + warp;
  if (ph >= (int64_t)n_build * H) return;
  const int64_t blk = block_ids[ph / H];
  const int h = (int)(ph % H);
  if (blk < 0 || blk >= num_blocks) {
    if (lane == 0) flag_status(status, LOCKS_FLAG_BAD_BLOCK);
    return;
  }
  const __nv_bfloat16* src = k_cache + (blk * H + h) * (int64_t)(kPage * kHeadDim);
  float* rec = reinterpret_cast<float*>(records + (blk * H + h) * (int64_t)(512 + 64 * rho));
  // lane holds dims 4 lane .. 4 lane + 3 of every key
  float mu[4] = {0.f, 0.f, 0.f, 0.f};
  float kv[kPage][4];
#pragma unroll
  for (int r = 0; r < kPage; ++r) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      kv[r][e] = __bfloat162float(src[r * kHeadDim + 4 * lane + e]);
      mu[e] += kv[r][e];
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    mu[e] *= 1.f / kPage;
    rec[4 * lane + e] = mu[e];
  }
#pragma unroll
  for (int r = 0; r < kPage; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) xs[warp][r][4 * lane + e] = kv[r][e] - mu[e];
  __syncwarp();
  // c[i][k] = sum_d X[i][d] U[d][k]: lane takes (i, k) pairs
  const float* U = basis + (int64_t)h * kHeadDim * rho;
  float* C = rec + kHeadDim;
  for (int idx = lane; idx < kPage * rho; idx += 32) {
    const int i = idx / rho, k = idx % rho;
    float acc = 0.f;
    for (int d = 0; d < kHeadDim; ++d) acc = fmaf(xs[warp][i][d], U[d * rho + k], acc);
    C[i * rho + k] = acc;
  }
}

// CTA per (64-page chunk, request x KV head): u = U^T q once, then one warp
// per page.
__global__ void __launch_bounds__(kSbWarps * 32) shared_basis_score_kernel(
    const __nv_bfloat16* q, const float* basis, int rho, const uint8_t* records, int64_t num_blocks,
    const int32_t* block_table, const int32_t* seq_lens, int H, int max_pages, float* scores, uint32_t* status) {
  extern __shared__ float sb_u[];              // [G][rho]
  __shared__ float qs[kGroup][kHeadDim];
  const int unit = blockIdx.y, b = unit / H, h = unit % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = seq_lens[b];
  if (L < 0 || (L + kPage - 1) / kPage > max_pages) {
    if (tid == 0 && h == 0 && blockIdx.x == 0) flag_status(status, LOCKS_FLAG_BAD_SEQLEN);
    return;
  }
  const int n = L / kPage;
  const int j0 = blockIdx.x * kSbPagesPerCta;
  if (j0 >= n) return;
  const __nv_bfloat16* qg = q + ((int64_t)b * H * kGroup + (int64_t)h * kGroup) * kHeadDim;
  for (int x = tid; x < kGroup * kHeadDim; x += blockDim.x) qs[x / kHeadDim][x % kHeadDim] = __bfloat162float(qg[x]);
  __syncthreads();
  const float* U = basis + (int64_t)h * kHeadDim * rho;
  for (int x = tid; x < kGroup * rho; x += blockDim.x) {
    const int g = x / rho, k = x % rho;
    float acc = 0.f;
    for (int d = 0; d < kHeadDim; ++d) acc = fmaf(qs[g][d], U[d * rho + k], acc);
    sb_u[g * rho + k] = acc;
  }
  __syncthreads();
  const float inv_sqrt_d = 0.08838834764831845f;
  const size_t rec_bytes = 512 + 64 * (size_t)rho;
  for (int j = j0 + warp; j < min(n, j0 + kSbPagesPerCta); j += kSbWarps) {
    const int64_t blk = block_table[(int64_t)b * max_pages + j];
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) flag_status(status, LOCKS_FLAG_BAD_BLOCK);
      continue;
    }
    const float* rec = reinterpret_cast<const float*>(records + (blk * H + h) * rec_bytes);
    float part[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc = fmaf(qs[g][4 * lane + e], rec[4 * lane + e], acc);
      part[g] = acc;
    }
#pragma unroll
    for (int g = 0; g < kGroup; ++g)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part[g] += __shfl_xor_sync(0xffffffffu, part[g], o);
    const float* C = rec + kHeadDim;
    const int i = lane & 15;
    float s_out[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int g = 2 * half + (lane >> 4);
      float dev = 0.f;
      for (int k = 0; k < rho; ++k) dev = fmaf(C[i * rho + k], sb_u[g * rho + k], dev);
      const float qmu = g == 0 ? part[0] : g == 1 ? part[1] : g == 2 ? part[2] : part[3];
      const float x = (qmu + dev) * inv_sqrt_d;
      float m = x;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float e = expf(x - m);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
      s_out[half] = m + logf(e);
    }
    float* srow = scores + (((int64_t)b * H + h) * max_pages + j) * kGroup;
    if (lane == 0) {
      srow[0] = s_out[0];
      srow[2] = s_out[1];
    } else if (lane == 16) {
      srow[1] = s_out[0];
      srow[3] = s_out[1];
    }
  }
}

cudaError_t launch_shared_basis_build(const __nv_bfloat16* k_cache, int64_t num_blocks, const int32_t* block_ids,
                                      int n_build, int H, const float* basis, int rho, uint8_t* records,
                                      uint32_t* status, cudaStream_t stream) {
  const int64_t warps = (int64_t)n_build * H;
  const int64_t grid = (warps + kSbBuildWarps - 1) / kSbBuildWarps;
  if (grid == 0) return cudaSuccess;
  shared_basis_build_kernel<<<(unsigned)grid, kSbBuildWarps * 32, 0, stream>>>(k_cache, num_blocks, block_ids, n_build,
                                                                         H, basis, rho, records, status);
  return cudaGetLastError();
}

cudaError_t launch_shared_basis_score(const __nv_bfloat16* q, const float* basis, int rho, const uint8_t* records,
                                      int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                                      int batch, int H, int max_pages, float* scores, uint32_t* status,
                                      cudaStream_t stream) {
  const dim3 grid((max_pages + kSbPagesPerCta - 1) / kSbPagesPerCta, batch * H);
  if (batch == 0) return cudaSuccess;
  shared_basis_score_kernel<<<grid, kSbWarps * 32, (size_t)kGroup * rho * sizeof(float), stream>>>(
      q, basis, rho, records, num_blocks, block_table, seq_lens, H, max_pages, scores, status);
  return cudaGetLastError();
}

}  // namespace locks
