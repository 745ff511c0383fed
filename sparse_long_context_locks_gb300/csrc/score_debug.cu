// score_debug.cu -- page scores from unquantised fp32 records (cfg quant = 0,
// rank r <= 16), the debug and reference configuration of the scorer.
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2, "Reconstruction and selection":
//   s_j(q) = log sum_i exp((q.mu_j + (V_j^T q).c_i) / sqrt(d)).
// With r = 16 the record reproduces the page's keys exactly (the centred keys
// have rank <= 15), so s_j is the exact page log-sum-exp of q.k / sqrt(d):
// the configuration that pins this arithmetic to a closed form.  Plain fp32
// on the CUDA cores, one warp per (request, KV head, page); it writes the same
// score table as the quantised scorer, so selection and attention run on it
// unchanged.

#include <cstdint>

#include "common.cuh"
#include "params.h"

namespace locks {

constexpr int kDebugScoreWarps = 8;

__global__ void __launch_bounds__(kDebugScoreWarps * 32) score_debug_kernel(const ScoreParams p, int rank_r) {
  __shared__ float u_s[kDebugScoreWarps][kGroup][16];
  __shared__ float qmu_s[kDebugScoreWarps][kGroup];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * kDebugScoreWarps + warp;
  const int64_t units = (int64_t)p.batch * p.H_kv;
  if (gw >= units * p.max_pages) return;
  const int unit = (int)(gw / p.max_pages), j = (int)(gw % p.max_pages);
  const int b = unit / p.H_kv, h = unit % p.H_kv;
  const int L = p.seq_lens[b];
  if (L < 0 || (L + kPage - 1) / kPage > p.max_pages) {
    if (j == 0 && h == 0 && lane == 0) flag_status(p.status, LOCKS_FLAG_BAD_SEQLEN);
    return;
  }
  if (j >= L / kPage) return;
  const int64_t blk = p.block_table[(int64_t)b * p.max_pages + j];
  if (blk < 0 || blk >= p.num_blocks) {
    if (lane == 0) flag_status(p.status, LOCKS_FLAG_BAD_BLOCK);
    return;
  }
  const size_t rec_bytes = 528 + 576 * (size_t)rank_r;
  const float* rec = reinterpret_cast<const float*>(p.summ + (blk * p.H_kv + h) * rec_bytes);
  const float* mu = rec;
  const float* V = rec + kHeadDim;             // [128][r]
  const float* C = V + kHeadDim * rank_r;      // [16][r]
  const __nv_bfloat16* qg = p.q + ((int64_t)b * p.H_kv * kGroup + (int64_t)h * kGroup) * kHeadDim;

  // q . mu per head: lane holds dims 4 lane .. 4 lane + 3
  float part[kGroup];
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc = fmaf(__bfloat162float(qg[g * kHeadDim + 4 * lane + e]), mu[4 * lane + e], acc);
    part[g] = acc;
  }
#pragma unroll
  for (int g = 0; g < kGroup; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part[g] += __shfl_xor_sync(0xffffffffu, part[g], o);
  }
  if (lane < kGroup) qmu_s[warp][lane] = part[lane == 0 ? 0 : lane == 1 ? 1 : lane == 2 ? 2 : 3];
  // u = V^T q: lane takes (head, direction) pairs lane and lane + 32
  for (int idx = lane; idx < kGroup * rank_r; idx += 32) {
    const int g = idx / rank_r, k = idx % rank_r;
    float acc = 0.f;
    for (int d = 0; d < kHeadDim; ++d) acc = fmaf(__bfloat162float(qg[g * kHeadDim + d]), V[d * rank_r + k], acc);
    u_s[warp][g][k] = acc;
  }
  __syncwarp();
  // logits: lane = token i (0..15) for heads (lane >> 4) and 2 + (lane >> 4)
  const int i = lane & 15;
  const float inv_sqrt_d = 0.08838834764831845f;
  float s_out[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int g = 2 * half + (lane >> 4);
    float dev = 0.f;
    for (int k = 0; k < rank_r; ++k) dev = fmaf(u_s[warp][g][k], C[i * rank_r + k], dev);
    const float x = (qmu_s[warp][g] + dev) * inv_sqrt_d;
    float m = x;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float e = expf(x - m);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
    s_out[half] = m + logf(e);
  }
  float* srow = p.scores + (((int64_t)b * p.H_kv + h) * p.max_pages + j) * kGroup;
  if (lane == 0) {
    srow[0] = s_out[0];
    srow[2] = s_out[1];
  } else if (lane == 16) {
    srow[1] = s_out[0];
    srow[3] = s_out[1];
  }
}

cudaError_t launch_score_debug(const ScoreParams& p, int rank_r, cudaStream_t stream) {
  const int64_t warps = (int64_t)p.batch * p.H_kv * p.max_pages;
  const int64_t grid = (warps + kDebugScoreWarps - 1) / kDebugScoreWarps;
  if (grid == 0) return cudaSuccess;
  score_debug_kernel<<<(unsigned)grid, kDebugScoreWarps * 32, 0, stream>>>(p, rank_r);
  return cudaGetLastError();
}

}  // namespace locks
