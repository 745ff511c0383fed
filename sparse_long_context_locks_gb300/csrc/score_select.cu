// score_select.cu -- LOCKS page scoring (a3) and group-shared top-k selection (a4, a5).
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2, "Reconstruction and selection":
//   s_j(q) = log sum_{i in P_j} exp((q.mu_j + (V_j^T q).c_i) / sqrt(d)),
// the log-sum-exp estimate of page j's attention mass from its resident
// summary; selection reads no candidate key or value.  §2 "Group-shared
// selection (GQA)": the per-head mass shares are averaged over the query
// heads of a KV group into one table that all heads attend by.
//
// score_kernel streams only the 784-byte records (one cp.async.bulk per page
// covering the CTA's KV heads, 4-stage mbarrier ring, one producer warp and 8
// consumer warps).  Per warp and group of 4 pages the arithmetic runs on the
// tensor cores as three small dense contractions:
//   u  = V^T q     m16n8k16 f16: rows = (2 pages x 8 directions), cols = the
//                  4 query heads (duplicated to 8), K = 128 dims; A comes
//                  straight from the int4 codes (one 16-byte load per lane);
//   q.mu           m16n8k16 f16: rows = the 4 pages' int8 centroids;
//   u . c_i        m16n8k16 f16, block-diagonal A = u of 4 pages x 4 heads
//                  (split hi + lo f16 for ~22-bit precision), B = int8 c;
// then a 4-lane shuffle log-sum-exp per (page, head).  Scores go to global
// memory together with per-(chunk, warp) partial log-sum-exps per head, which
// select_kernel combines into Z_{b,h,g} before ranking.

#include <cstdint>

#include "common.cuh"
#include "params.h"
#include "cluster_select.cuh"

namespace locks {


constexpr int kScoreConsumers = 8;
constexpr int kScoreThreads = (kScoreConsumers + 1) * 32;
constexpr int kScoreStages = 4;
constexpr int kScoreStageBytes = 32 * kRecord;  // 32 page-heads per stage
constexpr int kScoreSmem = kScoreStages * kScoreStageBytes + 128;

__device__ __forceinline__ int request_full_pages(const ScoreParams& p, int b) {
  const int L = p.seq_lens[b];
  if (L < 0 || (L + kPage - 1) / kPage > p.max_pages) {
    return -1;
  }
  return L / kPage;
}

// Scores of one group of 4 consecutive page slots for this warp's KV head.
// rec0: first slot's record in shared memory, stride: bytes between slots.
// Returns s for the lane's two rows: row gid = (page gid>>2, head gid&3) and
// row gid+8 = (page 2 + (gid>>2), head gid&3); identical on the 4 lanes of a
// row quad.
// bias_v / bias_mu: the constant parts the biased code conversions add to
// V^T q and q . mu for this lane's columns 2t and 2t+1 (removed by starting
// the accumulators at -bias).
__device__ __forceinline__ void score_group4(const uint8_t* rec0, int stride,
                                             const uint32_t (&qb)[8][2], float pow2e,
                                             const float (&bias_v)[2], const float (&bias_mu)[2],
                                             int lane, float& s_r0, float& s_r1) {
  const int gid = lane >> 2, t = lane & 3;
  const float inv_sqrt_d = 0.08838834764831845f;

  float4 sc[4];
#pragma unroll
  for (int P = 0; P < 4; ++P) sc[P] = *reinterpret_cast<const float4*>(rec0 + P * stride + 768);

  // ---- u = V^T q for page pairs (0,1) and (2,3)
  float d1[2][4];
#pragma unroll
  for (int pr = 0; pr < 2; ++pr) {
    float e1[4] = {0.f, 0.f, 0.f, 0.f};   // second chain: odd k-steps
    const uint4 va = *reinterpret_cast<const uint4*>(rec0 + (2 * pr) * stride + gid * 64 + t * 16);
    const uint4 vb = *reinterpret_cast<const uint4*>(rec0 + (2 * pr + 1) * stride + gid * 64 + t * 16);
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
    d1[pr][0] = d1[pr][2] = -bias_v[0];
    d1[pr][1] = d1[pr][3] = -bias_v[1];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
      nib8_to_h2x4_b72(wa[w], a04, a15, a26, a37);
      nib8_to_h2x4_b72(wb[w], b04, b15, b26, b37);
      mma_f16(d1[pr], a04, b04, a15, b15, qb[2 * w][0], qb[2 * w][1]);
      mma_f16(e1, a26, b26, a37, b37, qb[2 * w + 1][0], qb[2 * w + 1][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) d1[pr][i] += e1[i];
  }

  // ---- q . mu for the 4 pages (rows 0..3 of one m16 tile)
  float dmu[4] = {-bias_mu[0], -bias_mu[1], -bias_mu[0], -bias_mu[1]};
  {
    uint4 m0 = make_uint4(0, 0, 0, 0), m1 = make_uint4(0, 0, 0, 0);
    if (gid < 4) {
      const uint8_t* mp = rec0 + gid * stride + 512 + t * 32;
      m0 = *reinterpret_cast<const uint4*>(mp);
      m1 = *reinterpret_cast<const uint4*>(mp + 16);
    }
    const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t lo = 0, hi = 0;
      if (gid < 4) i8x4_to_h2x2_b1152(mw[s], lo, hi);
      mma_f16(dmu, lo, 0u, hi, 0u, qb[s][0], qb[s][1]);
    }
  }

  // ---- u -> f16 hi/lo, transposed into the block-diagonal A operand
  uint32_t th[4], tl[4];
#pragma unroll
  for (int pr = 0; pr < 2; ++pr) {
    const float f0 = sc[2 * pr].x * inv_sqrt_d;
    const float f1 = sc[2 * pr + 1].x * inv_sqrt_d;
    uint32_t h0, l0, h1, l1;
    split_h2(d1[pr][0] * f0, d1[pr][1] * f0, h0, l0);
    split_h2(d1[pr][2] * f1, d1[pr][3] * f1, h1, l1);
    th[2 * pr] = movmatrix_t(h0);
    tl[2 * pr] = movmatrix_t(l0);
    th[2 * pr + 1] = movmatrix_t(h1);
    tl[2 * pr + 1] = movmatrix_t(l1);
  }

  // ---- coefficients, B operand: (token gid | gid+8) x (directions 2t, 2t+1)
  uint32_t cb[4][2];
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(rec0 + P * stride + 640 + (gid * 4 + t) * 4);
    i8x4_to_h2x2(w, cb[P][0], cb[P][1]);
  }

  // ---- deviation logits: rows (page, head), cols tokens (2 n-tiles)
  const bool lowg = gid < 4;
  float d2[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) d2[nt][i] = 0.f;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const uint32_t* T = part == 0 ? th : tl;
      mma_f16(d2[nt], lowg ? T[0] : 0u, 0u, lowg ? 0u : T[1], 0u, cb[0][nt], cb[1][nt]);
      mma_f16(d2[nt], 0u, lowg ? T[2] : 0u, 0u, lowg ? 0u : T[3], cb[2][nt], cb[3][nt]);
    }
  }

  // ---- per-row log-sum-exp over the 16 tokens
  const int pr0 = gid >> 2;        // page of row gid   (0 or 1)
  const int pr1 = 2 + (gid >> 2);  // page of row gid+8 (2 or 3)
  const float sc_c0 = (pr0 == 0 ? sc[0].z : sc[1].z) * pow2e;
  const float sc_c1 = (pr1 == 2 ? sc[2].z : sc[3].z) * pow2e;
  float x0[4] = {d2[0][0] * sc_c0, d2[0][1] * sc_c0, d2[1][0] * sc_c0, d2[1][1] * sc_c0};
  float x1[4] = {d2[0][2] * sc_c1, d2[0][3] * sc_c1, d2[1][2] * sc_c1, d2[1][3] * sc_c1};
  float m0 = fmaxf(fmaxf(x0[0], x0[1]), fmaxf(x0[2], x0[3]));
  float m1 = fmaxf(fmaxf(x1[0], x1[1]), fmaxf(x1[2], x1[3]));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  float e0 = 0.f, e1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e0 += fast_exp2((x0[i] - m0) * kLog2e);
    e1 += fast_exp2((x1[i] - m1) * kLog2e);
  }
  e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
  e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
  e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
  e1 += __shfl_xor_sync(0xffffffffu, e1, 2);

  // ---- centroid term for the two rows, fetched from the mu tile's lanes
  const int hh = gid & 3;
  const int src0 = pr0 * 4 + (hh >> 1);
  const int src1 = pr1 * 4 + (hh >> 1);
  const float a0 = __shfl_sync(0xffffffffu, dmu[0], src0);
  const float a1 = __shfl_sync(0xffffffffu, dmu[1], src0);
  const float b0 = __shfl_sync(0xffffffffu, dmu[0], src1);
  const float b1 = __shfl_sync(0xffffffffu, dmu[1], src1);
  const float qmu0 = (hh & 1) ? a1 : a0;
  const float qmu1 = (hh & 1) ? b1 : b0;
  const float smu0 = (pr0 == 0 ? sc[0].y : sc[1].y);
  const float smu1 = (pr1 == 2 ? sc[2].y : sc[3].y);
  s_r0 = qmu0 * smu0 * pow2e * inv_sqrt_d + m0 + fast_log2(e0) * kLn2;
  s_r1 = qmu1 * smu1 * pow2e * inv_sqrt_d + m1 + fast_log2(e1) * kLn2;
}

__device__ __forceinline__ void lse_push(float& m, float& s, float x) {
  const float mn = fmaxf(m, x);
  s = s * fast_exp2((m - mn) * kLog2e) + fast_exp2((x - mn) * kLog2e);
  m = mn;
}


__global__ void __launch_bounds__(kScoreThreads, 2) score_kernel(const ScoreParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kScoreStages * kScoreStageBytes);
  uint64_t* empty = full + kScoreStages;
  uint32_t* live = reinterpret_cast<uint32_t*>(empty + kScoreStages);

  // a programmatic dependent (the fused select + attention pass) may start its
  // prologue as SMs free up; it waits for this grid's results before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kScoreStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kScoreConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // This CTA's contiguous range of work items (one stage = pps pages of one
  // (request, head group) unit each), split evenly over the grid.
  const int it_begin = (int)(((long long)blockIdx.x * p.n_items) / gridDim.x);
  const int it_end = (int)(((long long)(blockIdx.x + 1) * p.n_items) / gridDim.x);
  const int per_head_rec = p.h_cta * kRecord;
  const int first_unit = it_begin / p.n_chunks;

  if (warp == kScoreConsumers) {
    // ------------------------------------------------------------ producer
    // Walks the same stage sequence as the consumers; the block ids of the
    // next stage are loaded while the current stage's copies are issued.
    uint32_t step = 0;
    bool ok = true;
    int unit = first_unit, c = it_begin - first_unit * p.n_chunks;
    int it = it_begin;
    int b = 0, hg = 0, n = 0;
    auto enter_unit = [&]() {
      b = unit / p.head_groups;
      hg = unit % p.head_groups;
      n = max(request_full_pages(p, b), 0);
    };
    // advance (it, c, unit) to the next stage that holds pages, or it_end
    auto skip_empty = [&]() {
      while (it < it_end && c * p.pps >= n) {
        const int unit_end = (unit + 1) * p.n_chunks;
        it = unit_end;
        c = 0;
        ++unit;
        if (it < it_end) enter_unit();
      }
    };
    if (it < it_end) enter_unit();
    skip_empty();
    int64_t blk = -1;
    if (it < it_end && lane < p.pps && c * p.pps + lane < n)
      blk = p.block_table[(int64_t)b * p.max_pages + c * p.pps + lane];
    while (it < it_end && ok) {
      const int s = step % kScoreStages;
      if (step >= kScoreStages) ok = mbar_wait(&empty[s], ((step / kScoreStages) - 1) & 1, p.status);
      if (!ok) break;
      bool is_live = lane < p.pps && c * p.pps + lane < n;
      if (is_live && (blk < 0 || blk >= p.num_blocks)) {
        flag_status(p.status, LOCKS_FLAG_BAD_BLOCK);
        is_live = false;
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, is_live);
      if (lane == 0) {
        live[s] = mask;
        mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(mask) * (uint32_t)per_head_rec);
      }
      __syncwarp();
      if (is_live) {
        const uint8_t* src = p.summ + ((int64_t)blk * p.H_kv + (int64_t)hg * p.h_cta) * kRecord;
        bulk_g2s(stages + s * kScoreStageBytes + lane * per_head_rec, src, per_head_rec, &full[s]);
      }
      ++step;
      ++it;
      ++c;
      if (c == p.n_chunks) {
        c = 0;
        ++unit;
        if (it < it_end) enter_unit();
      }
      skip_empty();
      blk = -1;
      if (it < it_end && lane < p.pps && c * p.pps + lane < n)
        blk = p.block_table[(int64_t)b * p.max_pages + c * p.pps + lane];
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int hl = warp / p.wph, sub = warp % p.wph;
  const int gid = lane >> 2, t = lane & 3;
  uint32_t step = 0;
  int cur_b = -1, cur_h = -1;
  uint32_t qb[8][2];
  float pow2e = 1.f;
  float bias_v[2] = {0.f, 0.f}, bias_mu[2] = {0.f, 0.f};
  bool ok = true;

  int it = it_begin;
  for (int unit = first_unit; it < it_end; ++unit) {
    // one segment: this unit's items inside the range
    const int unit_end = min(it_end, (unit + 1) * p.n_chunks);
    const int b = unit / p.head_groups, hg = unit % p.head_groups;
    const int h = hg * p.h_cta + hl;
    const int nraw = request_full_pages(p, b);
    if (nraw < 0 && lane == 0 && warp == 0) flag_status(p.status, LOCKS_FLAG_BAD_SEQLEN);
    const int n = max(nraw, 0);
    const int c0 = it - unit * p.n_chunks;
    const int pg_begin = c0 * p.pps;
    const int pg_end = min((unit_end - unit * p.n_chunks) * p.pps, n);

    if (pg_begin < pg_end && (b != cur_b || h != cur_h)) {
      // B operand = the group's 4 query heads (duplicated into columns 4..7),
      // pre-scaled by an exact power of two so every value fits f16.
      cur_b = b;
      cur_h = h;
      const __nv_bfloat16* qh = p.q + ((int64_t)b * p.H_kv * kGroup + (int64_t)h * kGroup + (gid & 3)) * kHeadDim;
      float qv[8][4];
      float amax = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(qh + 16 * s + 2 * t);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(qh + 16 * s + 2 * t + 8);
        qv[s][0] = __low2float(lo);
        qv[s][1] = __high2float(lo);
        qv[s][2] = __low2float(hi);
        qv[s][3] = __high2float(hi);
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(qv[s][i]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int ex = 0;
      frexpf(amax, &ex);
      const int e = ex > 15 ? ex - 15 : 0;
      pow2e = ldexpf(1.f, e);
      const float inv = ldexpf(1.f, -e);
      float qsum = 0.f;   // sum of this lane's f16 operand values of column gid
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const __half2 lo = __floats2half2_rn(qv[s][0] * inv, qv[s][1] * inv);
        const __half2 hi = __floats2half2_rn(qv[s][2] * inv, qv[s][3] * inv);
        qb[s][0] = *reinterpret_cast<const uint32_t*>(&lo);
        qb[s][1] = *reinterpret_cast<const uint32_t*>(&hi);
        const float2 lf = __half22float2(lo), hf = __half22float2(hi);
        qsum += (lf.x + lf.y) + (hf.x + hf.y);
      }
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);   // column gid's sum over all 128 dims
      // this lane's accumulator columns are 2t and 2t+1: their sums live on
      // the lanes with gid == 2t and gid == 2t+1
      const float q0 = __shfl_sync(0xffffffffu, qsum, (2 * t) * 4);
      const float q1 = __shfl_sync(0xffffffffu, qsum, (2 * t + 1) * 4);
      bias_v[0] = 72.f * q0;
      bias_v[1] = 72.f * q1;
      bias_mu[0] = 1152.f * q0;
      bias_mu[1] = 1152.f * q1;
    }

    float run_m = -INFINITY, run_s = 0.f;   // this lane's head (gid & 3), t == 0 lanes count
    float* srow = p.scores + (((int64_t)b * p.H_kv + h) * p.max_pages) * kGroup + (gid & 3);
    for (int pg = pg_begin; pg < pg_end; pg += p.pps, ++step) {
      const int s = step % kScoreStages;
      if (ok) ok = mbar_wait(&full[s], (step / kScoreStages) & 1, p.status);
      if (ok) {
        const uint32_t mask = live[s];
        const uint8_t* rec0 = stages + s * kScoreStageBytes + (sub * 4) * per_head_rec + hl * kRecord;
        float s_r0, s_r1;
        score_group4(rec0, per_head_rec, qb, pow2e, bias_v, bias_mu, lane, s_r0, s_r1);
        const int slot0 = sub * 4 + (gid >> 2), slot1 = sub * 4 + 2 + (gid >> 2);
        const bool v0 = (mask >> slot0) & 1u, v1 = (mask >> slot1) & 1u;
        if (t == 0) {
          if (v0) {
            srow[(int64_t)(pg + slot0) * kGroup] = s_r0;
            lse_push(run_m, run_s, s_r0);
          }
          if (v1) {
            srow[(int64_t)(pg + slot1) * kGroup] = s_r1;
            lse_push(run_m, run_s, s_r1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    it = unit_end;

    // partial log-sum-exp of this warp's pages of the segment, per query head
    // g = gid & 3: rows gid and gid ^ 4 hold the same head -> lanes l, l ^ 16.
    const float om = __shfl_xor_sync(0xffffffffu, run_m, 16);
    const float os = __shfl_xor_sync(0xffffffffu, run_s, 16);
    lse_merge(run_m, run_s, om, os);
    if (t == 0 && gid < 4) {
      // slot: this CTA's index among the CTAs covering the unit
      const int slot = (int)blockIdx.x - score_cta_of((long long)unit * p.n_chunks, p.n_items, gridDim.x);
      float* part = p.partials +
                    ((((int64_t)unit * p.seg_slots + slot) * kScoreConsumers + warp) * kGroup + gid) * 2;
      part[0] = run_m;
      part[1] = run_s;
    }
  }
}

// ---------------------------------------------------------------- select


__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads)
    select_kernel(const SelectParams p) {
  // [slice keys][cand keys][cand pages][cand blocks][selected list]
  extern __shared__ __align__(16) uint32_t sel_dyn[];
  const int slice_cap = (p.max_pages + kSelCluster - 1) / kSelCluster;
  const int stride = sel_cand_stride(p.max_pages, p.budget, select_fixed_bytes(p.max_pages, p.budget));
  SelScratch sc;
  sc.keys_s = sel_dyn;
  sc.bt_slice = nullptr;
  sc.cand_key = sel_dyn + slice_cap;
  sc.cand_page = reinterpret_cast<int*>(sc.cand_key + kSelCluster * stride);
  sc.cand_blk = sc.cand_page + kSelCluster * stride;
  sc.cand_stride = stride;
  sc.out_blk = sc.cand_blk + kSelCluster * stride;
  cluster_select(p, sc);
}

}  // namespace locks

// ---------------------------------------------------------------- launchers
namespace locks {

cudaError_t launch_score(const ScoreParams& p, int grid, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  score_kernel<<<grid, kScoreThreads, kScoreSmem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectParams& p, int units, cudaStream_t stream) {
  const size_t dyn = select_smem_bytes(p.max_pages, p.budget);
  static size_t attr_bytes = 0;
  if (dyn > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    attr_bytes = dyn;
  }
  dim3 grid(kSelCluster, units);
  select_kernel<<<grid, kSelThreads, dyn, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace locks
