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
//                  from the int4 codes (one 16-byte load per lane), each
//                  converted to its exact f16 value;
//   q.mu           m16n8k16 f16 over K = 64: rows 0..3 = the 4 pages' int8
//                  centroid dims 0..63 against columns 0..3 (the heads' dims
//                  0..63), rows 4..7 = dims 64..127 against columns 4..7;
//   u . c_i        m16n8k16 f16, block-diagonal A = u of 4 pages x 4 heads
//                  (split hi + lo f16 for ~22-bit precision), B = int8 c;
// then a 4-lane shuffle log-sum-exp per (page, head), without a max shift
// unless a row's sum leaves [2^-100, 2^100].  Scores go to global
// memory; the selection reads them back to form Z_{b,h,g} and rank the pages.

#include <cstdint>
#include <mutex>

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
// rec0: first slot's record in shared memory; kStride: bytes between slots.
// Returns s for the lane's two rows: row gid = (page gid>>2, head gid&3) and
// row gid+8 = (page 2 + (gid>>2), head gid&3); identical on the 4 lanes of a
// row quad.
// qb: B operand (the group's 4 query heads, columns duplicated to 8), scaled
// by 2^-e; qmb: the centroid's B operand (columns 0..3 dims 0..63, columns
// 4..7 dims 64..127 of the same heads).  Codes enter the tensor cores as
// their exact f16 values.
template <int kStride>
__device__ __forceinline__ void score_group4(const uint8_t* rec0, const uint32_t (&qb)[8][2],
                                             const uint32_t (&qmb)[4][2], float pow2e, int lane,
                                             float& s_r0, float& s_r1) {
  const int gid = lane >> 2, t = lane & 3;
  const float inv_sqrt_d = 0.08838834764831845f;

  // ---- u = V^T q for page pairs (0,1) and (2,3): two interleaved chains
  float d1[2][4];
  uint4 v[2][2];
#pragma unroll
  for (int pr = 0; pr < 2; ++pr) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      v[pr][j] = *reinterpret_cast<const uint4*>(rec0 + (2 * pr + j) * kStride + gid * 64 + t * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) d1[pr][i] = 0.f;
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const uint32_t wa = w == 0 ? v[pr][0].x : w == 1 ? v[pr][0].y : w == 2 ? v[pr][0].z : v[pr][0].w;
      const uint32_t wb = w == 0 ? v[pr][1].x : w == 1 ? v[pr][1].y : w == 2 ? v[pr][1].z : v[pr][1].w;
      uint32_t a04, a15, a26, a37, b04, b15, b26, b37;
      nib8_to_h2x4(wa, a04, a15, a26, a37);
      nib8_to_h2x4(wb, b04, b15, b26, b37);
      mma_f16(d1[pr], a04, b04, a15, b15, qb[2 * w][0], qb[2 * w][1]);
      mma_f16(d1[pr], a26, b26, a37, b37, qb[2 * w + 1][0], qb[2 * w + 1][1]);
    }
  }

  // ---- q . mu for the 4 pages in two halves of K: rows 0..3 hold the
  // pages' centroid dims 0..63 against B columns 0..3 (dims 0..63 of the 4
  // heads), rows 4..7 dims 64..127 against columns 4..7 (dims 64..127);
  // cross terms are never read, rows 8..15 are zero.  Row p, column h plus
  // row 4 + p, column 4 + h is q_h . mu_p: lane 4p + t adds lane 4p + t ^ 18.
  float dmu[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint4 mq = *reinterpret_cast<const uint4*>(rec0 + (gid & 3) * kStride + 512 + t * 32 + (gid & 4) * 4);
    const uint32_t mw[4] = {mq.x, mq.y, mq.z, mq.w};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t lo, hi;
      i8x4_to_h2x2(mw[s], lo, hi);
      mma_f16(dmu, lo, 0u, hi, 0u, qmb[s][0], qmb[s][1]);
    }
    dmu[0] += __shfl_xor_sync(0xffffffffu, dmu[0], 18);
    dmu[1] += __shfl_xor_sync(0xffffffffu, dmu[1], 18);
  }

  // ---- u -> f16 hi/lo, transposed into the block-diagonal A operand.  The
  // scalar steps from here on use explicitly rounded operations, so that the
  // compiler cannot fuse a multiply into a later add for one page pair and not
  // for the other: identical records then score bit-identically in any slot.
  uint32_t th[4], tl[4];
#pragma unroll
  for (int pr = 0; pr < 2; ++pr) {
    const float f0 = *reinterpret_cast<const float*>(rec0 + (2 * pr) * kStride + 768) * inv_sqrt_d;
    const float f1 = *reinterpret_cast<const float*>(rec0 + (2 * pr + 1) * kStride + 768) * inv_sqrt_d;
    uint32_t h0, l0, h1, l1;
    split_h2(__fmul_rn(d1[pr][0], f0), __fmul_rn(d1[pr][1], f0), h0, l0);
    split_h2(__fmul_rn(d1[pr][2], f1), __fmul_rn(d1[pr][3], f1), h1, l1);
    th[2 * pr] = movmatrix_t(h0);
    tl[2 * pr] = movmatrix_t(l0);
    th[2 * pr + 1] = movmatrix_t(h1);
    tl[2 * pr + 1] = movmatrix_t(l1);
  }

  // ---- coefficients, B operand: (token gid | gid+8) x (directions 2t, 2t+1)
  uint32_t cb[4][2];
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(rec0 + P * kStride + 640 + (gid * 4 + t) * 4);
    i8x4_to_h2x2(w, cb[P][0], cb[P][1]);
  }

  // ---- deviation logits: rows (page, head), cols tokens (2 n-tiles)
  const bool lowg = gid < 4;
  uint32_t ah[4], al[4];   // block-diagonal A: this lane's nonzero slot per mma
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    ah[2 * i] = lowg ? th[2 * i] : 0u;
    ah[2 * i + 1] = lowg ? 0u : th[2 * i + 1];
    al[2 * i] = lowg ? tl[2 * i] : 0u;
    al[2 * i + 1] = lowg ? 0u : tl[2 * i + 1];
  }
  float d2[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) d2[nt][i] = 0.f;
    mma_f16(d2[nt], ah[0], 0u, ah[1], 0u, cb[0][nt], cb[1][nt]);
    mma_f16(d2[nt], 0u, ah[2], 0u, ah[3], cb[2][nt], cb[3][nt]);
    mma_f16(d2[nt], al[0], 0u, al[1], 0u, cb[0][nt], cb[1][nt]);
    mma_f16(d2[nt], 0u, al[2], 0u, al[3], cb[2][nt], cb[3][nt]);
  }

  // ---- per-row log-sum-exp over the 16 tokens, in log2 units
  const int pr0 = gid >> 2;        // page of row gid   (0 or 1)
  const int pr1 = 2 + (gid >> 2);  // page of row gid+8 (2 or 3)
  // s_mu, s_c of the rows' pages (record bytes 772 and 776)
  const float smu0 = *reinterpret_cast<const float*>(rec0 + pr0 * kStride + 772);
  const float smu1 = *reinterpret_cast<const float*>(rec0 + pr1 * kStride + 772);
  const float sc_c0 = *reinterpret_cast<const float*>(rec0 + pr0 * kStride + 776) * (pow2e * kLog2e);
  const float sc_c1 = *reinterpret_cast<const float*>(rec0 + pr1 * kStride + 776) * (pow2e * kLog2e);
  float x0[4] = {__fmul_rn(d2[0][0], sc_c0), __fmul_rn(d2[0][1], sc_c0), __fmul_rn(d2[1][0], sc_c0),
                 __fmul_rn(d2[1][1], sc_c0)};
  float x1[4] = {__fmul_rn(d2[0][2], sc_c1), __fmul_rn(d2[0][3], sc_c1), __fmul_rn(d2[1][2], sc_c1),
                 __fmul_rn(d2[1][3], sc_c1)};
  // The sums of 2^x are taken without a max shift while they stay inside
  // [2^-100, 2^100], where every term above 2^-126 is a normal float and the
  // terms flushed to zero change the sum by less than 2^-22 of itself; a row
  // (page, head) whose sum leaves that range is redone with its max taken
  // out.  The choice is the row's own (all four lanes of a row quad hold the
  // same sum), so a page's score never depends on the other pages of its
  // group, or on stale slots past a unit's last page.
  float m0 = 0.f, m1 = 0.f;
  float e0 = 0.f, e1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e0 += fast_exp2(x0[i]);
    e1 += fast_exp2(x1[i]);
  }
  e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
  e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
  e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
  e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
  const bool in0 = e0 >= 0x1p-100f && e0 <= 0x1p100f;
  const bool in1 = e1 >= 0x1p-100f && e1 <= 0x1p100f;
  if (!__all_sync(0xffffffffu, in0 && in1)) {   // shuffles below need the whole warp
    float n0 = fmaxf(fmaxf(x0[0], x0[1]), fmaxf(x0[2], x0[3]));
    float n1 = fmaxf(fmaxf(x1[0], x1[1]), fmaxf(x1[2], x1[3]));
    n0 = fmaxf(n0, __shfl_xor_sync(0xffffffffu, n0, 1));
    n1 = fmaxf(n1, __shfl_xor_sync(0xffffffffu, n1, 1));
    n0 = fmaxf(n0, __shfl_xor_sync(0xffffffffu, n0, 2));
    n1 = fmaxf(n1, __shfl_xor_sync(0xffffffffu, n1, 2));
    float f0 = 0.f, f1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f0 += fast_exp2(__fsub_rn(x0[i], n0));
      f1 += fast_exp2(__fsub_rn(x1[i], n1));
    }
    f0 += __shfl_xor_sync(0xffffffffu, f0, 1);
    f1 += __shfl_xor_sync(0xffffffffu, f1, 1);
    f0 += __shfl_xor_sync(0xffffffffu, f0, 2);
    f1 += __shfl_xor_sync(0xffffffffu, f1, 2);
    if (!in0) {
      m0 = n0;
      e0 = f0;
    }
    if (!in1) {
      m1 = n1;
      e1 = f1;
    }
  }

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
  const float cq = pow2e * inv_sqrt_d;
  s_r0 = __fadd_rn(__fmul_rn(__fmul_rn(qmu0, smu0), cq), __fmul_rn(__fadd_rn(m0, fast_log2(e0)), kLn2));
  s_r1 = __fadd_rn(__fmul_rn(__fmul_rn(qmu1, smu1), cq), __fmul_rn(__fadd_rn(m1, fast_log2(e1)), kLn2));
}

// kHcta: KV heads per CTA (1, 2, 4 or 8); a stage holds kPps pages of kHcta
// heads each (32 records), warp w scores head w / kWph, pages 4 (w % kWph) ...
// Two CTAs an SM: 18 warps put 5 on some SM sub-partition, whose 16,384
// registers then allow at most 96 a thread; one register more halves the
// occupancy.
template <int kHcta>
__global__ void __launch_bounds__(kScoreThreads, 2) score_kernel(const ScoreParams p) {
  constexpr int kWph = 8 / kHcta;
  constexpr int kPps = 4 * kWph;
  constexpr int per_head_rec = kHcta * kRecord;
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
  // (request, head group) unit; unit u owns items [u n_chunks, (u + 1)
  // n_chunks)), split evenly over the grid.  With one unit the split is over
  // all of them (at most one past its full pages).  With several, requests of
  // different lengths leave different numbers of items empty, so warp 0
  // counts each unit's items that hold full pages (from the sequence
  // lengths), splits that count evenly, and maps the CTA's share back to item
  // indices; the loops below skip the empty items in between.
  int it_begin = (int)(((long long)blockIdx.x * p.n_items) / gridDim.x);
  int it_end = (int)(((long long)(blockIdx.x + 1) * p.n_items) / gridDim.x);
  const int n_units = p.batch * p.head_groups;
  if (n_units > 1) {
    __shared__ int s_range[2];
    if (warp == 0) {
      auto items_of = [&](int u) -> int {   // items of unit u holding full pages
        if (u >= n_units) return 0;
        const int nf = request_full_pages(p, u / p.head_groups);
        if (nf < 0 && blockIdx.x == 0 && u % p.head_groups == 0) flag_status(p.status, LOCKS_FLAG_BAD_SEQLEN);
        return (max(nf, 0) + kPps - 1) / kPps;
      };
      long long total = 0;
      for (int base = 0; base < n_units; base += 32) {
        int v = items_of(base + lane);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        total += v;
      }
      const long long x0 = (long long)blockIdx.x * total / gridDim.x;
      const long long x1 = (long long)(blockIdx.x + 1) * total / gridDim.x;
      // item index of compact position x: unit u with prefix <= x < prefix + count
      int r0 = p.n_items, r1 = p.n_items;
      long long prefix = 0;
      for (int base = 0; base < n_units && (r0 == p.n_items || r1 == p.n_items); base += 32) {
        const int v = items_of(base + lane);
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const long long lo = prefix + incl - v, hi = prefix + incl;   // this lane's unit: [lo, hi)
        const uint32_t in0 = __ballot_sync(0xffffffffu, v > 0 && x0 >= lo && x0 < hi);
        const uint32_t in1 = __ballot_sync(0xffffffffu, v > 0 && x1 >= lo && x1 < hi);
        if (in0 && r0 == p.n_items) {
          const int l = __ffs(in0) - 1;
          const long long lo_l = __shfl_sync(0xffffffffu, lo, l);
          r0 = (base + l) * p.n_chunks + (int)(x0 - lo_l);
        }
        if (in1 && r1 == p.n_items) {
          const int l = __ffs(in1) - 1;
          const long long lo_l = __shfl_sync(0xffffffffu, lo, l);
          r1 = (base + l) * p.n_chunks + (int)(x1 - lo_l);
        }
        prefix += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        s_range[0] = r0;
        s_range[1] = r1;
      }
    }
    __syncthreads();
    it_begin = s_range[0];
    it_end = s_range[1];
  }
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
    int cross_pg = -1;   // the page the request's current token completed (deferred)
    bool waited = false;
    auto enter_unit = [&]() {
      b = unit / p.head_groups;
      hg = unit % p.head_groups;
      n = max(request_full_pages(p, b), 0);
      cross_pg = (p.defer_crossing && n > 0 && p.seq_lens[b] % kPage == 0) ? n - 1 : -1;
    };
    // advance (it, c, unit) to the next stage that holds pages, or it_end
    auto skip_empty = [&]() {
      while (it < it_end && c * kPps >= n) {
        const int unit_end = (unit + 1) * p.n_chunks;
        it = unit_end;
        c = 0;
        ++unit;
        if (it < it_end) enter_unit();
      }
    };
    int64_t blk = -1;
    if (it < it_end) {
      // the first stage's block ids are fetched alongside the sequence length
      const int pg0 = c * kPps + lane;
      if (lane < kPps && pg0 < p.max_pages)
        blk = p.block_table[(int64_t)(first_unit / p.head_groups) * p.max_pages + pg0];
      enter_unit();
    }
    const int it0 = it;
    skip_empty();
    if (it != it0 || !(lane < kPps && c * kPps + lane < n)) {
      blk = -1;
      if (it < it_end && lane < kPps && c * kPps + lane < n)
        blk = p.block_table[(int64_t)b * p.max_pages + c * kPps + lane];
    }
    while (it < it_end && ok) {
      const int s = step % kScoreStages;
      if (step >= kScoreStages) ok = mbar_wait(&empty[s], ((step / kScoreStages) - 1) & 1, p.status);
      if (!ok) break;
      bool is_live = lane < kPps && c * kPps + lane < n;
      if (is_live && (blk < 0 || blk >= p.num_blocks)) {
        flag_status(p.status, LOCKS_FLAG_BAD_BLOCK);
        is_live = false;
      }
      // the crossing build's page: its record exists once that grid has ended
      if (!waited && __any_sync(0xffffffffu, is_live && c * kPps + lane == cross_pg)) {
        griddep_wait();
        waited = true;
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, is_live);
      if (lane == 0) {
        live[s] = mask;
        mbar_arrive_expect_tx(&full[s], (uint32_t)__popc(mask) * (uint32_t)per_head_rec);
      }
      __syncwarp();
      if (is_live) {
        const uint8_t* src = p.summ + ((int64_t)blk * p.H_kv + (int64_t)hg * kHcta) * kRecord;
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
      if (it < it_end && lane < kPps && c * kPps + lane < n)
        blk = p.block_table[(int64_t)b * p.max_pages + c * kPps + lane];
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int hl = warp / kWph, sub = warp % kWph;
  const int gid = lane >> 2, t = lane & 3;
  uint32_t step = 0;
  int cur_b = -1, cur_h = -1;
  uint32_t qb[8][2];
  uint32_t qmb[4][2];   // centroid B operand: columns 0..3 dims 0..63, columns 4..7 dims 64..127
  float pow2e = 1.f;
  bool ok = true;

  int it = it_begin;
  for (int unit = first_unit; it < it_end; ++unit) {
    // one segment: this unit's items inside the range
    const int unit_end = min(it_end, (unit + 1) * p.n_chunks);
    const int b = unit / p.head_groups, hg = unit % p.head_groups;
    const int h = hg * kHcta + hl;
    const int nraw = request_full_pages(p, b);
    if (nraw < 0 && lane == 0 && warp == 0) flag_status(p.status, LOCKS_FLAG_BAD_SEQLEN);
    const int n = max(nraw, 0);
    const int c0 = it - unit * p.n_chunks;
    const int pg_begin = c0 * kPps;
    const int pg_end = min((unit_end - unit * p.n_chunks) * kPps, n);

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
      const int e = ex > 15 ? ex - 15 : 0;   // amax 2^-e < 2^15
      pow2e = ldexpf(1.f, e);
      const float inv = ldexpf(1.f, -e);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const __half2 lo = __floats2half2_rn(qv[s][0] * inv, qv[s][1] * inv);
        const __half2 hi = __floats2half2_rn(qv[s][2] * inv, qv[s][3] * inv);
        qb[s][0] = *reinterpret_cast<const uint32_t*>(&lo);
        qb[s][1] = *reinterpret_cast<const uint32_t*>(&hi);
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        qmb[s][0] = gid < 4 ? qb[s][0] : qb[s + 4][0];
        qmb[s][1] = gid < 4 ? qb[s][1] : qb[s + 4][1];
      }
    }

    float* srow = p.scores + (((int64_t)b * p.H_kv + h) * p.max_pages) * kGroup + (gid & 3);
    for (int pg = pg_begin; pg < pg_end; pg += kPps, ++step) {
      const int s = step % kScoreStages;
      if (ok) ok = mbar_wait(&full[s], (step / kScoreStages) & 1, p.status);
      if (ok) {
        const uint32_t mask = live[s];
        const uint8_t* rec0 = stages + s * kScoreStageBytes + (sub * 4) * per_head_rec + hl * kRecord;
        float s_r0, s_r1;
        score_group4<per_head_rec>(rec0, qb, qmb, pow2e, lane, s_r0, s_r1);
        const int slot0 = sub * 4 + (gid >> 2), slot1 = sub * 4 + 2 + (gid >> 2);
        const bool v0 = (mask >> slot0) & 1u, v1 = (mask >> slot1) & 1u;
        if (t == 0) {
          if (v0) srow[(int64_t)(pg + slot0) * kGroup] = s_r0;
          if (v1) srow[(int64_t)(pg + slot1) * kGroup] = s_r1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    it = unit_end;
  }
}

// ---------------------------------------------------------------- select


// One cluster of C CTAs per (request, KV head).
// kStaged: each CTA first copies its slice of scores to shared memory.
// kExtZ: Z_g comes from per-shard (max, sum) pairs (context-parallel shards).
template <int C, bool kStaged, bool kExtZ>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(kSelThreads, C > 8 ? 2 : 4) select_kernel(const SelectParams p) {
  // launched as a programmatic dependent of the scoring pass, and the split-K
  // attention as one of this kernel
  griddep_launch_dependents();
  griddep_wait();
  // [slice keys][selected list][slice scores, when staged]
  extern __shared__ __align__(16) uint32_t sel_dyn[];
  const int slice_cap = (p.max_pages + C - 1) / C;
  SelScratch sc;
  sc.keys_s = sel_dyn;
  sc.bt_slice = nullptr;
  sc.out_blk = reinterpret_cast<int*>(sel_dyn + slice_cap);
  sc.stage = kStaged ? reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(sel_dyn) +
                                                 select_stage_offset(p.max_pages, p.budget, C))
                     : nullptr;
  cluster_select<C, kStaged, kExtZ>(p, sc);
}

}  // namespace locks

// ---------------------------------------------------------------- launchers
namespace locks {

template <int kHcta>
cudaError_t launch_score_t(const ScoreParams& p, int grid, cudaStream_t stream, bool programmatic) {
  static DynSmemAttr smem_attr;
  const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(score_kernel<kHcta>), kScoreSmem, smem_attr);
  if (e != cudaSuccess) return e;
  if (!programmatic) {
    score_kernel<kHcta><<<grid, kScoreThreads, kScoreSmem, stream>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kScoreThreads, 1, 1);
  cfg.dynamicSmemBytes = kScoreSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t el = cudaLaunchKernelEx(&cfg, score_kernel<kHcta>, p);
  if (el != cudaSuccess) return el;
  return cudaGetLastError();
}

cudaError_t launch_score(const ScoreParams& p, int grid, cudaStream_t stream, bool programmatic) {
  switch (p.h_cta) {
    case 8: return launch_score_t<8>(p, grid, stream, programmatic);
    case 4: return launch_score_t<4>(p, grid, stream, programmatic);
    case 2: return launch_score_t<2>(p, grid, stream, programmatic);
    case 1: return launch_score_t<1>(p, grid, stream, programmatic);
    default: return cudaErrorInvalidValue;
  }
}

template <int C, bool kStaged, bool kExtZ = false>
cudaError_t launch_select_c(const SelectParams& p, int units, cudaStream_t stream) {
  const size_t dyn = select_smem_bytes(p.max_pages, p.budget, C, kStaged);
  static DynSmemAttr smem_attr;
  const cudaError_t e =
      ensure_dyn_smem(reinterpret_cast<const void*>(select_kernel<C, kStaged, kExtZ>), dyn, smem_attr);
  if (e != cudaSuccess) return e;
  if (C > 8) {   // a non-portable cluster size
    const cudaError_t en = cudaFuncSetAttribute(reinterpret_cast<const void*>(select_kernel<C, kStaged, kExtZ>),
                                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (en != cudaSuccess) return en;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, units, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t el = cudaLaunchKernelEx(&cfg, select_kernel<C, kStaged, kExtZ>, p);
  if (el != cudaSuccess) return el;
  return cudaGetLastError();
}

// How many 16-CTA clusters of the selection kernel can be resident at once
// with this dynamic shared memory (0 when the size is refused); cached per
// device and size.
int select16_max_clusters(size_t dyn, bool staged) {
  struct Entry {
    int dev;
    size_t dyn;
    bool staged;
    int n;
  };
  static Entry cache[16];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].dyn == dyn && cache[i].staged == staged) return cache[i].n;
  const void* fn = staged ? reinterpret_cast<const void*>(select_kernel<16, true, false>)
                          : reinterpret_cast<const void*>(select_kernel<16, false, false>);
  int n = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(kSelThreads, 1, 1);
    cfg.dynamicSmemBytes = dyn;
    int clusters = 0;
    const cudaError_t e = staged ? cudaOccupancyMaxActiveClusters(&clusters, select_kernel<16, true, false>, &cfg)
                                 : cudaOccupancyMaxActiveClusters(&clusters, select_kernel<16, false, false>, &cfg);
    if (e == cudaSuccess) n = clusters;
  }
  cudaGetLastError();   // a refused query leaves no sticky error
  if (used < 16) cache[used++] = Entry{dev, dyn, staged, n};
  return n;
}

cudaError_t launch_select(const SelectParams& p, int units, int cluster, cudaStream_t stream) {
  const bool staged = p.stage_scores != 0;
  if (p.zpairs != nullptr) {   // context-parallel shard: Z_g given, scores read from L2
    switch (cluster) {
      case 16: return launch_select_c<16, false, true>(p, units, stream);
      case 8: return launch_select_c<8, false, true>(p, units, stream);
      case 4: return launch_select_c<4, false, true>(p, units, stream);
      case 2: return launch_select_c<2, false, true>(p, units, stream);
      case 1: return launch_select_c<1, false, true>(p, units, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (cluster) {
    case 16: return staged ? launch_select_c<16, true>(p, units, stream) : launch_select_c<16, false>(p, units, stream);
    case 8: return staged ? launch_select_c<8, true>(p, units, stream) : launch_select_c<8, false>(p, units, stream);
    case 4: return staged ? launch_select_c<4, true>(p, units, stream) : launch_select_c<4, false>(p, units, stream);
    case 2: return staged ? launch_select_c<2, true>(p, units, stream) : launch_select_c<2, false>(p, units, stream);
    case 1: return staged ? launch_select_c<1, true>(p, units, stream) : launch_select_c<1, false>(p, units, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace locks
