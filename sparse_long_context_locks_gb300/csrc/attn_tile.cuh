// attn_tile.cuh -- one 16-token K/V page of decode attention for the 4 query
// heads of a GQA group, on tensor cores (shared by the split-K attention
// kernel and the fused select+attend cluster kernel).
//
// The page's K and V tiles sit in shared memory as two 64-column boxes each,
// 128-byte swizzled (the layout cp.async.bulk.tensor writes).  Per page:
//   S = K q^T    mma.sync m16n8k16 bf16 (16 tokens x 8 columns; column n is
//                query head n & 3), K fragments by ldmatrix;
//   online softmax per head in log2 units (running max and sum);
//   O^T += V^T P V fragments by ldmatrix.trans, P^T by movmatrix.
#pragma once

#include "common.cuh"

namespace locks {

constexpr int kTileBytes = kPage * kHeadDim * 2;   // 4096: one page-head of K (or V)
constexpr int kStageBytes = 2 * kTileBytes;        // K + V

// Swizzled (128B) address of 16-byte chunk `chunk` (0..15 across the 128
// columns) of row `row` of a K/V tile made of two 64-column boxes.
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int row, int chunk) {
  const int half = chunk >> 3, c = chunk & 7;
  return tile + half * 2048 + row * 128 + ((c ^ (row & 7)) << 4);
}

struct PageAttnState {
  float acc[8][4];   // O^T fragments: dims 16i + (gid | gid+8), columns 2t, 2t+1
  float m[2];        // running max (log2 units) of columns 2t, 2t+1
  float l[2];        // running sum (this lane's rows only until attn_finish)
};

__device__ __forceinline__ void attn_init(PageAttnState& st) {
#pragma unroll
  for (int i = 0; i < 8; ++i) st.acc[i][0] = st.acc[i][1] = st.acc[i][2] = st.acc[i][3] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
}

// B operand of S = K q^T from the group's first query row `q_group`
// (bf16 [4][128]); column n holds query head n & 3.
__device__ __forceinline__ void attn_load_q(uint32_t (&qb)[8][2], const __nv_bfloat16* q_group, int lane) {
  const __nv_bfloat16* qh = q_group + ((lane >> 2) & 3) * kHeadDim;
  const int t4 = lane & 3;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    qb[s][0] = *reinterpret_cast<const uint32_t*>(qh + 16 * s + 2 * t4);
    qb[s][1] = *reinterpret_cast<const uint32_t*>(qh + 16 * s + 2 * t4 + 8);
  }
}

// Issue the four 2 KB tensor copies of page-head (blk, h) into a stage, or
// complete the stage's phase at once when there is nothing to load.
__device__ __forceinline__ void attn_issue_page(const void* tmk, const void* tmv, uint8_t* dst, uint64_t* bar,
                                                int64_t blk, int H, int h) {
  if (blk >= 0) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    const int32_t y = (int32_t)((blk * H + h) * kPage);
    tma_load_2d(dst, tmk, 0, y, bar);
    tma_load_2d(dst + 2048, tmk, 64, y, bar);
    tma_load_2d(dst + kTileBytes, tmv, 0, y, bar);
    tma_load_2d(dst + kTileBytes + 2048, tmv, 64, y, bar);
  } else {
    mbar_arrive(bar);
  }
}

// Fold one page with `valid` leading tokens into the state.
__device__ __forceinline__ void attn_page(PageAttnState& st, uint32_t ktile, uint8_t* vtile_ptr, int valid,
                                          const uint32_t (&qb)[8][2], float scale_log2, int lane) {
  const int gid = lane >> 2;
  const uint32_t vtile = ktile + kTileBytes;
  if (valid < kPage) {
    // tail page: zero the V rows past the valid tokens (they may hold
    // anything, and 0 * NaN would poison the accumulator)
    for (int idx = lane; idx < (kPage - valid) * 16; idx += 32) {
      const int row = valid + idx / 16, chunk = idx % 16;
      const int half = chunk >> 3, c = chunk & 7;
      *reinterpret_cast<uint4*>(vtile_ptr + half * 2048 + row * 128 + ((c ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
  }
  // ---- S = K q^T (rows = tokens, cols = heads)
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lchk = lane >> 4;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t a[4];
    ldsm_x4(a, tile_addr(ktile, lrow, 2 * ks + lchk));
    mma_bf16(s, a[0], a[1], a[2], a[3], qb[ks][0], qb[ks][1]);
  }
  // scale into log2 units, mask invalid tokens
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] *= scale_log2;
  if (gid >= valid) s[0] = s[1] = -INFINITY;
  if (gid + 8 >= valid) s[2] = s[3] = -INFINITY;
  // ---- online softmax, per column (2t4, 2t4+1)
  float mt0 = fmaxf(s[0], s[2]), mt1 = fmaxf(s[1], s[3]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
    mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
  }
  const float mn0 = fmaxf(st.m[0], mt0), mn1 = fmaxf(st.m[1], mt1);
  const float al0 = fast_exp2(st.m[0] - mn0), al1 = fast_exp2(st.m[1] - mn1);
  st.m[0] = mn0;
  st.m[1] = mn1;
  const float p0 = fast_exp2(s[0] - mn0), p1 = fast_exp2(s[1] - mn1);
  const float p2 = fast_exp2(s[2] - mn0), p3 = fast_exp2(s[3] - mn1);
  st.l[0] = st.l[0] * al0 + p0 + p2;
  st.l[1] = st.l[1] * al1 + p1 + p3;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    st.acc[i][0] *= al0;
    st.acc[i][1] *= al1;
    st.acc[i][2] *= al0;
    st.acc[i][3] *= al1;
  }
  // P^T as the B operand (k = tokens, n = heads)
  const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1));
  const uint32_t pb1 = movmatrix_t(pack_bf16(p2, p3));
  // ---- O^T[dim][head] += V^T P
  const int vrow = (lane & 7) + (lane >> 4) * 8;
  const int vsel = (lane >> 3) & 1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t a[4];
    ldsm_x4_trans(a, tile_addr(vtile, vrow, 2 * i + vsel));
    mma_bf16(st.acc[i], a[0], a[1], a[2], a[3], pb0, pb1);
  }
}

// Sum l over the 8 token rows (lanes with equal t4).
__device__ __forceinline__ void attn_finish(PageAttnState& st) {
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], o);
  }
}

// Write a warp's state to shared memory: O[head][dim] (heads 0..3) and m, l.
__device__ __forceinline__ void attn_store_warp(const PageAttnState& st, float* wO, float* wM, float* wL, int lane) {
  const int gid = lane >> 2, t4 = lane & 3;
  if (t4 < 2) {   // columns 2t4, 2t4+1 are heads 0..3
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d0 = 16 * i + gid, d1 = d0 + 8;
      wO[(2 * t4) * kHeadDim + d0] = st.acc[i][0];
      wO[(2 * t4 + 1) * kHeadDim + d0] = st.acc[i][1];
      wO[(2 * t4) * kHeadDim + d1] = st.acc[i][2];
      wO[(2 * t4 + 1) * kHeadDim + d1] = st.acc[i][3];
    }
    if (gid == 0) {
      wM[2 * t4] = st.m[0];
      wM[2 * t4 + 1] = st.m[1];
      wL[2 * t4] = st.l[0];
      wL[2 * t4 + 1] = st.l[1];
    }
  }
}

}  // namespace locks
