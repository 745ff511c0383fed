// build_summaries.cu -- LOCKS page summary builder (a1) with quantisation (a2).
//
// "LOCKS: Page-Local Compact Key Summaries for Efficient Long-Context
// Decoding", technical summary §2, "page-local spectral decomposition": when a
// page is finalised its keys are centred on the page centroid, a small
// eigendecomposition of the deviations is taken, and the top-r eigenvectors
// (the page's own basis) plus per-token coefficients are kept; "quantisation":
// basis in int4, coefficients and centroid in int8 (about 10 % of the page's
// KV bytes at B = 16, r = 8).  Built off the decode critical path.
//
// One half-warp per page-head (two per warp, four warps per CTA):
//   1. lane i loads 16-byte chunk i of every key row (coalesced), forms the
//      centroid of its 8 dims and writes the centred rows X to shared memory;
//   2. lane i computes row i of the Gram matrix G = X X^T (16 x 16, fp32);
//   3. parallel cyclic Jacobi (round-robin pairing, 8 disjoint rotations per
//      round, 15 rounds per sweep) with lane i owning row i of G and of the
//      eigenvector matrix W; kSweeps sweeps;
//   4. eigenvalues ranked (descending, lower index on ties), top 8 kept,
//      sign fixed so the largest |coefficient| of each direction is positive,
//      lambda_k <= 1e-6 lambda_1 -> zero direction;
//   5. V = X^T W_r Lambda^{-1/2} (lane i: dims 8i..8i+7), C = W_r Lambda^{1/2};
//   6. symmetric per-tensor quantisation (round half to even) and packing into
//      the 784-byte record, stored with 16-byte writes.

#include <cstdint>

#include "common.cuh"
#include "params.h"

namespace locks {

constexpr int kBuildWarps = 4;
constexpr int kBuildThreads = kBuildWarps * 32;
constexpr int kXStride = 132;          // padded fp32 row of X (conflict-free LDS.128)
constexpr int kSweeps = 8;

struct HalfWarpSmem {
  float X[kPage * kXStride];           // centred keys
  float G[kPage * kPage];              // current Gram rows (for diagonal reads)
  float W[kPage * kPage];              // eigenvectors (rows)
  float2 rot[kPage];                   // (c, s) of the pair containing index j
  float lift[kPage * kRank];           // W_r Lambda^{-1/2} (signed)
  float coef[kPage * kRank];           // C
  int order[kPage];
  int8_t vcode[kRank * kHeadDim];      // [k][dim]
  __align__(16) uint8_t rec[kRecord];
  float scratch[4];
};
constexpr int kBuildSmem = 2 * kBuildWarps * (int)sizeof(HalfWarpSmem);

// Round-robin partner of index i in round r (circle method on 16 players).
__host__ __device__ constexpr int jacobi_partner(int i, int r) {
  return i == 15 ? r : (i == r ? 15 : (2 * r - i + 15) % 15);
}

// The rotation of a pair and its updates, explicitly rounded (x is this
// row's or column's element, y the partner's).
__device__ __forceinline__ float rot_lo(float c, float s, float x, float y) { return __fmaf_rn(c, x, __fmul_rn(-s, y)); }
__device__ __forceinline__ float rot_hi(float c, float s, float x, float y) { return __fmaf_rn(c, x, __fmul_rn(s, y)); }

// (c, s) of the rotation that zeroes e in [[a, e], [e, b]] (the smaller of
// the two, |theta| <= pi/4), from the half-angle relations with d = b - a,
// f = 2e and h = sqrt(d^2 + f^2):
//   c^2 = (1 + |d| / h) / 2,   s = sign(d) f / (2 h c).
// Two dependent approximate reciprocal square roots (single instructions: the
// rotation is the serial part of every round).  d and f are first scaled by
// the power of two that brings |f| into [2, 4), and |d| is clamped to 2^60
// (where s < 2^-58, a rotation the fp32 updates cannot tell from none): h^2
// then lies in [4, 2^121] whatever the magnitudes of the page's keys, so both
// operands stay normal.
__device__ __forceinline__ float2 jacobi_cs(float a, float bb, float e) {
  float c = 1.f, s = 0.f;
  if (fabsf(e) > 1e-30f && __fmul_rn(e, e) > __fmul_rn(1e-24f, fabsf(__fmul_rn(a, bb)))) {
    const float d = __fsub_rn(bb, a);
    // k = 2^-(exponent of e): |e| k in [1, 2)
    const float k = __int_as_float(0x7F000000 - (__float_as_int(e) & 0x7F800000));
    const float fk = __fmul_rn(__fmul_rn(2.f, e), k);                 // exact: f scaled into [2, 4)
    const float ad = fminf(__fmul_rn(fabsf(d), k), 0x1p60f);
    const float h2 = __fmaf_rn(ad, ad, __fmul_rn(fk, fk));
    const float r = fast_rsqrt(h2);                                  // 1 / h
    const float c2 = __fmaf_rn(__fmul_rn(0.5f, ad), r, 0.5f);       // in [0.5, 1]
    const float sr = __fmul_rn(__fmul_rn(d < 0.f ? -0.5f : 0.5f, fk), r);
    const float q = fast_rsqrt(c2);                                  // 1 / c
    c = __fmul_rn(c2, q);
    s = __fmul_rn(sr, q);
  }
  return make_float2(c, s);
}

template <int R>
__device__ __forceinline__ void jacobi_round(float (&g)[kPage], float (&w)[kPage], int i, int hbase,
                                             HalfWarpSmem& S) {
  const int q = jacobi_partner(i, R);
  const int lo = min(i, q), hi = max(i, q);
  const float2 cs0 = jacobi_cs(S.G[lo * kPage + lo], S.G[hi * kPage + hi], S.G[lo * kPage + hi]);
  const float c = cs0.x, s = cs0.y;
  S.rot[i] = cs0;
  // row update: rows lo, hi of J^T G
  float pg[kPage];
#pragma unroll
  for (int j = 0; j < kPage; ++j) pg[j] = __shfl_sync(0xffffffffu, g[j], hbase + q);
  const bool is_lo = (i == lo);
#pragma unroll
  for (int j = 0; j < kPage; ++j) g[j] = is_lo ? rot_lo(c, s, g[j], pg[j]) : rot_hi(c, s, g[j], pg[j]);
  __syncwarp();
  // column update: (J^T G) J and W J; the pairing of column j is static
  float ng[kPage], nw[kPage];
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    const int pj = jacobi_partner(j, R);
    const float2 cs = S.rot[j];
    if (j < pj) {
      ng[j] = rot_lo(cs.x, cs.y, g[j], g[pj]);
      nw[j] = rot_lo(cs.x, cs.y, w[j], w[pj]);
    } else {
      ng[j] = rot_hi(cs.x, cs.y, g[j], g[pj]);
      nw[j] = rot_hi(cs.x, cs.y, w[j], w[pj]);
    }
  }
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    g[j] = ng[j];
    w[j] = nw[j];
  }
  // publish the new row for the next round's diagonal / pivot reads
#pragma unroll
  for (int j = 0; j < kPage; j += 4)
    *reinterpret_cast<float4*>(&S.G[i * kPage + j]) = make_float4(g[j], g[j + 1], g[j + 2], g[j + 3]);
  __syncwarp();
}

template <int R>
struct Sweep {
  static __device__ __forceinline__ void run(float (&g)[kPage], float (&w)[kPage], int i, int hbase,
                                             HalfWarpSmem& S) {
    jacobi_round<R>(g, w, i, hbase, S);
    Sweep<R + 1>::run(g, w, i, hbase, S);
  }
};
template <>
struct Sweep<15> {
  static __device__ __forceinline__ void run(float (&)[kPage], float (&)[kPage], int, int, HalfWarpSmem&) {}
};

// Steps 1-3 for the half-warp's page-head (block blk, KV head h; a zero page
// when !active): lane i ends with the centroid of dims 8i..8i+7 in mu8, row i
// of the rotated Gram matrix in g (its diagonal: the eigenvalues, also in
// S.G) and row i of the eigenvector matrix in w; S.X holds the centred keys.
__device__ __forceinline__ void build_eigen(const BuildParams& p, HalfWarpSmem& S, bool active, int64_t blk, int h,
                                            int i, int hbase, float (&mu8)[8], float (&g)[kPage],
                                            float (&w)[kPage]) {
  // ---- 1. load, centroid, centred rows
  {
    float kv[kPage][8];
    const __nv_bfloat16* src = p.k_cache + ((active ? blk : 0) * p.H_kv + h) * (int64_t)(kPage * kHeadDim);
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (active) raw = *reinterpret_cast<const uint4*>(src + r * kHeadDim + 8 * i);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kv[r][2 * e] = __low2float(b2[e]);
        kv[r][2 * e + 1] = __high2float(b2[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float sum = 0.f;
#pragma unroll
      for (int r = 0; r < kPage; ++r) sum += kv[r][e];
      mu8[e] = sum * (1.f / kPage);
    }
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      float* xr = &S.X[r * kXStride + 8 * i];
      *reinterpret_cast<float4*>(xr) = make_float4(kv[r][0] - mu8[0], kv[r][1] - mu8[1], kv[r][2] - mu8[2], kv[r][3] - mu8[3]);
      *reinterpret_cast<float4*>(xr + 4) = make_float4(kv[r][4] - mu8[4], kv[r][5] - mu8[5], kv[r][6] - mu8[6], kv[r][7] - mu8[7]);
    }
  }
  __syncwarp();

  // ---- 2. Gram row i
#pragma unroll
  for (int j = 0; j < kPage; ++j) g[j] = 0.f;
  for (int d = 0; d < kHeadDim; d += 4) {
    const float4 xi = *reinterpret_cast<const float4*>(&S.X[i * kXStride + d]);
#pragma unroll
    for (int j = 0; j < kPage; ++j) {
      const float4 xj = *reinterpret_cast<const float4*>(&S.X[j * kXStride + d]);
      g[j] = fmaf(xi.x, xj.x, g[j]);
      g[j] = fmaf(xi.y, xj.y, g[j]);
      g[j] = fmaf(xi.z, xj.z, g[j]);
      g[j] = fmaf(xi.w, xj.w, g[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < kPage; ++j) w[j] = (j == i) ? 1.f : 0.f;
#pragma unroll
  for (int j = 0; j < kPage; j += 4)
    *reinterpret_cast<float4*>(&S.G[i * kPage + j]) = make_float4(g[j], g[j + 1], g[j + 2], g[j + 3]);
  __syncwarp();

  // ---- 3. Jacobi sweeps.  A fixed count: stopping on the off-diagonal mass
  // relative to the whole matrix (dominated by lambda_1) leaves pairs of small
  // eigenvalues coupled; in fp32 the top-8 directions reach their rounding
  // floor after 7 sweeps on low-rank, noisy and full-rank pages alike.
  for (int sweep = 0; sweep < kSweeps; ++sweep) Sweep<0>::run(g, w, i, hbase, S);
}

// Page-head ph of this launch: its block and KV head, and whether it is
// built (a block id outside the cache is flagged, by the thread that
// reports, and skipped).
__device__ __forceinline__ bool target_of(const BuildParams& p, int64_t ph, bool report, int64_t& blk, int& h) {
  const int n_pages = p.n_dev != nullptr ? min(p.n_build, max(0, *p.n_dev)) : p.n_build;
  const int64_t total = (int64_t)n_pages * p.H_kv;
  bool active = ph < total;
  blk = -1;
  h = 0;
  if (active && p.block_table != nullptr) {
    // crossing mode: the page request b's current token completed, if any
    const int b = (int)(ph / p.H_kv);
    const int L = p.seq_lens[b];
    h = (int)(ph % p.H_kv);
    if (L > 0 && L % kPage == 0 && L / kPage <= p.max_pages)
      blk = p.block_table[(int64_t)b * p.max_pages + L / kPage - 1];
    else
      active = false;
    if (active && (blk < 0 || blk >= p.num_blocks)) {
      if (report) flag_status(p.status, LOCKS_FLAG_BAD_BLOCK);
      active = false;
    }
  } else if (active) {
    blk = p.block_ids[ph / p.H_kv];
    h = (int)(ph % p.H_kv);
    if (blk < 0 || blk >= p.num_blocks) {
      if (report) flag_status(p.status, LOCKS_FLAG_BAD_BLOCK);
      active = false;
    }
  }
  return active;
}

// The half-warp's page-head (lane i of the half).
__device__ __forceinline__ bool build_target(const BuildParams& p, int i, int64_t& blk, int& h) {
  const int warp = threadIdx.x >> 5, half = (threadIdx.x >> 4) & 1;
  const int64_t ph = ((int64_t)blockIdx.x * kBuildWarps + warp) * 2 + half;
  return target_of(p, ph, i == 0, blk, h);
}

// Byte positions in the 784-byte record (include/locks.h): the centroid code
// of dim, the coefficient code (token, direction k), and the dim held by
// nibble pos of basis word wi (word wi at byte 4 wi).
__device__ __forceinline__ int rec_mu_byte(int dim) {
  const int s = dim >> 4, wd = dim & 15, hh = wd >> 3, t = (wd & 7) >> 1, ee = wd & 1;
  return 512 + t * 32 + s * 4 + hh * 2 + ee;
}
__device__ __forceinline__ int rec_coef_byte(int token, int k) {
  const int nt = token >> 3, gd = token & 7, tk = k >> 1, ek = k & 1;
  return 640 + (gd * 4 + tk) * 4 + nt * 2 + ek;
}
__device__ __forceinline__ int basis_word_dim(int wi, int pos) {
  const int t = (wi >> 2) & 3, pp = wi & 3;
  const int e = pos >> 2, sp = (pos & 3) >> 1, hh = pos & 1;
  return 16 * (2 * pp + sp) + 8 * hh + 2 * t + e;
}

__global__ void __launch_bounds__(kBuildThreads) build_kernel(const BuildParams p) {
  extern __shared__ __align__(16) uint8_t smem_b[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, i = lane & 15, hbase = lane & 16;
  HalfWarpSmem& S = reinterpret_cast<HalfWarpSmem*>(smem_b)[warp * 2 + half];
  int64_t blk;
  int h;
  // a scorer launched as a programmatic dependent of this build may start now
  griddep_launch_dependents();
  // Both half-warps run every step (warp-synchronous shuffles); an inactive
  // half works on a zero page and stores nothing.
  const bool active = build_target(p, i, blk, h);
  float mu8[8], g[kPage], w[kPage];
  build_eigen(p, S, active, blk, h, i, hbase, mu8, g, w);

  // ---- 4. rank eigenvalues, pick the top r, fix signs
#pragma unroll
  for (int j = 0; j < kPage; j += 4)
    *reinterpret_cast<float4*>(&S.W[i * kPage + j]) = make_float4(w[j], w[j + 1], w[j + 2], w[j + 3]);
  __syncwarp();
  float lam[kPage];   // (a NaN would break the ranking below: it ranks last)
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    const float v = S.G[j * kPage + j];
    lam[j] = v == v ? v : -INFINITY;
  }
  const float my_lam = lam[i];
  int rank = 0;
  float lam1 = lam[0];
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    rank += (lam[j] > my_lam) || (lam[j] == my_lam && j < i);
    lam1 = fmaxf(lam1, lam[j]);
  }
  S.order[rank] = i;
  float tail = rank >= kRank ? fmaxf(my_lam, 0.f) : 0.f;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) tail += __shfl_xor_sync(0xffffffffu, tail, o);
  __syncwarp();
  if (i < kRank) {
    const int ev = S.order[i];
    const float l = S.G[ev * kPage + ev];
    const bool keep = l > 1e-6f * lam1 && l > 0.f;
    // sign: largest |component| of this eigenvector positive (first on ties)
    float best = -1.f, sgn = 1.f;
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const float v = S.W[r * kPage + ev];
      if (fabsf(v) > best) {
        best = fabsf(v);
        sgn = v < 0.f ? -1.f : 1.f;
      }
    }
    const float sig = keep ? sqrtf(l) : 0.f;
    const float inv = keep ? 1.f / sig : 0.f;
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const float v = S.W[r * kPage + ev] * sgn;
      S.lift[r * kRank + i] = v * inv;
      S.coef[r * kRank + i] = v * sig;
    }
  }
  __syncwarp();

  // ---- 5. V = X^T W_r Lambda^{-1/2}: lane i -> dims 8i..8i+7
  float V[8][kRank];
#pragma unroll
  for (int e = 0; e < 8; ++e)
#pragma unroll
    for (int k = 0; k < kRank; ++k) V[e][k] = 0.f;
#pragma unroll 4
  for (int r = 0; r < kPage; ++r) {
    const float4 x0 = *reinterpret_cast<const float4*>(&S.X[r * kXStride + 8 * i]);
    const float4 x1 = *reinterpret_cast<const float4*>(&S.X[r * kXStride + 8 * i + 4]);
    const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const float4 l0 = *reinterpret_cast<const float4*>(&S.lift[r * kRank]);
    const float4 l1 = *reinterpret_cast<const float4*>(&S.lift[r * kRank + 4]);
    const float ls[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int k = 0; k < kRank; ++k) V[e][k] = fmaf(xs[e], ls[k], V[e][k]);
  }

  // ---- 6. quantise and pack
  float vmax = 0.f, mmax = 0.f, cmax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mmax = fmaxf(mmax, fabsf(mu8[e]));
#pragma unroll
    for (int k = 0; k < kRank; ++k) vmax = fmaxf(vmax, fabsf(V[e][k]));
  }
  float crow[kRank];
#pragma unroll
  for (int k = 0; k < kRank; ++k) {
    crow[k] = S.coef[i * kRank + k];
    cmax = fmaxf(cmax, fabsf(crow[k]));
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  }
  const float sV = vmax / 7.f, sM = mmax / 127.f, sC = cmax / 127.f;
  // codes = round-half-even(x / s) taken as x * (1 / s): one rounding more,
  // which moves a code only for a quotient within an ulp of a half
  const float iV = sV > 0.f ? __frcp_rn(sV) : 0.f;
  const float iM = sM > 0.f ? __frcp_rn(sM) : 0.f;
  const float iC = sC > 0.f ? __frcp_rn(sC) : 0.f;
  // V codes -> [k][dim] bytes
#pragma unroll
  for (int e = 0; e < 8; ++e)
#pragma unroll
    for (int k = 0; k < kRank; ++k) {
      int c = __float2int_rn(V[e][k] * iV);
      c = max(-7, min(7, c));
      S.vcode[k * kHeadDim + 8 * i + e] = (int8_t)c;
    }
  // centroid codes straight into the record
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    int c = __float2int_rn(mu8[e] * iM);
    c = max(-127, min(127, c));
    S.rec[rec_mu_byte(8 * i + e)] = (uint8_t)(int8_t)c;
  }
  // coefficient codes of token i
#pragma unroll
  for (int k = 0; k < kRank; ++k) {
    int c = __float2int_rn(crow[k] * iC);
    c = max(-127, min(127, c));
    S.rec[rec_coef_byte(i, k)] = (uint8_t)(int8_t)c;
  }
  if (i == 0) {
    float* scl = reinterpret_cast<float*>(&S.rec[768]);
    scl[0] = sV;
    scl[1] = sM;
    scl[2] = sC;
    scl[3] = tail;
  }
  __syncwarp();
  // pack basis words: lane i builds words i, i+16, ..., i+112 (word = k*16 + t*4 + p)
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int wi = i + 16 * m, k = wi >> 4;
    uint32_t word = 0;
#pragma unroll
    for (int pos = 0; pos < 8; ++pos)
      word |= ((uint32_t)S.vcode[k * kHeadDim + basis_word_dim(wi, pos)] & 0xFu) << (4 * pos);
    *reinterpret_cast<uint32_t*>(&S.rec[4 * wi]) = word;
  }
  __syncwarp();
  if (active) {
    uint4* dst = reinterpret_cast<uint4*>(p.summ + (blk * p.H_kv + h) * (int64_t)kRecord);
    const uint4* srcr = reinterpret_cast<const uint4*>(S.rec);
    for (int c = i; c < kRecord / 16; c += 16) dst[c] = srcr[c];
  }
}

// ---------------------------------------------------------------- a few pages
// The pages a decode step completes are few (one a request), so their build
// is bound by the latency of one page-head's eigendecomposition, not by
// throughput.  build_page_kernel gives each page-head a CTA of 8 warps and
// decomposes G by Householder reduction, multisection and inverse iteration
// (page_eigen_tridiag), whose dependency chain is about a third of the 120
// Jacobi rounds'.  The loops stay rolled: a step's kernel runs with its code
// out of L2, and straight-line code pays for every instruction fetched.  The
// records meet the same bar as build_kernel's against the decomposition in
// fp64 (codes within one of it), not the bits of build_kernel's.
constexpr int kPbWarps = 8;
constexpr int kPbThreads = kPbWarps * 32;

struct PageSmem {
  float X[kPage * kXStride];           // keys, then centred keys
  float G[2][kPage * kPage];           // G, then its eigenvalues on the diagonal; the reflectors
  float W[2][kPage * kPage];           // the eigenvectors (columns); Gram-Schmidt scratch
  float mu[kHeadDim];
  float lift[kPage * kRank];
  float coef[kPage * kRank];
  int order[kPage];
  // tridiagonal matrix T (diagonal, subdiagonal), its eigenvalues, and the
  // scale, bracket and norm of T
  float tri_d[kPage], tri_e[kPage], tri_lam[kPage];
  float tri_s[4];
  float red[3][kPbWarps];
  float tail;
  int8_t vcode[kRank * kHeadDim];
  __align__(16) uint8_t rec[kRecord];
};

static_assert(offsetof(PageSmem, G) % 16 == 0 && (kPage * kPage * sizeof(float)) % 16 == 0,
              "the reflectors in G[1] are read as float4");

// Eigenpairs of the symmetric 16x16 matrix in S.G[0] by Householder
// tridiagonalisation, multisection on Sturm counts and inverse iteration,
// the classical alternative to Jacobi (Golub & Van Loan §8.3 for the
// tridiagonal reduction and Sturm sequences, §8.2 for inverse iteration).
// All kPbThreads threads call it.  On return S.G[0][i][i] holds eigenvalue i
// (ascending in i) and column i of S.W[0] its unit eigenvector; vectors of
// close eigenvalues are orthogonalised only among i >= kRank, the ones the
// record keeps.
//
// Built for latency, with three CTA barriers in all:
//  * the reduction runs in warp 0's registers, lane l holding column l; the
//    update keeps A symmetric bit for bit, so lane l's own element (k, l)
//    is the reflector's component l and no lane needs another's row;
//  * the tridiagonal matrix T is scaled by a power of two to a norm near 1,
//    and the Sturm counts use the three-term recurrence of the leading
//    minors (one fused multiply-add a step on the dependency chain, the
//    minors rescaled by a power of two every fourth step), 16 points an
//    eigenvalue a round;
//  * the inverse iteration factors T - lambda I once and solves twice.
__device__ __forceinline__ void page_eigen_tridiag(PageSmem& S, int tid) {
  float* HV = S.G[1];     // row k: unit Householder vector of step k
  const int warp = tid >> 5, lane = tid & 31;
  // ---- Householder: A = Q T Q^T, Q = H_0 H_1 ... H_13, H_k = I - 2 v_k v_k^T
  if (warp == 0) {
    const int l = lane & 15;
    // column l of A (equal to row l); at step k register i holds row k + i,
    // zero past row 15 (the rows shift down a register a step)
    float a[kPage];
#pragma unroll
    for (int i = 0; i < kPage; ++i) a[i] = S.G[0][i * kPage + l];
#pragma unroll 1
    for (int k = 0; k < kPage - 2; ++k) {
      float xs[kPage];   // column k, rows k, k + 1, ..
#pragma unroll
      for (int i = 0; i < kPage; ++i) xs[i] = __shfl_sync(0xffffffffu, a[i], k);
      float sig0 = 0.f, sig1 = 0.f;   // below the subdiagonal entry
#pragma unroll
      for (int i = 2; i < kPage; ++i) {
        if (i & 1) sig1 = fmaf(xs[i], xs[i], sig1);
        else sig0 = fmaf(xs[i], xs[i], sig0);
      }
      const float sig = sig0 + sig1;
      const float x0 = xs[1];
      float alpha = x0, v0 = 0.f, inv = 0.f;
      if (sig > 0.f) {
        // correctly rounded: the entries the reflection zeroes are dropped, not
        // formed, so an ulp of error here lands on the small eigenvalues
        const float nrm = sqrtf(fmaf(x0, x0, sig));
        alpha = x0 >= 0.f ? -nrm : nrm;
        v0 = x0 - alpha;
        inv = rsqrtf(fmaf(v0, v0, sig));
      }
      float v[kPage];
      v[0] = 0.f;
      v[1] = v0 * inv;
#pragma unroll
      for (int i = 2; i < kPage; ++i) v[i] = xs[i] * inv;
      // this lane's component: element (k, l) of A equals (l, k)
      const float vl = l == k + 1 ? v0 * inv : (l > k + 1 ? a[0] * inv : 0.f);
      if (lane < kPage) HV[k * kPage + lane] = vl;
      if (lane == 0) {
        S.tri_d[k] = xs[0];
        S.tri_e[k] = alpha;
      }
      // 2p = 2 A v (row l of A is column l), then w = 2p - 2 (v.p) v
      float p0 = 0.f, p1 = 0.f;
#pragma unroll
      for (int i = 1; i < kPage; ++i) {
        if (i & 1) p1 = fmaf(a[i], v[i], p1);
        else p0 = fmaf(a[i], v[i], p0);
      }
      const float pl2 = 2.f * (p0 + p1);
      float pv2[kPage];
#pragma unroll
      for (int i = 1; i < kPage; ++i) {
        const float t = __shfl_sync(0xffffffffu, pl2, k + i);
        pv2[i] = k + i < kPage ? t : 0.f;
      }
      float K0 = 0.f, K1 = 0.f;
#pragma unroll
      for (int i = 1; i < kPage; ++i) {
        if (i & 1) K1 = fmaf(v[i], pv2[i], K1);
        else K0 = fmaf(v[i], pv2[i], K0);
      }
      const float m2K = -(K0 + K1);   // -2 (v.p)
      const float wl = fmaf(m2K, vl, pl2);
      // A -= v w^T + w v^T on rows and columns past k: both products are
      // rounded, then added, so elements (i, l) and (l, i) stay equal (a
      // fused form drifts apart by an ulp a step, and the reflectors built
      // from one side then amplify it).  Lanes up to k hold columns no later
      // step reads; row and column k are final (d_k, e_k) and drop out.
#pragma unroll
      for (int i = 1; i < kPage; ++i) {
        const float wi = fmaf(m2K, v[i], pv2[i]);
        a[i - 1] = __fsub_rn(a[i], __fadd_rn(__fmul_rn(v[i], wl), __fmul_rn(wi, vl)));
      }
      a[kPage - 1] = 0.f;
    }
    const float d14 = __shfl_sync(0xffffffffu, a[0], 14);
    const float d15 = __shfl_sync(0xffffffffu, a[1], 15);
    const float e14 = __shfl_sync(0xffffffffu, a[1], 14);
    if (lane == 0) {
      S.tri_d[14] = d14;
      S.tri_d[15] = d15;
      S.tri_e[14] = e14;
      S.tri_e[15] = 0.f;
    }
    __syncwarp();
    // Gershgorin bracket of T, and the power of two that scales it to [1, 2)
    const int i = l;
    const float di = S.tri_d[i], ei = fabsf(S.tri_e[i]), em = i > 0 ? fabsf(S.tri_e[i - 1]) : 0.f;
    float lo = di - ei - em, hi = di + ei + em;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      const float bound = fmaxf(fabsf(lo), fabsf(hi));
      const int ex = (__float_as_int(bound) >> 23) & 0xFF;
      const float sc = bound > 1e-30f ? __int_as_float((254 - ex) << 23) : 1.f;   // bound * sc in [1, 2)
      const float span = (hi - lo) * sc;
      S.tri_s[0] = sc;
      S.tri_s[1] = fmaf(lo, sc, -(1e-6f * span + 1e-30f));
      S.tri_s[2] = fmaf(hi, sc, 1e-6f * span + 1e-30f);
      S.tri_s[3] = bound;
    }
  }
  __syncthreads();
  // ---- multisection on the scaled T: half-warp i brackets eigenvalue i
  // (ascending); lane t counts the eigenvalues below a + (t + 1)(b - a)/17
  {
    const int i = tid >> 4, t = tid & 15;
    const float sc = S.tri_s[0];
    // scaled diagonal, minus the scaled squared subdiagonal floored at 2^-60
    // (eigenvalues move by at most 2^-30 of |T|): a zero minor is then never
    // followed by another
    float d[kPage], me2[kPage];
#pragma unroll
    for (int j = 0; j < kPage; ++j) {
      d[j] = S.tri_d[j] * sc;
      const float ej = S.tri_e[j] * sc;
      me2[j] = -fmaxf(ej * ej, 0x1p-60f);
    }
    float a = S.tri_s[1], b = S.tri_s[2];
#pragma unroll 1
    for (int round = 0; round < 6; ++round) {
      const float x = fmaf((b - a) * (1.f / 17.f), (float)(t + 1), a);
      // leading minors P_j of T - x I: P_0 = 1, P_1 = d_0 - x,
      // P_{j+1} = (d_j - x) P_j - e_{j-1}^2 P_{j-1}; a sign change from P_j
      // to P_{j+1} is a negative pivot, one eigenvalue below x.  A zero minor
      // counts as positive: its successor -e^2 P_{j-1} then carries the one
      // change of the pair, as a pivot of -0 would have.
      float Pp = 1.f, P = d[0] - x;
      int cnt = P < 0.f;
#pragma unroll
      for (int j = 1; j < kPage; ++j) {
        const float Pn = fmaf(d[j] - x, P, me2[j - 1] * Pp);
        cnt += (Pn < 0.f) != (P < 0.f);
        Pp = P;
        P = Pn;
        if ((j & 3) == 3) {   // bring the larger of the two minors into [1, 2)
          const float mx = fmaxf(fabsf(P), fabsf(Pp));
          const float f = __int_as_float((254 - ((__float_as_int(mx) >> 23) & 0xFF)) << 23);
          P *= f;
          Pp *= f;
        }
      }
      // eigenvalue i lies in (x_t, x_t+1] where cnt(x_t) <= i < cnt(x_t+1)
      float lo = cnt <= i ? x : a, hi = cnt > i ? x : b;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        lo = fmaxf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fminf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
      a = lo;
      b = hi;
    }
    if (t == 0) S.tri_lam[i] = 0.5f * (a + b);
  }
  __syncthreads();
  // ---- inverse iteration (warp 0, lane i < 16: eigenvalue i) on the scaled
  // T: one factorisation of T - lambda I (no pivoting, pivots kept away from
  // zero), two solves from distinct start vectors, then Gram-Schmidt inside
  // clusters of close eigenvalues and the reflections back
  if (warp == 0) {
    const int i = lane & 15;
    const float sc = S.tri_s[0];
    float d[kPage], e[kPage];
#pragma unroll
    for (int j = 0; j < kPage; ++j) {
      d[j] = S.tri_d[j] * sc;
      e[j] = S.tri_e[j] * sc;
    }
    const float lam = S.tri_lam[i];
    const float tnorm = fmaxf(fabsf(S.tri_s[1]), fabsf(S.tri_s[2]));
    const float floor_p = 1e-7f * tnorm;
    float inv[kPage], cp[kPage];
    {
      float m = d[0] - lam;
#pragma unroll
      for (int j = 0; j < kPage; ++j) {
        if (j > 0) m = fmaf(-e[j - 1], cp[j - 1], d[j] - lam);
        if (fabsf(m) < floor_p) m = m < 0.f ? -floor_p : floor_p;
        inv[j] = fast_rcp(m);
        cp[j] = e[j] * inv[j];
      }
    }
    float x[kPage];
#pragma unroll
    for (int j = 0; j < kPage; ++j) x[j] = fmaf((float)(((j + 1) * (i + 3) * 7) % 13), 0.37f / 13.f, 1.f);
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {
      float y = x[0] * inv[0];
      x[0] = y;
#pragma unroll
      for (int j = 1; j < kPage; ++j) {
        y = fmaf(-e[j - 1], y, x[j]) * inv[j];
        x[j] = y;
      }
#pragma unroll
      for (int j = kPage - 2; j >= 0; --j) x[j] = fmaf(-cp[j], x[j + 1], x[j]);
      float m0 = 0.f, m1 = 0.f;
#pragma unroll
      for (int j = 0; j < kPage; j += 2) {
        m0 = fmaxf(m0, fabsf(x[j]));
        m1 = fmaxf(m1, fabsf(x[j + 1]));
      }
      const float mx = fmaxf(m0, m1);
      const float s = mx > 0.f ? fast_rcp(mx) : 1.f;
#pragma unroll
      for (int j = 0; j < kPage; ++j) x[j] *= s;
    }
    {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int j = 0; j < kPage; j += 2) {
        s0 = fmaf(x[j], x[j], s0);
        s1 = fmaf(x[j + 1], x[j + 1], s1);
      }
      const float rn = rsqrtf(fmaxf(s0 + s1, 1e-30f));
#pragma unroll
      for (int j = 0; j < kPage; ++j) x[j] *= rn;
    }
    // clusters among the top kRank eigenvalues (indices kRank .. 15, the only
    // vectors the record keeps; the ranking below breaks ties toward the
    // higher index): eigenvalue i joins i - 1's when closer than 1e-3 of |T|.
    // The small eigenvalues of a nearly low-rank page form one wide cluster,
    // whose serial orthogonalisation would buy nothing.
    const float ctol = 1e-3f * tnorm;
    const bool joins = i > kRank && (lam - S.tri_lam[i - 1]) <= ctol;
    if (__any_sync(0xffffffffu, lane < kPage && joins)) {
      float* Yv = S.W[1];   // [16][16]: eigenvector i at row i
      if (lane < kPage)
#pragma unroll
        for (int j = 0; j < kPage; ++j) Yv[i * kPage + j] = x[j];
      __syncwarp();
      // in index order, each member of a cluster is made orthogonal to the
      // members before it, then normalised
      for (int mbr = kRank + 1; mbr < kPage; ++mbr) {
        if (lane == mbr && joins) {
          int first = mbr;
          while (first > kRank && S.tri_lam[first] - S.tri_lam[first - 1] <= ctol) --first;
          for (int q = first; q < mbr; ++q) {
            float dot = 0.f;
#pragma unroll
            for (int j = 0; j < kPage; ++j) dot = fmaf(Yv[q * kPage + j], x[j], dot);
#pragma unroll
            for (int j = 0; j < kPage; ++j) x[j] = fmaf(-dot, Yv[q * kPage + j], x[j]);
          }
          float ss = 0.f;
#pragma unroll
          for (int j = 0; j < kPage; ++j) ss = fmaf(x[j], x[j], ss);
          const float rn = rsqrtf(fmaxf(ss, 1e-30f));
#pragma unroll
          for (int j = 0; j < kPage; ++j) {
            x[j] *= rn;
            Yv[i * kPage + j] = x[j];
          }
        }
        __syncwarp();
      }
    }
    // back to the Gram matrix's basis: z = H_0 (H_1 (... (H_13 x))); v_k is
    // zero at indices up to k, so the full-length products change nothing there
#pragma unroll 1
    for (int k = kPage - 3; k >= 0; --k) {
      float hv[kPage];
#pragma unroll
      for (int j = 0; j < kPage; j += 4) {
        const float4 q = *reinterpret_cast<const float4*>(&HV[k * kPage + j]);
        hv[j] = q.x;
        hv[j + 1] = q.y;
        hv[j + 2] = q.z;
        hv[j + 3] = q.w;
      }
      float t0 = 0.f, t1 = 0.f;
#pragma unroll
      for (int j = 0; j < kPage; j += 2) {
        t0 = fmaf(hv[j], x[j], t0);
        t1 = fmaf(hv[j + 1], x[j + 1], t1);
      }
      const float m2 = -2.f * (t0 + t1);
#pragma unroll
      for (int j = 0; j < kPage; ++j) x[j] = fmaf(m2, hv[j], x[j]);
    }
    if (lane < kPage) {
#pragma unroll
      for (int j = 0; j < kPage; ++j) S.W[0][j * kPage + i] = x[j];
      S.G[0][i * kPage + i] = S.tri_s[3] > 1e-30f ? lam / sc : 0.f;   // a zero matrix: every eigenvalue 0
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kPbThreads) build_page_kernel(const BuildParams p) {
  __shared__ PageSmem S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_launch_dependents();
  int64_t blk;
  int h;
  if (!target_of(p, blockIdx.x, tid == 0, blk, h)) return;   // uniform over the CTA

  // ---- 1. keys (key row t / 16, dims 8 (t % 16) ..), centroid, centred keys
  const int kr = tid >> 4, kc = tid & 15;
  const uint4 raw = *reinterpret_cast<const uint4*>(p.k_cache + (blk * p.H_kv + h) * (int64_t)(kPage * kHeadDim) +
                                                    kr * kHeadDim + 8 * kc);
  {
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float* xr = &S.X[kr * kXStride + 8 * kc];
    *reinterpret_cast<float4*>(xr) =
        make_float4(__low2float(b2[0]), __high2float(b2[0]), __low2float(b2[1]), __high2float(b2[1]));
    *reinterpret_cast<float4*>(xr + 4) =
        make_float4(__low2float(b2[2]), __high2float(b2[2]), __low2float(b2[3]), __high2float(b2[3]));
  }
  __syncthreads();
  if (tid < kHeadDim) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kPage; ++k) sum += S.X[k * kXStride + tid];
    S.mu[tid] = sum * (1.f / kPage);
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 8; ++e) S.X[kr * kXStride + 8 * kc + e] -= S.mu[8 * kc + e];
  __syncthreads();

  // ---- 2. Gram entry (kr, kc): four partial sums, each the same for (kc, kr),
  // so G is symmetric bit for bit (the reduction relies on it)
  {
    float g0 = 0.f, g1 = 0.f, g2 = 0.f, g3 = 0.f;
#pragma unroll 8
    for (int d = 0; d < kHeadDim; d += 4) {
      const float4 xi = *reinterpret_cast<const float4*>(&S.X[kr * kXStride + d]);
      const float4 xj = *reinterpret_cast<const float4*>(&S.X[kc * kXStride + d]);
      g0 = fmaf(xi.x, xj.x, g0);
      g1 = fmaf(xi.y, xj.y, g1);
      g2 = fmaf(xi.z, xj.z, g2);
      g3 = fmaf(xi.w, xj.w, g3);
    }
    S.G[0][tid] = (g0 + g1) + (g2 + g3);
  }
  __syncthreads();
  // ---- 3. eigenpairs: eigenvalue i at G[i][i], its vector in column i of W
  page_eigen_tridiag(S, tid);
  const float* Gf = S.G[0];
  const float* Wf = S.W[0];

  // ---- 4. rank the eigenvalues, top r, signs (warp 0; lanes 16..31 mirror
  // 0..15).  The eigenvalues ascend with the index, and ties rank the higher
  // index first, so the top r are indices 16 - r .. 15: the vectors that
  // went through the clusters' orthogonalisation.
  if (warp == 0) {
    const int i = lane & 15;
    float lam[kPage];
#pragma unroll
    for (int j = 0; j < kPage; ++j) {
      const float v = Gf[j * kPage + j];
      lam[j] = v == v ? v : -INFINITY;
    }
    const float vi = Gf[i * kPage + i];
    const float my_lam = vi == vi ? vi : -INFINITY;
    int pos = 0;
    float lam1 = lam[0];
#pragma unroll
    for (int j = 0; j < kPage; ++j) {
      pos += (lam[j] > my_lam) || (lam[j] == my_lam && j > i);   // ties: higher index first
      lam1 = fmaxf(lam1, lam[j]);
    }
    if (lane < kPage) S.order[pos] = i;
    float tail = pos >= kRank ? fmaxf(my_lam, 0.f) : 0.f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) tail += __shfl_xor_sync(0xffffffffu, tail, o);
    if (lane == 0) S.tail = tail;
    __syncwarp();
    if (lane < kRank) {
      const int ev = S.order[lane];
      const float l = Gf[ev * kPage + ev];
      const bool keep = l > 1e-6f * lam1 && l > 0.f;
      float best = -1.f, sgn = 1.f;
#pragma unroll
      for (int k = 0; k < kPage; ++k) {
        const float v = Wf[k * kPage + ev];
        if (fabsf(v) > best) {
          best = fabsf(v);
          sgn = v < 0.f ? -1.f : 1.f;
        }
      }
      const float sig = keep ? sqrtf(l) : 0.f;
      const float inv = keep ? 1.f / sig : 0.f;
#pragma unroll
      for (int k = 0; k < kPage; ++k) {
        const float v = Wf[k * kPage + ev] * sgn;
        S.lift[k * kRank + lane] = v * inv;
        S.coef[k * kRank + lane] = v * sig;
      }
    }
  }
  __syncthreads();

  // ---- 5. V = X^T W_r Lambda^{-1/2}: thread t < 256 -> dim t / 2, directions 4 (t % 2) ..
  float v4[4] = {0.f, 0.f, 0.f, 0.f};
  const int vdim = tid >> 1, k0 = 4 * (tid & 1);
  if (tid < kPage * kPage) {
#pragma unroll
    for (int k = 0; k < kPage; ++k) {
      const float x = S.X[k * kXStride + vdim];
#pragma unroll
      for (int m = 0; m < 4; ++m) v4[m] = fmaf(x, S.lift[k * kRank + k0 + m], v4[m]);
    }
  }

  // ---- 6. scales (block maxima), codes, packing
  float vmax = 0.f, mmax = 0.f, cmax = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) vmax = fmaxf(vmax, fabsf(v4[m]));
  if (tid < kHeadDim) mmax = fabsf(S.mu[tid]);
  if (tid < kPage * kRank) cmax = fabsf(S.coef[tid]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  }
  if (lane == 0) {
    S.red[0][warp] = vmax;
    S.red[1][warp] = mmax;
    S.red[2][warp] = cmax;
  }
  __syncthreads();
  vmax = mmax = cmax = 0.f;
#pragma unroll
  for (int w = 0; w < kPbWarps; ++w) {
    vmax = fmaxf(vmax, S.red[0][w]);
    mmax = fmaxf(mmax, S.red[1][w]);
    cmax = fmaxf(cmax, S.red[2][w]);
  }
  const float sV = vmax / 7.f, sM = mmax / 127.f, sC = cmax / 127.f;
  const float iV = sV > 0.f ? __frcp_rn(sV) : 0.f;
  const float iM = sM > 0.f ? __frcp_rn(sM) : 0.f;
  const float iC = sC > 0.f ? __frcp_rn(sC) : 0.f;
  if (tid < kPage * kPage) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      int code = __float2int_rn(v4[m] * iV);
      code = max(-7, min(7, code));
      S.vcode[(k0 + m) * kHeadDim + vdim] = (int8_t)code;
    }
  }
  if (tid < kHeadDim) {
    int code = __float2int_rn(S.mu[tid] * iM);
    code = max(-127, min(127, code));
    S.rec[rec_mu_byte(tid)] = (uint8_t)(int8_t)code;
  }
  if (tid < kPage * kRank) {
    int code = __float2int_rn(S.coef[tid] * iC);
    code = max(-127, min(127, code));
    S.rec[rec_coef_byte(tid / kRank, tid % kRank)] = (uint8_t)(int8_t)code;
  }
  if (tid == 0) {
    float* scl = reinterpret_cast<float*>(&S.rec[768]);
    scl[0] = sV;
    scl[1] = sM;
    scl[2] = sC;
    scl[3] = S.tail;
  }
  __syncthreads();
  if (tid < kRank * kHeadDim / 8) {   // basis word tid
    const int k = tid >> 4;
    uint32_t word = 0;
#pragma unroll
    for (int pos = 0; pos < 8; ++pos)
      word |= ((uint32_t)S.vcode[k * kHeadDim + basis_word_dim(tid, pos)] & 0xFu) << (4 * pos);
    *reinterpret_cast<uint32_t*>(&S.rec[4 * tid]) = word;
  }
  __syncthreads();
  if (tid < kRecord / 16)
    reinterpret_cast<uint4*>(p.summ + (blk * p.H_kv + h) * (int64_t)kRecord)[tid] =
        reinterpret_cast<const uint4*>(S.rec)[tid];
}

cudaError_t launch_build_pages(const BuildParams& p, cudaStream_t stream) {
  const int64_t grid = (int64_t)p.n_build * p.H_kv;
  if (grid == 0) return cudaSuccess;
  // The crossing step's scorer (98 KB of shared memory a CTA) shares SMs
  // with these CTAs: with the default carveout an SM running one holds too
  // little shared memory for any scorer CTA until it is idle again, and the
  // scorer's last CTAs then start only when the build ends.
  // (set on every call: the attribute belongs to the current device)
  const cudaError_t carve = cudaFuncSetAttribute(build_page_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 cudaSharedmemCarveoutMaxShared);
  if (carve != cudaSuccess) return carve;
  build_page_kernel<<<(unsigned)grid, kPbThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- fp32 records
// Unquantised records of rank r <= 16 (cfg quant = 0, a debug and reference
// configuration): the same centroid, Gram matrix and Jacobi eigenpairs, the
// top r directions (same ranking, sign and zero-floor rules), written as fp32
// [mu: 128][V: 128 x r, dim-major][C: 16 x r][tail energy, 0, 0, 0].
struct DebugLift {
  float lift[kPage * kPage];   // [token][direction]: W_r Lambda^{-1/2}
  float coef[kPage * kPage];   // [token][direction]: C
};
constexpr int kDebugSmem = 2 * kBuildWarps * (int)(sizeof(HalfWarpSmem) + sizeof(DebugLift));

__global__ void __launch_bounds__(kBuildThreads) build_debug_kernel(const BuildParams p, int rank_r) {
  extern __shared__ __align__(16) uint8_t smem_d[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, i = lane & 15, hbase = lane & 16;
  HalfWarpSmem& S = reinterpret_cast<HalfWarpSmem*>(smem_d)[warp * 2 + half];
  DebugLift& D = reinterpret_cast<DebugLift*>(smem_d + 2 * kBuildWarps * sizeof(HalfWarpSmem))[warp * 2 + half];
  int64_t blk;
  int h;
  const bool active = build_target(p, i, blk, h);
  float mu8[8], g[kPage], w[kPage];
  build_eigen(p, S, active, blk, h, i, hbase, mu8, g, w);

#pragma unroll
  for (int j = 0; j < kPage; j += 4)
    *reinterpret_cast<float4*>(&S.W[i * kPage + j]) = make_float4(w[j], w[j + 1], w[j + 2], w[j + 3]);
  __syncwarp();
  float lam[kPage];
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    const float v = S.G[j * kPage + j];
    lam[j] = v == v ? v : -INFINITY;
  }
  const float my_lam = lam[i];
  int pos = 0;
  float lam1 = lam[0];
#pragma unroll
  for (int j = 0; j < kPage; ++j) {
    pos += (lam[j] > my_lam) || (lam[j] == my_lam && j < i);
    lam1 = fmaxf(lam1, lam[j]);
  }
  S.order[pos] = i;
  float tail = pos >= rank_r ? fmaxf(my_lam, 0.f) : 0.f;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) tail += __shfl_xor_sync(0xffffffffu, tail, o);
  __syncwarp();
  {
    // lane i: direction i (when i < r)
    const int ev = S.order[i];
    const float l = S.G[ev * kPage + ev];
    const bool keep = i < rank_r && l > 1e-6f * lam1 && l > 0.f;
    float best = -1.f, sgn = 1.f;
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const float v = S.W[r * kPage + ev];
      if (fabsf(v) > best) {
        best = fabsf(v);
        sgn = v < 0.f ? -1.f : 1.f;
      }
    }
    const float sig = keep ? sqrtf(l) : 0.f;
    const float inv = keep ? 1.f / sig : 0.f;
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const float v = S.W[r * kPage + ev] * sgn;
      D.lift[r * kPage + i] = v * inv;
      D.coef[r * kPage + i] = v * sig;
    }
  }
  __syncwarp();
  if (!active) return;
  float* rec = reinterpret_cast<float*>(p.summ + (blk * p.H_kv + h) * (int64_t)(528 + 576 * rank_r));
  // centroid
#pragma unroll
  for (int e = 0; e < 8; ++e) rec[8 * i + e] = mu8[e];
  // V rows of dims 8i..8i+7: V[dim][k] = sum_r X[r][dim] lift[r][k]
  float* Vd = rec + kHeadDim;
  for (int k = 0; k < rank_r; ++k) {
    float v8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kPage; ++r) {
      const float lk = D.lift[r * kPage + k];
#pragma unroll
      for (int e = 0; e < 8; ++e) v8[e] = fmaf(S.X[r * kXStride + 8 * i + e], lk, v8[e]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) Vd[(8 * i + e) * rank_r + k] = v8[e];
  }
  // C row of token i
  float* Cd = Vd + kHeadDim * rank_r;
  for (int k = 0; k < rank_r; ++k) Cd[i * rank_r + k] = D.coef[i * kPage + k];
  if (i == 0) {
    float* t = Cd + kPage * rank_r;
    t[0] = tail;
    t[1] = t[2] = t[3] = 0.f;
  }
}

cudaError_t launch_build_debug(const BuildParams& p, int rank_r, cudaStream_t stream) {
  static DynSmemAttr smem_attr;
  const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(build_debug_kernel), kDebugSmem, smem_attr);
  if (e != cudaSuccess) return e;
  const int64_t page_heads = (int64_t)p.n_build * p.H_kv;
  const int64_t grid = (page_heads + 2 * kBuildWarps - 1) / (2 * kBuildWarps);
  if (grid == 0) return cudaSuccess;
  build_debug_kernel<<<(unsigned)grid, kBuildThreads, kDebugSmem, stream>>>(p, rank_r);
  return cudaGetLastError();
}

cudaError_t launch_build(const BuildParams& p, cudaStream_t stream) {
  static DynSmemAttr smem_attr;
  const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(build_kernel), kBuildSmem, smem_attr);
  if (e != cudaSuccess) return e;
  const int64_t page_heads = (int64_t)p.n_build * p.H_kv;
  const int64_t grid = (page_heads + 2 * kBuildWarps - 1) / (2 * kBuildWarps);
  if (grid == 0) return cudaSuccess;
  build_kernel<<<(unsigned)grid, kBuildThreads, kBuildSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace locks
