// common.cuh -- device helpers shared by the LOCKS kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement path (mbarrier, cp.async.bulk,
// cp.async.bulk.tensor), warp-level tensor-core fragments (ldmatrix,
// movmatrix, mma.sync) and small conversion tricks.  Every spin on an
// mbarrier is bounded: after ~1 s of %globaltimer it records
// LOCKS_FLAG_TIMEOUT in the status word and reports failure to the caller.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/locks.h"

namespace locks {

// Host side: the dynamic shared memory a kernel may use is an attribute of the
// kernel on the current device.  DynSmemAttr records, per device, the largest
// size already set, so a launcher sets it once per device and size (and again
// when a larger size is needed); safe to call from several host threads.
constexpr int kMaxDevices = 64;
struct DynSmemAttr {
  std::atomic<size_t> set[kMaxDevices] = {};
};
inline cudaError_t ensure_dyn_smem(const void* kernel, size_t bytes, DynSmemAttr& rec) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  size_t cur = rec.set[dev].load(std::memory_order_acquire);
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  while (cur < bytes && !rec.set[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
  }
  return cudaSuccess;
}


constexpr int kHeadDim = 128;
constexpr int kPage = 16;
constexpr int kRank = 8;
constexpr int kGroup = 4;
constexpr int kRecord = 784;
constexpr int kTargetCtas = 304;   // 2 resident CTAs x 152 SMs (GB300)
constexpr int kSelCluster = 8;     // CTAs per (request, KV head) in the selection
constexpr int kFusedMaxKeysPerCta = 16384; // keys per selecting CTA (fused: keys + block ids share the 128 KB ring)
constexpr int kFusedMaxBudget = 2047;      // fused pass: <= 32 items per warp of 64
constexpr int kSmemLimit = 200 * 1024;     // dynamic shared memory we allow a CTA (static <= 27 KB)

// Dynamic shared memory of the selection kernel: slice keys, the selected
// list (rank 0) and, when staged, the slice's scores (16 bytes a page).
__host__ __device__ inline size_t select_stage_offset(int max_pages, int budget, int cluster) {
  const int slice_cap = (max_pages + cluster - 1) / cluster;
  return (4 * ((size_t)slice_cap + (size_t)budget + 4) + 15) / 16 * 16;
}
__host__ __device__ inline size_t select_smem_bytes(int max_pages, int budget, int cluster = kSelCluster,
                                                    bool stage = false) {
  const int slice_cap = (max_pages + cluster - 1) / cluster;
  return stage ? select_stage_offset(max_pages, budget, cluster) + 16 * (size_t)slice_cap
               : 4 * ((size_t)slice_cap + (size_t)budget + 4);
}

// ---------------------------------------------------------------- status
__device__ __forceinline__ void flag_status(uint32_t* status, uint32_t bit) {
  if (status != nullptr) atomicOr(status, bit);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the kernel before it runs; it waits here for
// that kernel's results (a no-op when nothing precedes it).  The kernel
// before it lets it start early with griddep_launch_dependents.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait: true once the phase with this parity completed, false (and
// LOCKS_FLAG_TIMEOUT recorded) after limit_ns of %globaltimer (one second by
// default; every wait in the decode kernels uses the default).
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
      flag_status(status, LOCKS_FLAG_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
// 16-byte asynchronous copy global -> shared, completed by cp_async_wait_all
// in the issuing thread.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src_gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Untiled bulk copy global -> shared; completes `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 2-D tensor copy global -> shared (box and swizzle come from the map).
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const void* tmap, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst_smem)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch the 128-byte line holding `p` into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------- fragments
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// 8x8 b16 transpose across the warp (fragment layout: lane l holds row l/4,
// columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- conversions
// The conversions below use the known "magic number" method: a bitwise op
// places the integer under a fixed f16 exponent and one subtraction removes
// the exponent's value (for int4/int8 -> f16 with LOP3 see Kim et al., "Who
// Says Elephants Can't Run: Bringing Large Scale MoE Models into Cloud Scale
// Production", 2022).  The variants here are exact for two's-complement
// codes.
// (a & b) ^ c in one LOP3.
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Four int8 codes [b0 b1 b2 b3] -> exact f16x2 (b0,b1) and (b2,b3).
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;                        // offset binary
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);   // 0x64|b0, 0x64|b1
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342);
  lo = h2_sub(a, 0x64806480u);                               // - 1152
  hi = h2_sub(b, 0x64806480u);
}

// Eight int4 codes (two's complement nibbles) -> four exact f16x2 pairs, one
// shift, four LOP3s and four HSUB2s.  A nibble at bits 0-3 of a half (pairs
// 0|4 and 2|6) goes under the exponent of 1024, where a mantissa unit is 1:
// 1024 + (n ^ 8) - 1032 = code.  A nibble at bits 4-7 (pairs 1|5 and 3|7)
// goes under the exponent of 64, where bit 4 is worth 1: 64 + (n ^ 8) - 72.
// Exact values keep the tensor-core accumulators free of large offsets, whose
// cancellation would cost precision in proportion to |q|.
__device__ __forceinline__ void nib8_to_h2x4(uint32_t w, uint32_t& p04, uint32_t& p15, uint32_t& p26,
                                             uint32_t& p37) {
  const uint32_t w8 = w >> 8;
  p04 = h2_sub(and_xor(w, 0x000F000Fu, 0x64086408u), 0x64086408u);
  p15 = h2_sub(and_xor(w, 0x00F000F0u, 0x54805480u), 0x54805480u);
  p26 = h2_sub(and_xor(w8, 0x000F000Fu, 0x64086408u), 0x64086408u);
  p37 = h2_sub(and_xor(w8, 0x00F000F0u, 0x54805480u), 0x54805480u);
}

// fp32 pair -> f16x2 high part and f16x2 residual (x ~= hi + lo to ~2^-22).
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(__fsub_rn(x0, hf.x), __fsub_rn(x1, hf.y));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Single-instruction approximate reciprocal and reciprocal square root
// (flush-to-zero forms: callers pass normal, positive-range operands).
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_rsqrt(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace locks
