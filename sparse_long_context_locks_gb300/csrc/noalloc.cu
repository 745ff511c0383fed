// noalloc.cu -- locks_sparse_decode_noalloc: sparse decode attention that
// needs no caller-provided workspace.
//
// Some callers cannot allocate device memory at all: a serving engine that has
// handed all of HBM to its KV-cache pool, code on a latency-critical path where
// a cudaMalloc would synchronise the device, or a host integration with no
// allocator of its own.  This entry point runs the same split-K attention
// kernel as locks_sparse_decode, but its scratch (per-split partial softmax
// states, merge tickets and the status word) lives in one file-scope device
// array of fixed size that every GPU loading the library holds until the
// process exits.  It calls no cudaMalloc, cudaFree or allocating routine.
//
// Set-up: the first call on a device looks up the array's device address with
// cudaGetSymbolAddress (the host-side symbol is only a stand-in, never a device
// pointer) and caches it per device; make that first call before any stream
// capture.  Every call clears the status word and the tickets with one
// cudaMemsetAsync on `stream`.  All calls share the one array and it keeps the
// last call's contents, so calls that overlap on the GPU (two streams, two
// host threads) race on it: serialise them.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/locks.h"
#include "common.cuh"
#include "params.h"

namespace {

using namespace locks;

constexpr size_t kScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr size_t kHeaderBytes = 256;                 // status word

__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

bool encode_map(CUtensorMap* map, const void* base, int64_t num_blocks, int H) {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)(num_blocks * H * kPage)};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, kPage};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool a16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" locks_status locks_sparse_decode_noalloc(
    const locks_cfg* cfg, const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
    const int32_t* block_table, const int32_t* seq_lens, const int32_t* selected,
    const int32_t* n_selected, int32_t batch, int32_t max_pages, int32_t budget_pages, float sm_scale,
    float* out, locks_stream_t stream) {
  if (cfg == nullptr) return LOCKS_ERR_INVALID_ARG;
  if (cfg->head_dim != kHeadDim || cfg->page_size != kPage || cfg->rank != kRank || cfg->quant != 1 ||
      cfg->group_size != kGroup || cfg->num_kv_heads < 1)
    return LOCKS_ERR_UNSUPPORTED;
  const int H = cfg->num_kv_heads;
  if (batch < 0 || max_pages < 1 || budget_pages < 0 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f)) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(block_table) || !a16(seq_lens) || !a16(out) ||
      !a16(n_selected) || (budget_pages > 0 && !a16(selected)))
    return LOCKS_ERR_INVALID_ARG;
  if (num_blocks * H * kPage >= (int64_t)1 << 31) return LOCKS_ERR_UNSUPPORTED;

  // same split rule as the workspace entry point: one wave of resident CTAs,
  // at least one item per warp
  const int64_t units = (int64_t)batch * H;
  const int64_t items = (int64_t)budget_pages + 1;
  const int64_t by_items = (items + 3) / 4;
  const int64_t want = units > 0 ? kTargetCtas / units : 1;
  const int splits = (int)std::max<int64_t>(1, std::min(by_items, want));
  const int ips = (int)((items + splits - 1) / splits);
  const size_t tickets_bytes = ((size_t)units * sizeof(uint32_t) + 255) / 256 * 256;
  const size_t need = kHeaderBytes + tickets_bytes + (size_t)units * splits * kGroup * (2 + kHeadDim) * sizeof(float);
  if (need > kScratchBytes) return LOCKS_ERR_WORKSPACE;   // batch too large for the fixed scratch

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return LOCKS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* scratch = static_cast<uint8_t*>(base);
  if (cudaMemsetAsync(scratch, 0, kHeaderBytes + tickets_bytes, s) != cudaSuccess) return LOCKS_ERR_CUDA;

  CUtensorMap tmk, tmv;
  if (!encode_map(&tmk, k_cache, num_blocks, H) || !encode_map(&tmv, v_cache, num_blocks, H))
    return LOCKS_ERR_CUDA;
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.selected = selected;
  p.n_selected = n_selected;
  p.out = out;
  p.status = reinterpret_cast<uint32_t*>(scratch);
  p.tickets = reinterpret_cast<uint32_t*>(scratch + kHeaderBytes);
  p.part = reinterpret_cast<float*>(scratch + kHeaderBytes + tickets_bytes);
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.max_pages = max_pages;
  p.H_kv = H;
  p.budget = budget_pages;
  p.dense = 0;
  p.splits = splits;
  p.items_per_split = ips;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  return launch_attn(tmk, tmv, p, s) == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}
