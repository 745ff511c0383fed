// noalloc.cu -- locks_sparse_decode_noalloc and locks_noalloc_read_status:
// sparse decode attention that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory at all: a serving engine that has
// handed all of HBM to its KV-cache pool, code on a latency-critical path where
// a cudaMalloc would synchronise the device, or a host integration with no
// allocator of its own.  This entry point runs the same split-K attention
// kernel as locks_sparse_decode, with the same validation and the same split
// of each unit's items (host_plan.h), but its scratch (per-split partial
// softmax states, merge tickets and the status word) lives in one file-scope
// device array of fixed size that every GPU loading the library holds until
// the process exits.  It calls no cudaMalloc, cudaFree or allocating routine.
//
// Set-up: in host code the array's name is only a stand-in, never a device
// address.  The first call in a CUDA context looks up the array's device
// address there with cudaGetSymbolAddress and keeps it, keyed by the
// context's unique id (a context created after cudaDeviceReset, or another
// context made current, gets its own look-up); make that first call before any
// stream capture.  Every call clears the merge tickets with one cudaMemsetAsync
// on `stream`; the status word keeps accumulating flags until
// locks_noalloc_read_status reads and clears it.  All calls share the one
// array and it keeps the last call's contents, so calls that overlap on the
// GPU (two streams, two host threads) race on it: serialise them.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/locks.h"
#include "common.cuh"
#include "host_plan.h"
#include "params.h"

namespace {

using namespace locks;

constexpr size_t kScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr size_t kHeaderBytes = 256;                 // status word
constexpr size_t kPartBytes = (size_t)kGroup * (2 + kHeadDim) * sizeof(float);   // one split's state

__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

// ---- the array's device address, per CUDA context
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return fns;
}

constexpr int kCacheSlots = 64;
struct AddrSlot {
  unsigned long long ctx_id;
  void* ptr;
};
std::mutex g_mu;
AddrSlot g_slots[kCacheSlots] = {};
int g_next_slot = 0;

// Unique id of the current CUDA context, 0 if none is current or the driver
// entry points are missing.
unsigned long long current_ctx_id() {
  const DriverFns& fns = driver_fns();
  unsigned long long id = 0;
  CUcontext ctx = nullptr;
  if (fns.get_current == nullptr || fns.get_id == nullptr) return 0;
  if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current context.
cudaError_t scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = current_ctx_id();
  if (id != 0) {
    for (const AddrSlot& s : g_slots)
      if (s.ctx_id == id) {
        *out = s.ptr;
        return cudaSuccess;
      }
  }
  // first use in this context (the look-up also makes the runtime's primary
  // context current when none was)
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_ctx_id();
  if (id != 0) {
    g_slots[g_next_slot] = AddrSlot{id, p};
    g_next_slot = (g_next_slot + 1) % kCacheSlots;
  }
  *out = p;
  return cudaSuccess;
}

bool a16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t tickets_bytes(int64_t units) { return ((size_t)units * sizeof(uint32_t) + 255) / 256 * 256; }

}  // namespace

extern "C" locks_status locks_sparse_decode_noalloc(
    const locks_cfg* cfg, const void* q, const void* k_cache, const void* v_cache, int64_t num_blocks,
    const int32_t* block_table, const int32_t* seq_lens, const int32_t* selected,
    const int32_t* n_selected, int32_t batch, int32_t max_pages, int32_t budget_pages, float sm_scale,
    float* out, locks_stream_t stream) {
  if (cfg == nullptr) return LOCKS_ERR_INVALID_ARG;
  if (!cfg_supported(cfg)) return LOCKS_ERR_UNSUPPORTED;
  const int H = cfg->num_kv_heads;
  if (batch < 0 || max_pages < 1 || budget_pages < 0 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f)) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(block_table) || !a16(seq_lens) || !a16(out) ||
      !a16(n_selected) || (budget_pages > 0 && !a16(selected)))
    return LOCKS_ERR_INVALID_ARG;
  if (num_blocks * H * kPage >= (int64_t)1 << 31) return LOCKS_ERR_UNSUPPORTED;

  // the same split as the workspace entry point; the size check comes before
  // any CUDA call
  const int64_t units = (int64_t)batch * H;
  int splits = 1, ips = 1;
  sparse_split(units, budget_pages, &splits, &ips);
  const size_t tb = tickets_bytes(units);
  const size_t need = kHeaderBytes + tb + (size_t)units * (size_t)splits * kPartBytes;
  if (need > kScratchBytes) return LOCKS_ERR_WORKSPACE;   // batch too large for the fixed scratch

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return LOCKS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* scratch = static_cast<uint8_t*>(base);
  if (cudaMemsetAsync(scratch + kHeaderBytes, 0, tb, s) != cudaSuccess) return LOCKS_ERR_CUDA;

  CUtensorMap tmk, tmv;
  if (!encode_cache_map(&tmk, k_cache, num_blocks, H) || !encode_cache_map(&tmv, v_cache, num_blocks, H))
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
  p.part = reinterpret_cast<float*>(scratch + kHeaderBytes + tb);
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

extern "C" locks_status locks_noalloc_read_status(uint32_t* flags, locks_stream_t stream) {
  if (flags == nullptr) return LOCKS_ERR_INVALID_ARG;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return LOCKS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, base, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(base, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return LOCKS_ERR_CUDA;
  *flags = v;
  return (v & LOCKS_FLAG_TIMEOUT) ? LOCKS_ERR_TIMEOUT : LOCKS_OK;
}
