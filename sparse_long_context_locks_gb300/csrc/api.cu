// api.cu -- extern "C" entry points of liblocks (declared in include/locks.h).
//
// Host side only: argument validation (before any launch), work planning
// (grid shapes and workspace regions, a pure function of the batch shape so
// that locks_workspace_bytes and every launch agree), tensor-map encoding for
// the attention kernel, and launches.  No allocation, no synchronisation on
// the decode path.

#include <algorithm>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/locks.h"
#include "common.cuh"

#include "host_plan.h"
#include "params.h"

namespace locks {

bool cfg_supported(const locks_cfg* c) {
  if (c == nullptr) return false;
  if (c->head_dim != kHeadDim || c->page_size != kPage || c->group_size != kGroup) return false;
  // quantised records at rank 8, or unquantised fp32 records of rank 1..16
  if (!((c->quant == 1 && c->rank == kRank) || (c->quant == 0 && c->rank >= 1 && c->rank <= kPage))) return false;
  const int H = c->num_kv_heads;
  if (H < 1) return false;
  const int h_cta = H < 8 ? H : 8;
  return (8 % h_cta == 0) && (H % h_cta == 0);
}

// Sparse units all hold about budget + 1 items, so the split is sized for
// one wave: every CTA resident at once, each with the longest slice (and at
// least one item per warp).  Measured at batch 16: 0.59 of peak against 0.34
// with eight waves of short CTAs.
void sparse_split(int64_t units, int budget_pages, int* splits, int* items_per_split) {
  const int64_t items = (int64_t)budget_pages + 1;
  const int64_t by_items = (items + 3) / 4;
  const int64_t want = kTargetCtas / (units > 0 ? units : 1);
  const int64_t sp = by_items < want ? by_items : want;
  *splits = (int)(sp > 1 ? sp : 1);
  *items_per_split = (int)((items + *splits - 1) / *splits);
}

}  // namespace locks

namespace {

using namespace locks;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Plan {
  // scoring
  int h_cta, wph, pps, head_groups, ch_pages, n_chunks, n_items, score_grid;
  // selection
  // attention
  int sparse_splits, sparse_ips, dense_splits, dense_ips, max_splits;
  // workspace regions
  size_t off_scores, off_attn, off_tickets, total;
};

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Longest context (in pages) for which locks_decode_step takes the fused kernel.
constexpr int kFusedStepMaxPages = 32768;

int pick_splits(int units, int max_items) {
  // aim for ~8 waves of resident CTAs, at least 4 items (one per warp) each
  const int by_items = max(1, ceil_div(max_items, 4));
  const int want = max(1, ceil_div(8 * kTargetCtas, units));
  return max(1, min(by_items, want));
}

Plan make_plan(const locks_cfg* c, int batch, int max_pages, int budget) {
  Plan pl{};
  const int H = c->num_kv_heads;
  pl.h_cta = H < 8 ? H : 8;
  pl.wph = 8 / pl.h_cta;
  pl.pps = 4 * pl.wph;
  pl.head_groups = H / pl.h_cta;
  pl.ch_pages = pl.pps;   // one stage per work item: the grid splits evenly
  pl.n_chunks = ceil_div(max_pages, pl.ch_pages);
  const int64_t items = (int64_t)batch * pl.head_groups * pl.n_chunks;
  pl.n_items = (int)items;
  pl.score_grid = (int)(items < kTargetCtas ? items : kTargetCtas);
  const int units = batch * H;
  sparse_split(units, budget, &pl.sparse_splits, &pl.sparse_ips);
  // Dense units vary with the context, so larger batches keep about eight
  // waves for balance (batch 16: 0.98 of peak, against 0.94 with one wave);
  // a few units would leave eight waves of very short CTAs, so they take one
  // wave (one request at 128K: 0.84 of peak, against 0.53).
  pl.dense_splits = units <= kTargetCtas / 8
                        ? max(1, min(ceil_div(max_pages, 4), kTargetCtas / max(1, units)))
                        : pick_splits(units, max_pages);
  pl.dense_ips = ceil_div(max_pages, pl.dense_splits);
  pl.max_splits = max(pl.sparse_splits, pl.dense_splits);

  // Regions whose size or position does not depend on the budget come first,
  // so every call of a step (whatever budget it passes) agrees on them.
  size_t off = kAlign;  // [0, 256): status word
  pl.off_tickets = off;
  off = align_up(off + (size_t)units * sizeof(uint32_t));
  pl.off_scores = off;
  off = align_up(off + (size_t)batch * H * max_pages * kGroup * sizeof(float));
  pl.off_attn = off;   // last: its size depends on the split counts
  off = align_up(off + (size_t)units * pl.max_splits * kGroup * (2 + kHeadDim) * sizeof(float));
  pl.total = off;
  return pl;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device (queried once per device; host only).
int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

// CTAs per (request, KV head) in the selection kernel (16, 8, 4 or 2).  Its
// clusters are latency-bound.  When every 8-CTA cluster of the batch is
// resident at once (4 CTAs an SM), 8 keeps each CTA's slice shortest: one
// request at 128K selects in ~15 us (26.6 with 2).  Past 2,048 pages a CTA
// (a request of more than 256K tokens), 16-CTA clusters (non-portable, 2 CTAs
// an SM by registers) halve the slices again when the occupancy query says
// they are all resident at once.  With more units the
// waves cost more than the slices save, and the smallest cluster whose slices
// fit the per-CTA key limit is best: batch 16 x 32K selects in 14.5 us with 2
// (16.4 with 4, 24.7 with 8), batch 64 x 256K in 85.6 us (116.5 with 8).
bool select_stage(int units, int cluster, int max_pages, int budget);

int select_cluster(int units, int max_pages, int budget) {
  if ((int64_t)units * kSelCluster <= 4 * (int64_t)num_sms()) {
    // A few requests at long context: 16 CTAs a unit halve every CTA's
    // slice, when all the clusters are resident at once.
    if ((max_pages + kSelCluster - 1) / kSelCluster > 2048 && (int64_t)units * 16 <= 2 * (int64_t)num_sms()) {
      const bool staged = select_stage(units, 16, max_pages, budget);
      if (select_smem_bytes(max_pages, budget, 16, staged) <= (size_t)kSmemLimit &&
          select16_max_clusters(select_smem_bytes(max_pages, budget, 16, staged), staged) >= units)
        return 16;
    }
    return kSelCluster;
  }
  int c = 2;
  while (c < kSelCluster && ((max_pages + c - 1) / c > kFusedMaxKeysPerCta ||
                             select_smem_bytes(max_pages, budget, c) > (size_t)kSmemLimit))
    c *= 2;
  return c;
}

// Whether the selection kernel copies each CTA's slice of scores to shared
// memory before its two passes over them.  Read from L2, a thread holds the
// first four of its scores in registers and then keeps only a few loads in
// flight: a slice of up to 1,024 pages is requested at once anyway (staging
// it costs ~1 us at 128K tokens), a longer one makes the passes latency-bound
// (one request at 1M tokens, 8,192 pages a CTA: 5.5 and 5 us; staged, the
// selection takes 21.9 us instead of 27.9).  The staged copy takes 16 bytes a
// page of shared memory, so it is used only while the grid stays resident in
// one wave (228 KB of shared memory an SM, the kernel's static part rounded
// up to 20 KB, 1 KB reserved a CTA, at most 4 CTAs an SM).
bool select_stage(int units, int cluster, int max_pages, int budget) {
  if ((max_pages + cluster - 1) / cluster <= 1024) return false;
  const size_t dyn = select_smem_bytes(max_pages, budget, cluster, true);
  if (dyn > (size_t)kSmemLimit) return false;
  const int64_t per_sm =
      std::min<int64_t>(cluster > 8 ? 2 : 4, (int64_t)(228 * 1024) / (int64_t)(dyn + 21 * 1024));
  return (int64_t)units * cluster <= per_sm * num_sms();
}

#define LOCKS_CHECK_PTR(p) \
  do {                     \
    if ((p) == nullptr || !aligned16(p)) return LOCKS_ERR_INVALID_ARG; \
  } while (0)

uint32_t* status_word(void* ws) { return ws ? reinterpret_cast<uint32_t*>(ws) : nullptr; }

}  // namespace

// ---------------------------------------------------------------- tensor maps
namespace locks {
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_blocks, int H) {
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)(num_blocks * H * kPage)};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, kPage};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace locks

namespace {

using namespace locks;

locks_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA; }

locks_status attention_common(const locks_cfg* cfg, const void* q, const void* k_cache,
                              const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                              const int32_t* seq_lens, const int32_t* selected,
                              const int32_t* n_selected, int32_t batch, int32_t max_pages,
                              int32_t budget_pages, float sm_scale, float* out, void* workspace,
                              size_t ws_bytes, cudaStream_t stream, bool dense, float* state_out = nullptr) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || budget_pages < 0 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(q);
  LOCKS_CHECK_PTR(k_cache);
  LOCKS_CHECK_PTR(v_cache);
  LOCKS_CHECK_PTR(block_table);
  LOCKS_CHECK_PTR(seq_lens);
  if (state_out == nullptr) LOCKS_CHECK_PTR(out);
  LOCKS_CHECK_PTR(workspace);
  if (!dense) {
    LOCKS_CHECK_PTR(n_selected);
    if (budget_pages > 0) LOCKS_CHECK_PTR(selected);
  }
  const int H = cfg->num_kv_heads;
  if (num_blocks * H * kPage >= (int64_t)1 << 31) return LOCKS_ERR_UNSUPPORTED;
  const Plan pl = make_plan(cfg, batch, max_pages, budget_pages);
  if (ws_bytes < pl.total) return LOCKS_ERR_WORKSPACE;

  CUtensorMap tmk, tmv;
  if (!encode_cache_map(&tmk, k_cache, num_blocks, H) || !encode_cache_map(&tmv, v_cache, num_blocks, H))
    return LOCKS_ERR_CUDA;

  AttnParams p{};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.selected = selected;
  p.n_selected = n_selected;
  p.out = out;
  p.state_out = state_out;
  p.part = reinterpret_cast<float*>(ws + pl.off_attn);
  p.tickets = reinterpret_cast<uint32_t*>(ws + pl.off_tickets);
  p.status = status_word(workspace);
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.max_pages = max_pages;
  p.H_kv = H;
  p.budget = budget_pages;
  p.dense = dense ? 1 : 0;
  p.splits = dense ? pl.dense_splits : pl.sparse_splits;
  p.items_per_split = dense ? pl.dense_ips : pl.sparse_ips;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  return from_cuda(launch_attn(tmk, tmv, p, stream));
}

}  // namespace

extern "C" {

size_t locks_summary_bytes(const locks_cfg* cfg) {
  if (!cfg_supported(cfg)) return 0;
  return cfg->quant == 1 ? (size_t)kRecord : (size_t)(528 + 576 * cfg->rank);
}

locks_status locks_workspace_bytes(const locks_cfg* cfg, int32_t batch, int32_t max_pages,
                                   int32_t budget_pages, size_t* bytes) {
  if (cfg == nullptr || bytes == nullptr) return LOCKS_ERR_INVALID_ARG;
  if (!cfg_supported(cfg)) return LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || budget_pages < 0) return LOCKS_ERR_INVALID_ARG;
  *bytes = make_plan(cfg, batch, max_pages, budget_pages).total;
  return LOCKS_OK;
}

locks_status locks_workspace_init(void* workspace, size_t workspace_bytes, locks_stream_t stream) {
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < kAlign) return LOCKS_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

locks_status locks_read_status(void* workspace, uint32_t* flags, locks_stream_t stream) {
  if (workspace == nullptr || flags == nullptr) return LOCKS_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return LOCKS_ERR_CUDA;
  *flags = v;
  return (v & LOCKS_FLAG_TIMEOUT) ? LOCKS_ERR_TIMEOUT : LOCKS_OK;
}

int32_t locks_device_accessible(const void* p) {
  if (p == nullptr) return 0;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();   // an unknown pointer leaves no sticky error
    return 0;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return 1;
    case cudaMemoryTypeHost:
      return a.devicePointer == p ? 1 : 0;
    default:
      return 0;
  }
}

locks_status locks_build_summaries(const locks_cfg* cfg, const void* k_cache, int64_t num_blocks,
                                   const int32_t* block_ids, int32_t n_build, void* summaries,
                                   void* workspace, size_t workspace_bytes, locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (n_build < 0 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (n_build == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(k_cache);
  LOCKS_CHECK_PTR(block_ids);
  LOCKS_CHECK_PTR(summaries);
  if (workspace != nullptr && (!aligned16(workspace) || workspace_bytes < sizeof(uint32_t)))
    return LOCKS_ERR_INVALID_ARG;
  BuildParams p{};
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.block_ids = block_ids;
  p.summ = static_cast<uint8_t*>(summaries);
  p.status = status_word(workspace);
  p.num_blocks = num_blocks;
  p.n_build = n_build;
  p.H_kv = cfg->num_kv_heads;
  if (cfg->quant == 0) return from_cuda(launch_build_debug(p, cfg->rank, reinterpret_cast<cudaStream_t>(stream)));
  return from_cuda(launch_build(p, reinterpret_cast<cudaStream_t>(stream)));
}

locks_status locks_build_pending(const locks_cfg* cfg, const void* k_cache, int64_t num_blocks,
                                 const int32_t* block_ids, const int32_t* n_pending, int32_t max_pending,
                                 void* summaries, void* workspace, size_t workspace_bytes,
                                 locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (max_pending < 0 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (max_pending == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(k_cache);
  LOCKS_CHECK_PTR(block_ids);
  LOCKS_CHECK_PTR(summaries);
  if (n_pending == nullptr || (reinterpret_cast<uintptr_t>(n_pending) & 3u) != 0) return LOCKS_ERR_INVALID_ARG;
  if (workspace != nullptr && (!aligned16(workspace) || workspace_bytes < sizeof(uint32_t)))
    return LOCKS_ERR_INVALID_ARG;
  BuildParams p{};
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  p.block_ids = block_ids;
  p.n_dev = n_pending;
  p.summ = static_cast<uint8_t*>(summaries);
  p.status = status_word(workspace);
  p.num_blocks = num_blocks;
  p.n_build = max_pending;
  p.H_kv = cfg->num_kv_heads;
  if (cfg->quant == 0) return from_cuda(launch_build_debug(p, cfg->rank, reinterpret_cast<cudaStream_t>(stream)));
  return from_cuda(launch_build_pages(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// locks_score; with defer_crossing the scorer is a programmatic dependent of
// the crossing build just launched on the stream, and copies the page each
// request's current token completed only after that build has ended.
locks_status score_impl(const locks_cfg* cfg, const void* q, const void* summaries, int64_t num_blocks,
                        const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t max_pages,
                        float* scores, void* workspace, size_t workspace_bytes, locks_stream_t stream,
                        bool defer_crossing) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(q);
  LOCKS_CHECK_PTR(summaries);
  LOCKS_CHECK_PTR(block_table);
  LOCKS_CHECK_PTR(seq_lens);
  LOCKS_CHECK_PTR(workspace);
  if (scores != nullptr && !aligned16(scores)) return LOCKS_ERR_INVALID_ARG;
  const Plan pl = make_plan(cfg, batch, max_pages, 0);
  if (workspace_bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ScoreParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.summ = static_cast<const uint8_t*>(summaries);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.scores = scores ? scores : reinterpret_cast<float*>(ws + pl.off_scores);
  p.status = status_word(workspace);
  p.num_blocks = num_blocks;
  p.batch = batch;
  p.max_pages = max_pages;
  p.H_kv = cfg->num_kv_heads;
  p.h_cta = pl.h_cta;
  p.wph = pl.wph;
  p.pps = pl.pps;
  p.ch_pages = pl.ch_pages;
  p.n_chunks = pl.n_chunks;
  p.head_groups = pl.head_groups;
  p.n_items = pl.n_items;
  // (the fp32 scorer is launched in stream order: after the whole build)
  if (cfg->quant == 0) return from_cuda(launch_score_debug(p, cfg->rank, reinterpret_cast<cudaStream_t>(stream)));
  p.defer_crossing = defer_crossing ? 1 : 0;
  // In a crossing step each SM running a page-build CTA has room (registers)
  // for one scorer CTA instead of two; the grid leaves those slots out
  // (up to 16), so every scorer CTA starts at once instead of the last ones
  // waiting for the build to end.
  int grid = pl.score_grid;
  if (defer_crossing) grid = max(1, min(grid, kTargetCtas - min(batch * cfg->num_kv_heads, 16)));
  return from_cuda(launch_score(p, grid, reinterpret_cast<cudaStream_t>(stream), defer_crossing));
}

}  // namespace

extern "C" {

locks_status locks_score(const locks_cfg* cfg, const void* q, const void* summaries, int64_t num_blocks,
                         const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                         int32_t max_pages, float* scores, void* workspace, size_t workspace_bytes,
                         locks_stream_t stream) {
  return score_impl(cfg, q, summaries, num_blocks, block_table, seq_lens, batch, max_pages, scores, workspace,
                    workspace_bytes, stream, false);
}

}  // extern "C"

namespace {

void fill_select(SelectParams& p, const Plan& pl, const locks_cfg* cfg, const int32_t* seq_lens, int32_t batch,
                 int32_t max_pages, int32_t budget_pages, const float* scores, int32_t* selected,
                 int32_t* n_selected, void* workspace) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.seq_lens = seq_lens;
  p.scores = scores ? scores : reinterpret_cast<const float*>(ws + pl.off_scores);
  p.selected = selected;
  p.n_selected = n_selected;
  p.status = status_word(workspace);
  p.batch = batch;
  p.max_pages = max_pages;
  p.H_kv = cfg->num_kv_heads;
  p.budget = budget_pages;
}

}  // namespace

extern "C" {

locks_status locks_select(const locks_cfg* cfg, const int32_t* seq_lens, int32_t batch, int32_t max_pages,
                          int32_t budget_pages, const float* scores, int32_t* selected,
                          int32_t* n_selected, void* workspace, size_t workspace_bytes,
                          locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || budget_pages < 0) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(seq_lens);
  LOCKS_CHECK_PTR(n_selected);
  LOCKS_CHECK_PTR(workspace);
  if (budget_pages > 0) LOCKS_CHECK_PTR(selected);
  if (scores != nullptr && !aligned16(scores)) return LOCKS_ERR_INVALID_ARG;
  if ((max_pages + kSelCluster - 1) / kSelCluster > kFusedMaxKeysPerCta ||
      select_smem_bytes(max_pages, budget_pages) > (size_t)kSmemLimit)
    return LOCKS_ERR_UNSUPPORTED;
  const Plan pl = make_plan(cfg, batch, max_pages, budget_pages);
  if (workspace_bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  SelectParams p{};
  fill_select(p, pl, cfg, seq_lens, batch, max_pages, budget_pages, scores, selected, n_selected, workspace);
  const int units = batch * cfg->num_kv_heads;
  const int cluster = select_cluster(units, max_pages, budget_pages);
  p.stage_scores = select_stage(units, cluster, max_pages, budget_pages) ? 1 : 0;
  return from_cuda(launch_select(p, units, cluster, reinterpret_cast<cudaStream_t>(stream)));
}

locks_status locks_select_sparse_decode(const locks_cfg* cfg, const void* q, const void* k_cache,
                                        const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                                        const int32_t* seq_lens, int32_t batch, int32_t max_pages,
                                        int32_t budget_pages, const float* scores, int32_t* selected,
                                        int32_t* n_selected, float sm_scale, float* out, void* workspace,
                                        size_t workspace_bytes, locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || budget_pages < 0 || num_blocks < 1) return LOCKS_ERR_INVALID_ARG;
  if (!(sm_scale > 0.f)) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(q);
  LOCKS_CHECK_PTR(k_cache);
  LOCKS_CHECK_PTR(v_cache);
  LOCKS_CHECK_PTR(block_table);
  LOCKS_CHECK_PTR(seq_lens);
  LOCKS_CHECK_PTR(n_selected);
  LOCKS_CHECK_PTR(out);
  LOCKS_CHECK_PTR(workspace);
  if (budget_pages > 0) LOCKS_CHECK_PTR(selected);
  if (scores != nullptr && !aligned16(scores)) return LOCKS_ERR_INVALID_ARG;
  const int H = cfg->num_kv_heads;
  // one cluster per (request, KV head): its 64 warps take at most 32 items
  // each, and its 8 slices of keys fit in the 128 KB staging ring
  if (budget_pages > kFusedMaxBudget || (max_pages + kSelCluster - 1) / kSelCluster > kFusedMaxKeysPerCta ||
      fused_smem_bytes(max_pages, budget_pages) > (size_t)kSmemLimit)
    return LOCKS_ERR_UNSUPPORTED;
  if (num_blocks * H * kPage >= (int64_t)1 << 31) return LOCKS_ERR_UNSUPPORTED;
  const Plan pl = make_plan(cfg, batch, max_pages, budget_pages);
  if (workspace_bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  CUtensorMap tmk, tmv;
  if (!encode_cache_map(&tmk, k_cache, num_blocks, H) || !encode_cache_map(&tmv, v_cache, num_blocks, H))
    return LOCKS_ERR_CUDA;
  FusedParams p{};
  fill_select(p.sel, pl, cfg, seq_lens, batch, max_pages, budget_pages, scores, selected, n_selected, workspace);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.block_table = block_table;
  p.out = out;
  p.num_blocks = num_blocks;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  return from_cuda(launch_select_attend(tmk, tmv, p, batch * H, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

locks_status decode_step_impl(const locks_cfg* cfg, const void* q, void* summaries, const void* k_cache,
                              const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                              const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages,
                              float sm_scale, float* scores, int32_t* selected, int32_t* n_selected, float* out,
                              void* workspace, size_t workspace_bytes, locks_stream_t stream, bool crossing) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (budget_pages < 0 || budget_pages > kFusedMaxBudget) return budget_pages < 0 ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch > 0 && (max_pages + kSelCluster - 1) / kSelCluster > kFusedMaxKeysPerCta) return LOCKS_ERR_UNSUPPORTED;
  if (batch > 0) {
    LOCKS_CHECK_PTR(k_cache);
    LOCKS_CHECK_PTR(v_cache);
    LOCKS_CHECK_PTR(n_selected);
    LOCKS_CHECK_PTR(out);
    if (budget_pages > 0) LOCKS_CHECK_PTR(selected);
    if (!(sm_scale > 0.f)) return LOCKS_ERR_INVALID_ARG;
  }
  if (crossing && batch > 0) {
    // the pages the current tokens completed: built first, the scorer
    // overlapping all of it but those pages' copies
    LOCKS_CHECK_PTR(k_cache);
    LOCKS_CHECK_PTR(block_table);
    LOCKS_CHECK_PTR(seq_lens);
    LOCKS_CHECK_PTR(summaries);
    LOCKS_CHECK_PTR(workspace);
    BuildParams bp{};
    bp.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
    bp.summ = static_cast<uint8_t*>(summaries);
    bp.status = status_word(workspace);
    bp.num_blocks = num_blocks;
    bp.n_build = batch;
    bp.H_kv = cfg->num_kv_heads;
    bp.block_table = block_table;
    bp.seq_lens = seq_lens;
    bp.max_pages = max_pages;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = cfg->quant == 0 ? launch_build_debug(bp, cfg->rank, s) : launch_build_pages(bp, s);
    if (e != cudaSuccess) return LOCKS_ERR_CUDA;
  }
  locks_status st = score_impl(cfg, q, summaries, num_blocks, block_table, seq_lens, batch, max_pages, scores,
                               workspace, workspace_bytes, stream, crossing);
  if (st != LOCKS_OK) return st;
  // One cluster per (request, KV head): when they all fit on the GPU at once
  // the fused kernel keeps the selection on chip; with more units its
  // latency-bound clusters would run in many waves, so the selection kernel
  // (small CTAs, many resident per SM) and the split-K attention run instead,
  // each a programmatic dependent of the kernel before it.  Past 32,768 pages
  // a fused CTA's slice (4,096+ keys) and its attention share make the
  // separate path faster too: one request at 1M tokens takes 133.3 us that
  // way against 137.7 us fused (equal at 512K, fused ahead below).
  if ((int64_t)batch * cfg->num_kv_heads * kSelCluster <= num_sms() && max_pages <= kFusedStepMaxPages)
    return locks_select_sparse_decode(cfg, q, k_cache, v_cache, num_blocks, block_table, seq_lens, batch, max_pages,
                                      budget_pages, scores, selected, n_selected, sm_scale, out, workspace,
                                      workspace_bytes, stream);
  st = locks_select(cfg, seq_lens, batch, max_pages, budget_pages, scores, selected, n_selected, workspace,
                    workspace_bytes, stream);
  if (st != LOCKS_OK) return st;
  return locks_sparse_decode(cfg, q, k_cache, v_cache, num_blocks, block_table, seq_lens, selected, n_selected,
                             batch, max_pages, budget_pages, sm_scale, out, workspace, workspace_bytes, stream);
}

}  // namespace

extern "C" {

locks_status locks_decode_step(const locks_cfg* cfg, const void* q, const void* summaries, const void* k_cache,
                               const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                               const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t budget_pages,
                               float sm_scale, float* scores, int32_t* selected, int32_t* n_selected, float* out,
                               void* workspace, size_t workspace_bytes, locks_stream_t stream) {
  return decode_step_impl(cfg, q, const_cast<void*>(summaries), k_cache, v_cache, num_blocks, block_table,
                          seq_lens, batch, max_pages, budget_pages, sm_scale, scores, selected, n_selected, out,
                          workspace, workspace_bytes, stream, false);
}

locks_status locks_decode_step_crossing(const locks_cfg* cfg, const void* q, void* summaries, const void* k_cache,
                                        const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                                        const int32_t* seq_lens, int32_t batch, int32_t max_pages,
                                        int32_t budget_pages, float sm_scale, float* scores, int32_t* selected,
                                        int32_t* n_selected, float* out, void* workspace, size_t workspace_bytes,
                                        locks_stream_t stream) {
  return decode_step_impl(cfg, q, summaries, k_cache, v_cache, num_blocks, block_table, seq_lens, batch,
                          max_pages, budget_pages, sm_scale, scores, selected, n_selected, out, workspace,
                          workspace_bytes, stream, true);
}

locks_status locks_score_select(const locks_cfg* cfg, const void* q, const void* summaries,
                                int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                                int32_t batch, int32_t max_pages, int32_t budget_pages, float* scores,
                                int32_t* selected, int32_t* n_selected, void* workspace,
                                size_t workspace_bytes, locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (budget_pages < 0) return LOCKS_ERR_INVALID_ARG;
  if (batch > 0) {
    LOCKS_CHECK_PTR(n_selected);
    if (budget_pages > 0) LOCKS_CHECK_PTR(selected);
  }
  locks_status st = locks_score(cfg, q, summaries, num_blocks, block_table, seq_lens, batch, max_pages,
                                scores, workspace, workspace_bytes, stream);
  if (st != LOCKS_OK) return st;
  return locks_select(cfg, seq_lens, batch, max_pages, budget_pages, scores, selected, n_selected,
                      workspace, workspace_bytes, stream);
}

locks_status locks_sparse_decode(const locks_cfg* cfg, const void* q, const void* k_cache,
                                 const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                                 const int32_t* seq_lens, const int32_t* selected,
                                 const int32_t* n_selected, int32_t batch, int32_t max_pages,
                                 int32_t budget_pages, float sm_scale, float* out, void* workspace,
                                 size_t workspace_bytes, locks_stream_t stream) {
  return attention_common(cfg, q, k_cache, v_cache, num_blocks, block_table, seq_lens, selected, n_selected,
                          batch, max_pages, budget_pages, sm_scale, out, workspace, workspace_bytes,
                          reinterpret_cast<cudaStream_t>(stream), false);
}

locks_status locks_dense_decode(const locks_cfg* cfg, const void* q, const void* k_cache,
                                const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                                const int32_t* seq_lens, int32_t batch, int32_t max_pages, float sm_scale,
                                float* out, void* workspace, size_t workspace_bytes, locks_stream_t stream) {
  return attention_common(cfg, q, k_cache, v_cache, num_blocks, block_table, seq_lens, nullptr, nullptr,
                          batch, max_pages, 0, sm_scale, out, workspace, workspace_bytes,
                          reinterpret_cast<cudaStream_t>(stream), true);
}

// ---------------------------------------------------------------- shared-basis ablation
locks_status locks_shared_basis_build(const locks_cfg* cfg, const void* k_cache, int64_t num_blocks,
                                      const int32_t* block_ids, int32_t n_build, const float* basis, int32_t rho,
                                      void* records, void* workspace, size_t workspace_bytes,
                                      locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (n_build < 0 || num_blocks < 1 || rho < 1 || rho > 64) return LOCKS_ERR_INVALID_ARG;
  if (n_build == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(k_cache);
  LOCKS_CHECK_PTR(block_ids);
  LOCKS_CHECK_PTR(basis);
  LOCKS_CHECK_PTR(records);
  if (workspace != nullptr && (!aligned16(workspace) || workspace_bytes < sizeof(uint32_t)))
    return LOCKS_ERR_INVALID_ARG;
  return from_cuda(launch_shared_basis_build(static_cast<const __nv_bfloat16*>(k_cache), num_blocks, block_ids,
                                             n_build, cfg->num_kv_heads, basis, rho,
                                             static_cast<uint8_t*>(records), status_word(workspace),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

locks_status locks_shared_basis_score(const locks_cfg* cfg, const void* q, const float* basis, int32_t rho,
                                      const void* records, int64_t num_blocks, const int32_t* block_table,
                                      const int32_t* seq_lens, int32_t batch, int32_t max_pages, float* scores,
                                      void* workspace, size_t workspace_bytes, locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || num_blocks < 1 || rho < 1 || rho > 64) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(q);
  LOCKS_CHECK_PTR(basis);
  LOCKS_CHECK_PTR(records);
  LOCKS_CHECK_PTR(block_table);
  LOCKS_CHECK_PTR(seq_lens);
  LOCKS_CHECK_PTR(workspace);
  if (scores != nullptr && !aligned16(scores)) return LOCKS_ERR_INVALID_ARG;
  const Plan pl = make_plan(cfg, batch, max_pages, 0);
  if (workspace_bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  float* sc = scores ? scores : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.off_scores);
  return from_cuda(launch_shared_basis_score(static_cast<const __nv_bfloat16*>(q), basis, rho,
                                             static_cast<const uint8_t*>(records), num_blocks, block_table, seq_lens,
                                             batch, cfg->num_kv_heads, max_pages, sc, status_word(workspace),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- context-parallel shards
locks_status locks_cp_score_pairs(const locks_cfg* cfg, const int32_t* shard_lens, int32_t batch, int32_t max_pages,
                                  const float* scores, float* pairs, void* workspace, size_t workspace_bytes,
                                  locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(shard_lens);
  LOCKS_CHECK_PTR(pairs);
  LOCKS_CHECK_PTR(workspace);
  if (scores != nullptr && !aligned16(scores)) return LOCKS_ERR_INVALID_ARG;
  const Plan pl = make_plan(cfg, batch, max_pages, 0);
  if (workspace_bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  const float* sc = scores ? scores : reinterpret_cast<const float*>(static_cast<uint8_t*>(workspace) + pl.off_scores);
  return from_cuda(launch_cp_pairs(shard_lens, sc, pairs, status_word(workspace), batch * cfg->num_kv_heads,
                                   cfg->num_kv_heads, max_pages, reinterpret_cast<cudaStream_t>(stream)));
}

locks_status locks_cp_select_local(const locks_cfg* cfg, const int32_t* shard_lens, const int32_t* page_offset,
                                   int32_t batch, int32_t max_pages, int32_t budget_pages, const float* scores,
                                   const float* pairs_all, int32_t n_shards, int32_t* cand_pages, uint32_t* cand_keys,
                                   int32_t* cand_counts, void* workspace, size_t workspace_bytes,
                                   locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages < 1 || budget_pages < 0 || n_shards < 1) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(shard_lens);
  LOCKS_CHECK_PTR(page_offset);
  LOCKS_CHECK_PTR(pairs_all);
  LOCKS_CHECK_PTR(cand_counts);
  LOCKS_CHECK_PTR(workspace);
  if (budget_pages > 0) {
    LOCKS_CHECK_PTR(cand_pages);
    LOCKS_CHECK_PTR(cand_keys);
  }
  if (scores != nullptr && !aligned16(scores)) return LOCKS_ERR_INVALID_ARG;
  if (!cp_merge_fits(n_shards, budget_pages)) return LOCKS_ERR_UNSUPPORTED;
  if ((max_pages + kSelCluster - 1) / kSelCluster > kFusedMaxKeysPerCta ||
      select_smem_bytes(max_pages, budget_pages) > (size_t)kSmemLimit)
    return LOCKS_ERR_UNSUPPORTED;
  const Plan pl = make_plan(cfg, batch, max_pages, budget_pages);
  if (workspace_bytes < pl.total) return LOCKS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  SelectParams p{};
  fill_select(p, pl, cfg, shard_lens, batch, max_pages, budget_pages, scores, cand_pages, cand_counts, workspace);
  p.zpairs = pairs_all;
  p.z_shards = n_shards;
  const int units = batch * cfg->num_kv_heads;
  const int cluster = select_cluster(units, max_pages, budget_pages);
  p.stage_scores = 0;
  cudaError_t e = launch_select(p, units, cluster, s);
  if (e != cudaSuccess || budget_pages == 0) return from_cuda(e);
  return from_cuda(launch_cp_candidates(p.scores, pairs_all, n_shards, page_offset, cand_pages, cand_keys,
                                        cand_counts, units, cfg->num_kv_heads, max_pages, budget_pages, s));
}

locks_status locks_cp_merge_select(const locks_cfg* cfg, const int32_t* page_offset, int32_t batch,
                                   int32_t budget_pages, int32_t n_shards, int32_t shard,
                                   const int32_t* cand_pages_all, const uint32_t* cand_keys_all,
                                   const int32_t* cand_counts_all, int32_t* selected, int32_t* n_selected,
                                   locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || budget_pages < 0 || n_shards < 1 || shard < 0 || shard >= n_shards) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  if (!cp_merge_fits(n_shards, budget_pages)) return LOCKS_ERR_UNSUPPORTED;
  LOCKS_CHECK_PTR(page_offset);
  LOCKS_CHECK_PTR(cand_counts_all);
  LOCKS_CHECK_PTR(n_selected);
  if (budget_pages > 0) {
    LOCKS_CHECK_PTR(cand_pages_all);
    LOCKS_CHECK_PTR(cand_keys_all);
    LOCKS_CHECK_PTR(selected);
  }
  return from_cuda(launch_cp_merge_select(cand_pages_all, cand_keys_all, cand_counts_all, n_shards, shard,
                                          page_offset, selected, n_selected, batch * cfg->num_kv_heads,
                                          cfg->num_kv_heads, budget_pages, reinterpret_cast<cudaStream_t>(stream)));
}

locks_status locks_cp_sparse_decode_partial(const locks_cfg* cfg, const void* q, const void* k_cache,
                                            const void* v_cache, int64_t num_blocks, const int32_t* block_table,
                                            const int32_t* shard_lens, const int32_t* selected,
                                            const int32_t* n_selected, int32_t batch, int32_t max_pages,
                                            int32_t budget_pages, float sm_scale, float* states, void* workspace,
                                            size_t workspace_bytes, locks_stream_t stream) {
  if (states == nullptr || !aligned16(states)) return LOCKS_ERR_INVALID_ARG;
  return attention_common(cfg, q, k_cache, v_cache, num_blocks, block_table, shard_lens, selected, n_selected,
                          batch, max_pages, budget_pages, sm_scale, nullptr, workspace, workspace_bytes,
                          reinterpret_cast<cudaStream_t>(stream), false, states);
}

locks_status locks_cp_merge_attention(const locks_cfg* cfg, int32_t batch, int32_t n_shards, const float* states_all,
                                      float* out, locks_stream_t stream) {
  if (!cfg_supported(cfg)) return cfg == nullptr ? LOCKS_ERR_INVALID_ARG : LOCKS_ERR_UNSUPPORTED;
  if (batch < 0 || n_shards < 1) return LOCKS_ERR_INVALID_ARG;
  if (batch == 0) return LOCKS_OK;
  LOCKS_CHECK_PTR(states_all);
  LOCKS_CHECK_PTR(out);
  return from_cuda(launch_cp_merge_attn(states_all, n_shards, batch * cfg->num_kv_heads * kGroup, out,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

const char* locks_status_str(locks_status s) {
  switch (s) {
    case LOCKS_OK: return "ok";
    case LOCKS_ERR_INVALID_ARG: return "invalid argument";
    case LOCKS_ERR_UNSUPPORTED: return "unsupported configuration";
    case LOCKS_ERR_WORKSPACE: return "workspace too small";
    case LOCKS_ERR_CUDA: return "CUDA error";
    case LOCKS_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
