// params.h -- launch parameter blocks shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace locks {

struct ScoreParams {
  const __nv_bfloat16* q;
  const uint8_t* summ;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* scores;      // [batch][H_kv][max_pages][G]
  uint32_t* status;
  int64_t num_blocks;
  int batch, max_pages, H_kv;
  int h_cta;          // KV heads per CTA (<= 8, divides 8)
  int wph;            // warps per head = 8 / h_cta
  int pps;            // pages per stage = 4 * wph
  int ch_pages;       // pages per work item (chunk)
  int n_chunks;       // chunks per (b, head group)
  int head_groups;    // H_kv / h_cta
  int n_items;        // batch * head_groups * n_chunks
  // 1: launched as a programmatic dependent of the crossing build; the page a
  // request's current token completed is copied only after that build ends
  int defer_crossing;
};

struct SelectParams {
  const int32_t* seq_lens;
  const float* scores;
  int32_t* selected;       // [batch][H_kv][budget]
  int32_t* n_selected;     // [batch][H_kv]
  uint32_t* status;
  int batch, max_pages, H_kv, budget;
  int stage_scores;        // 1: each CTA copies its slice of scores to shared memory first
  // context-parallel selection only: Z_g from per-shard (max, sum) pairs
  // [z_shards][batch * H_kv][G] (float2, log2 units) instead of the scores
  const float* zpairs;
  int z_shards;
};

struct AttnParams {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* selected;     // sparse only
  const int32_t* n_selected;   // sparse only
  float* out;
  float* state_out;            // optional: [batch][H_kv*G][2 + 128] unnormalised (m log2, l, o) instead of out
  float* part;                 // [units][splits][G][2 + 128]
  uint32_t* tickets;           // [units]
  uint32_t* status;
  int64_t num_blocks;
  int batch, max_pages, H_kv, budget;
  int splits, items_per_split;
  int dense;
  float scale_log2;            // sm_scale * log2(e)
};

struct BuildParams {
  const __nv_bfloat16* k_cache;
  const int32_t* block_ids;
  const int32_t* n_dev;    // optional device count: build block_ids[0, min(n_build, *n_dev))
  uint8_t* summ;
  uint32_t* status;
  int64_t num_blocks;
  int n_build, H_kv;
  // crossing mode (block_ids unused): request b = page-head / H_kv builds the
  // page its current token completed, page L_b / 16 - 1, when L_b % 16 == 0
  const int32_t* block_table;
  const int32_t* seq_lens;
  int max_pages;
};

struct FusedParams {
  SelectParams sel;
  const __nv_bfloat16* q;
  const int32_t* block_table;
  float* out;                  // [batch][H_kv*G][128]
  int64_t num_blocks;
  float scale_log2;            // sm_scale * log2(e)
};

cudaError_t launch_score(const ScoreParams& p, int grid, cudaStream_t stream, bool programmatic = false);
cudaError_t launch_select_attend(const CUtensorMap& tmk, const CUtensorMap& tmv, const FusedParams& p,
                                 int units, cudaStream_t stream);
size_t fused_smem_bytes(int max_pages, int budget);
// cluster: CTAs per (request, KV head): 1, 2, 4, 8 or 16
cudaError_t launch_select(const SelectParams& p, int units, int cluster, cudaStream_t stream);
int select16_max_clusters(size_t dyn, bool staged);
cudaError_t launch_attn(const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p,
                        cudaStream_t stream);
cudaError_t launch_build(const BuildParams& p, cudaStream_t stream);
// the same records from one CTA a page-head: for a step's few new pages
cudaError_t launch_build_pages(const BuildParams& p, cudaStream_t stream);
// unquantised fp32 records of rank r <= 16 (cfg quant = 0)
cudaError_t launch_build_debug(const BuildParams& p, int rank_r, cudaStream_t stream);
cudaError_t launch_score_debug(const ScoreParams& p, int rank_r, cudaStream_t stream);
// shared-basis ablation (shared_basis.cu)
cudaError_t launch_shared_basis_build(const __nv_bfloat16* k_cache, int64_t num_blocks, const int32_t* block_ids,
                                      int n_build, int H, const float* basis, int rho, uint8_t* records,
                                      uint32_t* status, cudaStream_t stream);
cudaError_t launch_shared_basis_score(const __nv_bfloat16* q, const float* basis, int rho, const uint8_t* records,
                                      int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                                      int batch, int H, int max_pages, float* scores, uint32_t* status,
                                      cudaStream_t stream);

// context-parallel shards (context_parallel.cu)
cudaError_t launch_cp_pairs(const int32_t* shard_lens, const float* scores, float* pairs, uint32_t* status,
                            int units, int H, int max_pages, cudaStream_t stream);
cudaError_t launch_cp_candidates(const float* scores, const float* zpairs, int n_shards, const int32_t* page_offset,
                                 int32_t* pages, uint32_t* keys, const int32_t* counts, int units, int H,
                                 int max_pages, int budget, cudaStream_t stream);
bool cp_merge_fits(int n_shards, int budget);
cudaError_t launch_cp_merge_select(const int32_t* cand_pages, const uint32_t* cand_keys, const int32_t* cand_counts,
                                   int n_shards, int shard, const int32_t* page_offset, int32_t* selected,
                                   int32_t* n_selected, int units, int H, int budget, cudaStream_t stream);
cudaError_t launch_cp_merge_attn(const float* states, int n_shards, int rows, float* out, cudaStream_t stream);

}  // namespace locks
