// host_plan.h -- host-side rules shared by the entry points of liblocks:
// which configurations are supported, how the split-K sparse attention splits
// a unit's items, and the tensor map of a K/V cache.  Every entry point that
// launches those kernels takes them from here, so the workspace and the
// allocation-free paths validate and plan identically.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "../../include/locks.h"

namespace locks {

// head_dim 128, page 16, rank 8, quantised records, group 4, and a KV-head
// count the scorer's head grouping can tile (1, 2, 4, or a multiple of 8).
bool cfg_supported(const locks_cfg* c);

// Split of a sparse unit's items (budget pages + the tail) over CTAs: one wave
// of resident CTAs for the whole batch, at least one item per warp.
void sparse_split(int64_t units, int budget_pages, int* splits, int* items_per_split);

// 2-D tiled view of a bf16 [num_blocks][H][16][128] cache: rows are page-head
// tokens, 128 columns; boxes of 16 rows x 64 columns, 128-byte swizzle (the
// layout attn_tile.cuh addresses).  False if the driver entry point is missing
// or the encoder rejects the arguments.
bool encode_cache_map(CUtensorMap* map, const void* base, int64_t num_blocks, int H);

}  // namespace locks
