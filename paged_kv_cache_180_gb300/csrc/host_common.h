// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The one geometry this build compiles.
inline bool supported_geometry(int page_tokens, int num_kv_heads, int head_dim) {
  return page_tokens == 16 && num_kv_heads == 8 && head_dim == 64;
}

// Checks a pool descriptor; PKV_OK or an error code.
inline int check_pool(const pkv_pool *pool) {
  if (pool == nullptr || pool->k_base == nullptr || pool->v_base == nullptr) return PKV_ERR_NULL;
  if (pool->num_pages <= 0) return PKV_ERR_SHAPE;
  if (!supported_geometry(pool->page_tokens, pool->num_kv_heads, pool->head_dim)) return PKV_ERR_UNSUPPORTED;
  const int64_t half = int64_t(pool->num_kv_heads) * pool->page_tokens * pool->head_dim * 2;
  if (pool->page_stride_bytes < half) return PKV_ERR_SHAPE;
  if (!aligned16(pool->k_base) || !aligned16(pool->v_base) || (pool->page_stride_bytes & 15) != 0)
    return PKV_ERR_ALIGN;
  return PKV_OK;
}

// Number of SMs of the current device (cached per device); 0 if it cannot be queried.
int device_sm_count();

// TMA tensor maps of the K and V halves of a checked pool, for boxes of box_rows
// 128-byte rows of one page (128B swizzle); cached per pool.  PKV_OK or an error.
int pool_tensor_maps(const pkv_pool *pool, int box_rows, CUtensorMap *tk, CUtensorMap *tv);

// TMA tensor map of queries q[rows][num_q_heads][head_dim] (bf16) for boxes of
// head_dim x box_heads x box_rows, 128-byte swizzled; cached.  PKV_OK or an error.
int query_tensor_map(const void *q, int rows, int num_q_heads, int head_dim, int box_heads, int box_rows,
                     CUtensorMap *map);

}  // namespace pkv
