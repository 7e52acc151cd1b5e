// TMA tensor maps of a page pool (host only), shared by the decode and prefill kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.h"
#include "pkv.h"

namespace pkv {
namespace {

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map of the K (or V) halves of a pool: element (d, row, page) with row =
// kv_head * page_tokens + token, row stride 2 * head_dim bytes, page stride
// page_stride_bytes; one box is box_rows rows of one page (64 x box_rows x 1),
// delivered 128-byte swizzled.
int encode_half_pages(CUtensorMap *map, const pkv_pool *pool, const void *base, int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return PKV_ERR_CUDA;
  const int rows = pool->num_kv_heads * pool->page_tokens;
  const cuuint64_t dims[3] = {cuuint64_t(pool->head_dim), cuuint64_t(rows), cuuint64_t(pool->num_pages)};
  const cuuint64_t strides[2] = {cuuint64_t(pool->head_dim) * 2u, cuuint64_t(pool->page_stride_bytes)};
  const cuuint32_t box[3] = {cuuint32_t(pool->head_dim), cuuint32_t(box_rows), 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

// Tensor map of prefill queries q[rows][num_q_heads][head_dim] (bf16): element (d, head, row),
// one box = head_dim x box_heads x box_rows, 128-byte swizzled; rows past `rows` read as zeros.
// Cached by address and shape (the encoding costs host time on every call otherwise).
int query_tensor_map(const void *q, int rows, int num_q_heads, int head_dim, int box_heads, int box_rows,
                     CUtensorMap *map) {
  struct Entry {
    const void *q;
    int rows, heads, dim, bh, br;
    CUtensorMap m;
  };
  constexpr int kEntries = 16;
  static std::mutex mu;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  if (rows <= 0 || num_q_heads <= 0 || head_dim <= 0 || box_heads <= 0 || box_rows <= 0 || box_rows > 256 ||
      box_heads > num_q_heads || head_dim * 2 > 128)
    return PKV_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    const Entry &e = cache[i];
    if (e.q == q && e.rows == rows && e.heads == num_q_heads && e.dim == head_dim && e.bh == box_heads &&
        e.br == box_rows) {
      *map = e.m;
      return PKV_OK;
    }
  }
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return PKV_ERR_CUDA;
  Entry e;
  e.q = q;
  e.rows = rows;
  e.heads = num_q_heads;
  e.dim = head_dim;
  e.bh = box_heads;
  e.br = box_rows;
  const cuuint64_t dims[3] = {cuuint64_t(head_dim), cuuint64_t(num_q_heads), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(head_dim) * 2u, cuuint64_t(num_q_heads) * cuuint64_t(head_dim) * 2u};
  const cuuint32_t box[3] = {cuuint32_t(head_dim), cuuint32_t(box_heads), cuuint32_t(box_rows)};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUresult r = fn(&e.m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return PKV_ERR_CUDA;
  cache[next] = e;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  *map = e.m;
  return PKV_OK;
}

// The two tensor maps of a pool for boxes of box_rows rows, from a small cache keyed by
// the pool's addresses and shape (encoding them costs host time on every call otherwise).
int pool_tensor_maps(const pkv_pool *pool, int box_rows, CUtensorMap *tk, CUtensorMap *tv) {
  struct Entry {
    const void *k, *v;
    long long stride;
    int pages, box_rows;
    CUtensorMap mk, mv;
  };
  constexpr int kEntries = 16;
  static std::mutex mu;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  if (box_rows <= 0 || box_rows > 256 || box_rows > pool->num_kv_heads * pool->page_tokens) return PKV_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    const Entry &e = cache[i];
    if (e.k == pool->k_base && e.v == pool->v_base && e.stride == pool->page_stride_bytes &&
        e.pages == pool->num_pages && e.box_rows == box_rows) {
      *tk = e.mk;
      *tv = e.mv;
      return PKV_OK;
    }
  }
  Entry e;
  e.k = pool->k_base;
  e.v = pool->v_base;
  e.stride = pool->page_stride_bytes;
  e.pages = pool->num_pages;
  e.box_rows = box_rows;
  int rc = encode_half_pages(&e.mk, pool, pool->k_base, box_rows);
  if (rc == PKV_OK) rc = encode_half_pages(&e.mv, pool, pool->v_base, box_rows);
  if (rc != PKV_OK) return rc;
  cache[next] = e;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  *tk = e.mk;
  *tv = e.mv;
  return PKV_OK;
}

}  // namespace pkv
