// Pool descriptors and status strings (host only).
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.h"
#include "pkv.h"

namespace pkv {

int device_sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace pkv

extern "C" size_t pkv_kv_pool_bytes(int num_pages, int page_tokens, int num_kv_heads, int head_dim) {
  if (num_pages <= 0 || page_tokens <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return size_t(num_pages) * 2u * size_t(num_kv_heads) * size_t(page_tokens) * size_t(head_dim) * 2u;
}

extern "C" int pkv_kv_pool_create(void *k_pool, void *v_pool, int64_t page_stride_bytes, int num_pages,
                                  int page_tokens, int num_kv_heads, int head_dim, pkv_pool *out) {
  if (out == nullptr || k_pool == nullptr || v_pool == nullptr) return PKV_ERR_NULL;
  if (num_pages <= 0 || page_tokens <= 0 || num_kv_heads <= 0 || head_dim <= 0) return PKV_ERR_SHAPE;
  if (!pkv::supported_geometry(page_tokens, num_kv_heads, head_dim)) return PKV_ERR_UNSUPPORTED;
  const int64_t half = int64_t(num_kv_heads) * page_tokens * head_dim * 2;
  if (page_stride_bytes == 0) page_stride_bytes = 2 * half;
  pkv_pool p;
  p.k_base = k_pool;
  p.v_base = v_pool;
  p.page_stride_bytes = page_stride_bytes;
  p.num_pages = num_pages;
  p.page_tokens = page_tokens;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  const int rc = pkv::check_pool(&p);
  if (rc != PKV_OK) return rc;
  *out = p;
  return PKV_OK;
}

extern "C" const char *pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is null";
    case PKV_ERR_SHAPE: return "a size or count is out of range";
    case PKV_ERR_UNSUPPORTED: return "geometry not compiled in this build (needs page 16, head_dim 64, 8 kv heads, 32 q heads)";
    case PKV_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case PKV_ERR_SCALE: return "scale is not finite";
    case PKV_ERR_WORKSPACE: return "workspace too small";
    case PKV_ERR_LAUNCH: return "kernel launch failed";
    case PKV_ERR_CUDA: return "CUDA runtime call failed";
    case PKV_ERR_EXCEEDS_POOL: return "request page budget exceeds the whole pool";
    case PKV_ERR_NO_PAGE: return "no free page";
    case PKV_ERR_STATE: return "call out of order";
    case PKV_ERR_NO_CREDIT: return "request credits do not fit beside the admitted ones now (wait)";
    case PKV_ERR_NOALLOC_LIMIT: return "num_seqs above PKV_NOALLOC_MAX_SEQS (fixed scratch of the allocation-free entry point)";
    default: return "unknown status";
  }
}
