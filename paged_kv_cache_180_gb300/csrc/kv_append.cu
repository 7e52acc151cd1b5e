// kv_append: scatter each new token's K and V rows into the page and row its slot names.
//
// Write side of the paged cache ("tiny-vllm part 3: the prefill path", section
// "Distributing K/V into paged blocks": a token's logical block is token / 16,
// its physical block comes from the block table, K goes to the block's K area
// and V to its V area; samir-vllm README, "What works so far": decode appends
// one new token at its absolute position).  Here the caller has already turned
// (block table, position) into slot = page * 16 + row, and one kernel writes all
// tokens of a step at once instead of two device-to-device copies per block.
//
// Layout written: [page][kv_head][row][dim] in each of the K and V areas.
#include <cuda_runtime.h>

#include "host_common.h"
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kChunksPerRow = kRowBytes / 16;                 // 8 x 16 B per (head, token) row
constexpr int kChunksPerThread = 4;                           // one thread moves half a row (64 B)
constexpr int kThreadsPerToken = 2 * kKvHeads * kChunksPerRow / kChunksPerThread;  // K and V: 32
constexpr int kAppendThreads = 256;

// One thread moves 4 consecutive 16-byte chunks: token i, K or V, kv head g, half h of the
// row (the four loads are in flight together).
__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(
    uint8_t *__restrict__ k_base, uint8_t *__restrict__ v_base, long long page_stride, long long num_slots,
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, const int32_t *__restrict__ slot_mapping,
    int num_tokens, int32_t *status) {
  // a kernel launched after this one with PKV_OVERLAP_PREVIOUS may start its set-up now (it
  // reads the pool only once this kernel has completed)
  griddep_launch_dependents();
  const long long idx = (long long)blockIdx.x * kAppendThreads + threadIdx.x;
  const long long token = idx / kThreadsPerToken;
  if (token >= num_tokens) return;
  const int r = int(idx % kThreadsPerToken);
  const int is_v = r / (kThreadsPerToken / 2);
  const int g = (r / 2) % kKvHeads;
  const int h = r % 2;
  const long long slot = slot_mapping[token];
  if (slot < 0) return;  // padding
  if (slot >= num_slots) {
    if (r == 0) report(status, PKV_DEV_BAD_SLOT);
    return;
  }
  const long long page = slot / kPageTokens;
  const int row = int(slot % kPageTokens);
  const uint4 *src = (is_v ? v_new : k_new) + (token * kKvHeads + g) * kChunksPerRow + h * kChunksPerThread;
  uint4 *dst = reinterpret_cast<uint4 *>((is_v ? v_base : k_base) + page * page_stride +
                                         (long long)(g * kPageTokens + row) * kRowBytes) +
               h * kChunksPerThread;
  uint4 x[kChunksPerThread];
#pragma unroll
  for (int c = 0; c < kChunksPerThread; ++c) x[c] = __ldg(src + c);
#pragma unroll
  for (int c = 0; c < kChunksPerThread; ++c) dst[c] = x[c];
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_kv_append(const pkv_pool *pool, const void *k_new, const void *v_new,
                             const int32_t *slot_mapping, int num_tokens, int32_t *device_status, void *stream) {
  const int rc = pkv::check_pool(pool);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return PKV_ERR_NULL;
  if (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3u))
    return PKV_ERR_ALIGN;
  const long long threads = (long long)num_tokens * pkv::kThreadsPerToken;
  const long long blocks = (threads + pkv::kAppendThreads - 1) / pkv::kAppendThreads;
  if (blocks > 0x7fffffffLL) return PKV_ERR_SHAPE;
  pkv::kv_append_kernel<<<unsigned(blocks), pkv::kAppendThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t *>(pool->k_base), static_cast<uint8_t *>(pool->v_base), pool->page_stride_bytes,
      (long long)pool->num_pages * pool->page_tokens, static_cast<const uint4 *>(k_new),
      static_cast<const uint4 *>(v_new), slot_mapping, num_tokens, device_status);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}
