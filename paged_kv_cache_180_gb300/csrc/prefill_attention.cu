// Paged prefill (and chunked prefill) attention: the last n_s tokens of each
// sequence attend causally over its cached K/V, read page by page through its
// block table, with grouped-query heads.
//
// What is computed ("tiny-vllm part 3: the prefill path", sections "Per-head
// attention scores and GQA" and "causalMask and online softmax": per query head
// h, scores q_i . K_t / sqrt(64) against K/V head h / 4, future tokens masked,
// softmax, times V - here read from the pages instead of contiguous buffers, with
// the softmax evaluated online):
//
//   out[i][h] = sum_{t <= p_i} softmax_t(scale * q[i][h] . K_t[h/4]) V_t[h/4],
//   p_i = context_lens[s] - n_s + (i - query_start[s])
//
// GB300 design (tcgen05 tensor cores, accumulators in tensor memory)
//  * Tile: one CTA per (32 query tokens of a sequence, K/V head g).  Its 128 rows
//    (row = 4 * token + head in group) share every K/V row it loads: M = 128.
//    Tiles are numbered latest-first over the whole grid, so the longest causal
//    spans start first.
//  * Keys in blocks of 64 (4 pages).  S = Q K^T is 4 tcgen05.mma (M 128, N 64,
//    K 16 each; Q and K K-major, 128-byte swizzled) into one of two TMEM
//    buffers, so S of block j + 1 runs while the softmax reads block j.
//    O += P V is 8 tcgen05.mma into a TMEM accumulator: P is split into bf16
//    hi + lo halves (weights keep ~16 significant bits), both multiplied by the
//    same V tile (MN-major, 128-byte swizzled).
//  * Warp roles: warps 0-3 own one row each per thread (TMEM lane = row): they
//    load Q, read S from TMEM, mask, keep the row's running max and sum, write P
//    to shared memory and finally read O, divide and store.  Warp 4 streams head
//    g's K and V rows of each page with tiled TMA (2 KiB boxes) into a 3-stage
//    ring; pages past the query span are loaded from a coordinate outside the
//    pool, which TMA fills with zeros.  Warp 5 owns the TMEM allocation and
//    issues the MMAs (one thread), completion signalled by tcgen05.commit.
//  * Online softmax in the exp2 domain with a lazily moved maximum: a row's
//    reference maximum moves only when a block's maximum exceeds it by more than
//    8 (a factor 256), and only then is the row of O in TMEM rescaled (after the
//    previous P V completed).  The final division by the row sum uses the same
//    reference, so the result is the exact softmax up to rounding.
//  * Masks: key t counts for a row at position p when t <= p (p < ctx); other
//    scores become -inf.  V rows at or past the context in a sequence's last page
//    are zeroed in shared memory so stale pool bytes (even NaN) never reach O.
//  * Every mbarrier wait is bounded (about 2 s): on expiry the CTA reports
//    PKV_DEV_TIMEOUT, stops issuing work, waits (bounded) for what is in flight,
//    frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>

#include "host_common.h"
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kPfTok = 32;                             // query tokens per CTA
constexpr int kPfRows = kPfTok * kGroup;               // M = 128
constexpr int kPfKeys = 64;                            // keys per block
constexpr int kPfPagesPerBlock = kPfKeys / kPageTokens;
constexpr int kPfStages = 3;
constexpr int kPfThreads = 192;                        // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int kPfBox = kPageTokens * kRowBytes;        // one head's rows of one page: 2 KiB
constexpr int kPfTileBytes = kPfKeys * kRowBytes;      // K (or V) of one block: 8 KiB
constexpr uint32_t kPfTmemCols = 256;
constexpr uint32_t kColS = 0;                          // S buffers at columns 0 and 64
constexpr uint32_t kColO = 128;                        // O accumulator: columns 128 .. 191
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;                    // move a row's reference max when exceeded by more

constexpr uint32_t kIdescS = idesc_bf16(kPfRows, kPfKeys, false);   // B = K rows (K-major)
constexpr uint32_t kIdescPV = idesc_bf16(kPfRows, kHeadDim, true);  // B = V rows (MN-major)

struct PrefillArgs {
  CUtensorMap tmap_k;  // boxes of one head's 16 rows of one page
  CUtensorMap tmap_v;
  int num_pages;
  const uint4 *q;  // [total][32][64] bf16, 8 uint4 per head row
  float *out;      // [total][32][64]
  const int32_t *query_start;
  const int32_t *block_tables;
  long long bt_stride;
  const int32_t *context_lens;
  int num_seqs;
  int max_context;
  int tiles_per_seq;
  float scale_log2;
  int32_t *status;
};

struct __align__(1024) PfSmem {
  uint8_t q[kPfRows * kRowBytes];          // 16 KiB, row = 4 * token + head, 128-byte swizzled
  uint8_t k[kPfStages][kPfTileBytes];      // 64 keys x 128 B per stage
  uint8_t v[kPfStages][kPfTileBytes];
  uint8_t p_hi[kPfRows * kRowBytes];       // P of the current block: 128 rows x 64 keys bf16
  uint8_t p_lo[kPfRows * kRowBytes];
  uint64_t q_full;
  uint64_t kv_full[kPfStages];
  uint64_t kv_empty[kPfStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t p_free;  // P V of a block done (P buffer and O free)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kPfSmemBytes = sizeof(PfSmem) + 1024;

// Bounded wait that gives up at once when another role has already aborted.
// Returns true when the phase completed.
__device__ __forceinline__ bool pf_wait(PfSmem &sm, uint64_t *bar, uint32_t parity, int32_t *status) {
  if (*reinterpret_cast<volatile int *>(&sm.abort)) return false;
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int *>(&sm.abort) = 1;
  report(status, PKV_DEV_TIMEOUT);
  return false;
}

// Writes 8 16-byte chunks as row r of a 128-byte-swizzled tile.
__device__ __forceinline__ void put_row_sw128(uint8_t *tile, int r, const uint4 (&c)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(tile + r * kRowBytes + ((i ^ (r & 7)) << 4)) = c[i];
}

__global__ void __launch_bounds__(kPfThreads, 2) paged_prefill_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  PfSmem &sm = *reinterpret_cast<PfSmem *>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // tile rank r (latest tiles first over the grid), then sequence, then K/V head
  const int per_rank = a.num_seqs * kKvHeads;
  const int rank = int(blockIdx.x) / per_rank, rem = int(blockIdx.x) % per_rank;
  const int s = rem / kKvHeads, g = rem % kKvHeads;
  const int tile = a.tiles_per_seq - 1 - rank;
  const int q0 = __ldg(a.query_start + s);
  const int n = __ldg(a.query_start + s + 1) - q0;
  const int ctx = __ldg(a.context_lens + s);
  const int t0 = tile * kPfTok;
  if (n <= 0 || t0 >= n) return;
  const int tend = min(t0 + kPfTok, n);
  if (ctx < 0 || ctx > a.max_context || n > ctx) {
    // invalid sequence: zero this CTA's rows (its tokens, query heads 4g .. 4g+3)
    if (tile == 0 && g == 0 && tid == 0) report(a.status, PKV_DEV_BAD_CONTEXT);
    for (int k = tid; k < (tend - t0) * kGroup * kHeadDim; k += kPfThreads) {
      const int tok = t0 + k / (kGroup * kHeadDim), r = k % (kGroup * kHeadDim);
      a.out[((long long)(q0 + tok) * kQHeads + g * kGroup) * kHeadDim + r] = 0.f;
    }
    return;
  }
  const int base_pos = ctx - n;                         // position of query token 0
  const int last_pos = base_pos + tend - 1;             // latest position in this tile
  const int nblocks = last_pos / kPfKeys + 1;
  const int npages = last_pos / kPageTokens + 1;        // pages holding keys 0 .. last_pos
  const int32_t *table = a.block_tables + (long long)s * a.bt_stride;

  if (tid == 0) {
    mbar_init(&sm.q_full, 128);
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_free[b], 128);
    }
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.p_free, 1);
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    mbar_init_fence();
  }
  if (warp == 5) tmem_alloc(&sm.tmem_base, kPfTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 4) {
    // ================= TMA producer: head g's K and V rows, 4 pages per block =================
    if (lane == 0) {
      const uint64_t policy = policy_evict_last();
      prefetch_tensormap(&a.tmap_k);
      prefetch_tensormap(&a.tmap_v);
      int issued = 0;
      for (int j = 0; j < nblocks; ++j) {
        const int st = j % kPfStages;
        if (j >= kPfStages && !pf_wait(sm, &sm.kv_empty[st], uint32_t(j / kPfStages - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kPfTileBytes);
        for (int pp = 0; pp < kPfPagesPerBlock; ++pp) {
          const int lp = j * kPfPagesPerBlock + pp;
          int page = -1;  // outside the pool: TMA fills the box with zeros
          if (lp < npages) {
            page = __ldg(table + lp);
            if (page < 0 || page >= a.num_pages) {
              report(a.status, PKV_DEV_BAD_PAGE);
              page = -1;
            }
          }
          tma_load_3d(sm.k[st] + pp * kPfBox, &a.tmap_k, 0, g * kPageTokens, page, &sm.kv_full[st], policy);
          tma_load_3d(sm.v[st] + pp * kPfBox, &a.tmap_v, 0, g * kPageTokens, page, &sm.kv_full[st], policy);
        }
        issued = j + 1;
      }
      // every copy issued has landed before the CTA exits
      for (int j = max(0, issued - kPfStages); j < issued; ++j)
        mbar_wait(&sm.kv_full[j % kPfStages], uint32_t(j / kPfStages) & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ================= MMA issuer =================
    const uint32_t q_base = smem_addr(sm.q), phi = smem_addr(sm.p_hi), plo = smem_addr(sm.p_lo);
    bool ok = pf_wait(sm, &sm.q_full, 0, a.status);
    ok = __all_sync(0xffffffffu, ok);
    auto issue_pv = [&](int i) {
      bool w = pf_wait(sm, &sm.p_full, uint32_t(i) & 1, a.status);
      w = __all_sync(0xffffffffu, w);
      if (!w) return false;
      tc_fence_after();
      if (lane == 0) {
        const int st = i % kPfStages;
        const uint32_t vb = smem_addr(sm.v[st]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tmem + kColO, sw128_desc(phi + kk * 32, 16, 1024), sw128_desc(vb + kk * 2048, 1024, 1024), kIdescPV,
                 (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tmem + kColO, sw128_desc(plo + kk * 32, 16, 1024), sw128_desc(vb + kk * 2048, 1024, 1024), kIdescPV,
                 1u);
        tc_commit(&sm.p_free);
        tc_commit(&sm.kv_empty[st]);
      }
      __syncwarp();
      return true;
    };
    for (int j = 0; ok && j < nblocks; ++j) {
      const int st = j % kPfStages, b = j & 1;
      bool w = pf_wait(sm, &sm.kv_full[st], uint32_t(j / kPfStages) & 1, a.status);
      w = __all_sync(0xffffffffu, w);
      if (!w) break;
      // V rows at or past the context (stale pool bytes) in this block become zeros
      const int z0 = max(ctx, j * kPfKeys), z1 = min(npages * kPageTokens, (j + 1) * kPfKeys);
      if (z0 < z1) {
        uint8_t *vt = sm.v[st];
        for (int idx = lane; idx < (z1 - z0) * 8; idx += 32)
          *reinterpret_cast<uint4 *>(vt + (z0 - j * kPfKeys + idx / 8) * kRowBytes + (idx % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (j >= 2) {
        w = pf_wait(sm, &sm.s_free[b], uint32_t(j / 2 - 1) & 1, a.status);
        w = __all_sync(0xffffffffu, w);
        if (!w) break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kb = smem_addr(sm.k[st]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tmem + kColS + b * kPfKeys, sw128_desc(q_base + kk * 32, 16, 1024), sw128_desc(kb + kk * 32, 16, 1024),
                 kIdescS, kk > 0 ? 1u : 0u);
        tc_commit(&sm.s_full[b]);
      }
      __syncwarp();
      if (j >= 1 && !issue_pv(j - 1)) {
        ok = false;
        break;
      }
      if (j == nblocks - 1 && !issue_pv(j)) ok = false;
    }
    // every MMA issued has completed before the tensor memory is freed
    if (lane == 0) {
      tc_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0);
    }
    __syncwarp();
  } else {
    // ================= softmax warps: thread = row = 4 * token + head =================
    const int r = tid, tok = r >> 2, hh = r & 3;
    {
      // Q row (a padding row past n repeats the last real token; it is not written)
      const uint4 *src = a.q + ((long long)(q0 + min(t0 + tok, n - 1)) * kQHeads + g * kGroup + hh) * 8;
      uint4 c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = __ldg(src + i);
      put_row_sw128(sm.q, r, c);
      fence_proxy_async_smem();
      mbar_arrive(&sm.q_full);
    }
    const int pos = base_pos + min(t0 + tok, n - 1);
    const uint32_t lane_base = tmem + (uint32_t(32 * warp) << 16);
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < nblocks; ++j) {
      const int b = j & 1;
      bool w = pf_wait(sm, &sm.s_full[b], uint32_t(j >> 1) & 1, a.status);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[64];
      {
        uint32_t x0[32], x1[32];
        tmem_ld32(lane_base + kColS + b * kPfKeys, x0);
        tmem_ld32(lane_base + kColS + b * kPfKeys + 32, x1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          sv[c] = x0[c];
          sv[32 + c] = x1[c];
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.s_free[b]);
      // scores in log2 units; keys after this row's position, and the keys of
      // invalid pages (loaded as zeros), are masked
      const int key0 = j * kPfKeys;
      int bad = 0;
#pragma unroll
      for (int pp = 0; pp < kPfPagesPerBlock; ++pp) {
        const int lp = j * kPfPagesPerBlock + pp;
        if (lp < npages) {
          const int page = __ldg(table + lp);
          if (page < 0 || page >= a.num_pages) bad |= 1 << pp;
        }
      }
      float x[64];
      float mx = -INFINITY;
      if (key0 + kPfKeys - 1 <= pos && bad == 0) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          x[c] = __uint_as_float(sv[c]) * a.scale_log2;
          mx = fmaxf(mx, x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          x[c] = (key0 + c <= pos && !((bad >> (c / kPageTokens)) & 1)) ? __uint_as_float(sv[c]) * a.scale_log2
                                                                          : -INFINITY;
          mx = fmaxf(mx, x[c]);
        }
      }
      // move the reference max only when this block's max exceeds it by more than 2^8
      const bool move = mx > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (move) {
        alpha = exp2f(m_ref - mx);  // 0 for the first block (m_ref = -inf)
        m_ref = mx;
        l_sum *= alpha;
      }
      float psum = 0.f;
      uint4 hi[8], lo[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t h4[4], l4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = exp2f(x[8 * c + 2 * e] - m_ref), p1 = exp2f(x[8 * c + 2 * e + 1] - m_ref);
          psum += p0 + p1;
          h4[e] = pack_bf16x2(p0, p1);
          l4[e] = pack_bf16x2(p0 - bf16_lo(h4[e]), p1 - bf16_hi(h4[e]));
        }
        hi[c] = make_uint4(h4[0], h4[1], h4[2], h4[3]);
        lo[c] = make_uint4(l4[0], l4[1], l4[2], l4[3]);
      }
      l_sum += psum;
      if (j >= 1) {
        // P V of the previous block has finished: P may be overwritten and O rescaled
        w = pf_wait(sm, &sm.p_free, uint32_t(j - 1) & 1, a.status);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, move)) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + 32 * half, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(lane_base + kColO + 32 * half, o);
          }
        }
      }
      put_row_sw128(sm.p_hi, r, hi);
      put_row_sw128(sm.p_lo, r, lo);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.p_full);
    }
    // ---- epilogue: O / l for the rows of real query tokens ----
    bool w = ok && pf_wait(sm, &sm.p_free, uint32_t(nblocks - 1) & 1, a.status);
    if (__all_sync(0xffffffffu, w)) {
      tc_fence_after();
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      float *dst = a.out + ((long long)(q0 + t0 + tok) * kQHeads + g * kGroup + hh) * kHeadDim;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        tmem_ld32(lane_base + kColO + 32 * half, o);
        if (t0 + tok < n) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4 *>(dst + 32 * half + c) =
                make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                            __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

int setup_prefill_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kPfSmemBytes));
  });
  return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_prefill_attention(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                           const int32_t *query_start, const int32_t *block_tables,
                                           int64_t block_table_stride, const int32_t *context_lens, int num_seqs,
                                           int max_query, int max_context, float scale, int32_t *device_status,
                                           void *stream) {
  int rc = pkv::check_pool(pool);
  if (rc != PKV_OK) return rc;
  if (num_q_heads != pkv::kQHeads) return PKV_ERR_UNSUPPORTED;
  if (num_seqs < 0 || max_query < 0 || max_context < 0 || block_table_stride < 0) return PKV_ERR_SHAPE;
  if (num_seqs == 0 || max_query == 0) return PKV_OK;
  if (out == nullptr || q == nullptr || query_start == nullptr || block_tables == nullptr || context_lens == nullptr)
    return PKV_ERR_NULL;
  if (!isfinite(scale)) return PKV_ERR_SCALE;
  if (!pkv::aligned16(q) || !pkv::aligned16(out) || (reinterpret_cast<uintptr_t>(query_start) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_ALIGN;
  const long long tiles = (max_query + pkv::kPfTok - 1) / pkv::kPfTok;
  if ((long long)num_seqs * tiles * pkv::kKvHeads > 0x7fffffffLL) return PKV_ERR_SHAPE;
  rc = pkv::setup_prefill_attributes();
  if (rc != PKV_OK) return rc;
  pkv::PrefillArgs a;
  rc = pkv::pool_tensor_maps(pool, pkv::kPageTokens, &a.tmap_k, &a.tmap_v);
  if (rc != PKV_OK) return rc;
  a.num_pages = pool->num_pages;
  a.q = static_cast<const uint4 *>(q);
  a.out = out;
  a.query_start = query_start;
  a.block_tables = block_tables;
  a.bt_stride = block_table_stride;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.max_context = max_context;
  a.tiles_per_seq = int(tiles);
  a.scale_log2 = scale * pkv::kLog2e;
  a.status = device_status;
  const unsigned grid = unsigned((long long)num_seqs * tiles * pkv::kKvHeads);
  pkv::paged_prefill_kernel<<<grid, pkv::kPfThreads, pkv::kPfSmemBytes, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}
