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
// GB300 design
//  * Grid: one CTA per (32-query tile of a sequence, K/V head g).  Warp w serves
//    query head 4g + (w % 4) for 16 query tokens (w / 4 picks which 16), so the
//    8 warps share every K/V row the CTA loads.  Tiles are numbered latest-first
//    within a sequence so the longest causal spans start first.
//  * Staging: head g's 16 rows of each page arrive as two tiled TMA boxes
//    (2 KiB of K, 2 KiB of V, 128-byte swizzle) into a ring of stages with
//    mbarriers; the last warp done with a stage refills it (no producer warp).
//  * Math on the tensor cores: S[16 tokens x 16 keys] = Q K^T as 2 x 4
//    mma.sync m16n8k16 (bf16 in, fp32 accumulate; K by ldmatrix), online softmax
//    per row on the accumulator fragments (exp2 domain, quad shuffles), and
//    O += P V with P split into bf16 hi + lo parts (two MMAs per 8-dim tile; V by
//    ldmatrix.trans) so the weights keep ~16 significant bits.
//  * Masks: key t counts for query i when t <= p_i; keys at or past the context
//    get -inf and zeroed V fragments, so stale pool bytes never reach the sums.
//    A warp skips pages that lie wholly after its last query's position.
//  * Every mbarrier wait is bounded (about 2 s) and reports PKV_DEV_TIMEOUT.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>

#include "host_common.h"
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kPfStages = 4;
constexpr int kPfWarps = 8;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfTile = 32;                          // query tokens per CTA (2 x 16)
constexpr int kBox = kPageTokens * kRowBytes;        // one head's rows of one page: 2 KiB
constexpr float kLog2e = 1.4426950408889634f;

struct PrefillArgs {
  CUtensorMap tmap_k;  // boxes of one head's 16 rows of one page
  CUtensorMap tmap_v;
  int num_pages;
  const uint32_t *q;  // [total][32][64] bf16 as pairs
  float *out;         // [total][32][64]
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
  uint8_t kv[kPfStages][2][kBox];  // [stage][K|V], 2 KiB each (1024-byte aligned)
  uint64_t full[kPfStages];
  int stage_ok[kPfStages];
  unsigned stage_done[kPfStages];
  unsigned long long issued;
  int any_aborted;
};
constexpr size_t kPfSmemBytes = sizeof(PfSmem) + 1024;

__device__ __forceinline__ void pf_issue(const PrefillArgs &a, PfSmem &sm, int st, int page, int g, uint64_t policy) {
  if (page >= 0 && page < a.num_pages) {
    sm.stage_ok[st] = 1;
    mbar_arrive_expect_tx(&sm.full[st], 2 * kBox);
    tma_load_3d(sm.kv[st][0], &a.tmap_k, 0, g * kPageTokens, page, &sm.full[st], policy);
    tma_load_3d(sm.kv[st][1], &a.tmap_v, 0, g * kPageTokens, page, &sm.full[st], policy);
  } else {
    report(a.status, PKV_DEV_BAD_PAGE);
    sm.stage_ok[st] = 0;
    mbar_arrive(&sm.full[st]);
  }
}

__global__ void __launch_bounds__(kPfThreads, 2) paged_prefill_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  PfSmem &sm = *reinterpret_cast<PfSmem *>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x / a.tiles_per_seq;
  const int tile = a.tiles_per_seq - 1 - int(blockIdx.x % a.tiles_per_seq);
  const int g = blockIdx.y;
  const int q0 = __ldg(a.query_start + s);
  const int n = __ldg(a.query_start + s + 1) - q0;
  const int ctx = __ldg(a.context_lens + s);
  const int t0 = tile * kPfTile;
  if (n <= 0 || t0 >= n) return;
  const int tend = min(t0 + kPfTile, n);
  if (ctx < 0 || ctx > a.max_context || n > ctx) {
    // invalid sequence: zero this CTA's rows (its tokens, query heads 4g .. 4g+3)
    if (tile == 0 && g == 0 && tid == 0) report(a.status, PKV_DEV_BAD_CONTEXT);
    for (int k = tid; k < (tend - t0) * kGroup * kHeadDim; k += kPfThreads) {
      const int tok = t0 + k / (kGroup * kHeadDim), rem = k % (kGroup * kHeadDim);
      a.out[((long long)(q0 + tok) * kQHeads + g * kGroup) * kHeadDim + rem] = 0.f;
    }
    return;
  }
  const int base_pos = ctx - n;                      // position of query token 0
  const int npages = (base_pos + tend - 1) / kPageTokens + 1;
  const int32_t *table = a.block_tables + (long long)s * a.bt_stride;

  if (tid == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&sm.full[i], 1);
      sm.stage_done[i] = 0;
    }
    sm.issued = 0;
    sm.any_aborted = 0;
    mbar_init_fence();
  }
  __syncthreads();
  const uint64_t policy = policy_evict_first();
  if (tid == 0) {
    prefetch_tensormap(&a.tmap_k);
    prefetch_tensormap(&a.tmap_v);
    const int first = npages < kPfStages ? npages : kPfStages;
    for (int j = 0; j < first; ++j) pf_issue(a, sm, j, __ldg(table + j), g, policy);
    atomicMax(&sm.issued, (unsigned long long)first);
  }

  // ---- this warp: query head hq, tokens tw .. tw+15 (rows r = lane/4 and r + 8) ----
  const int hq = g * kGroup + (warp & 3);
  const int tw = t0 + 16 * (warp >> 2);
  const int quad = lane & 3, r = lane >> 2;
  const int tok_a = tw + r, tok_b = tw + r + 8;      // query tokens of fragment rows r and r + 8
  // a query row past n is padding: it attends like the last real row and is not written
  const int pos_a = base_pos + min(tok_a, n - 1), pos_b = base_pos + min(tok_b, n - 1);
  const int warp_last_pos = base_pos + min(tw + 15, n - 1);
  const int warp_first_pos = base_pos + min(tw, n - 1);
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t krow = uint32_t((((mi >> 1) << 3) + ri) * kRowBytes);
  const uint32_t kchunk = uint32_t(mi & 1);
  const uint32_t vrow = uint32_t((((mi & 1) << 3) + ri) * kRowBytes);
  const uint32_t vchunk = uint32_t(mi >> 1);
  uint32_t qa[4][4];  // A fragments per k-step: rows r, r+8; k pairs 2 quad and 8 + 2 quad
  {
    const bool va = tw < n && tok_a < n, vb = tok_b < n;
    const uint32_t *ra = a.q + ((long long)(q0 + min(tok_a, n - 1)) * kQHeads + hq) * (kHeadDim / 2);
    const uint32_t *rb = a.q + ((long long)(q0 + min(tok_b, n - 1)) * kQHeads + hq) * (kHeadDim / 2);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qa[ks][0] = va ? __ldg(ra + ks * 8 + quad) : 0u;
      qa[ks][1] = vb ? __ldg(rb + ks * 8 + quad) : 0u;
      qa[ks][2] = va ? __ldg(ra + ks * 8 + 4 + quad) : 0u;
      qa[ks][3] = vb ? __ldg(rb + ks * 8 + 4 + quad) : 0u;
    }
  }
  float o[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  bool aborted = false;

  for (int pg = 0; pg < npages; ++pg) {
    const int st = pg % kPfStages;
    if (!aborted && !mbar_wait(&sm.full[st], uint32_t(pg / kPfStages) & 1)) {
      report(a.status, PKV_DEV_TIMEOUT);
      aborted = true;
    }
    const int key0 = pg * kPageTokens;
    if (!aborted && sm.stage_ok[st] && key0 <= warp_last_pos) {
      const uint32_t kbase = smem_addr(sm.kv[st][0]);
      const uint32_t vbase = smem_addr(sm.kv[st][1]);
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t b00, b01, b10, b11;
        ldmatrix_x4(kbase + krow + (((2 * ks + kchunk) ^ ri) << 4), b00, b01, b10, b11);
        mma_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
        mma_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
      }
      // scores in log2 units; key t counts for a row at position p when t <= p (p < ctx).
      // Pages wholly at or before every row's position need no mask.
      float xa[4], xb[4];
      if (key0 + kPageTokens - 1 <= warp_first_pos) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            xa[2 * nt + j] = sc[nt][j] * a.scale_log2;
            xb[2 * nt + j] = sc[nt][2 + j] * a.scale_log2;
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int t = key0 + 8 * nt + 2 * quad + j;
            xa[2 * nt + j] = (t <= pos_a) ? sc[nt][j] * a.scale_log2 : -INFINITY;
            xb[2 * nt + j] = (t <= pos_b) ? sc[nt][2 + j] * a.scale_log2 : -INFINITY;
          }
      }
      float mxa = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
      float mxb = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
      // a row whose keys here are all masked keeps its state (its max stays as it was)
      const float na = fmaxf(m_a, mxa), nb = fmaxf(m_b, mxb);
      const float alpha_a = (na == -INFINITY) ? 1.f : exp2f(m_a - na);
      const float alpha_b = (nb == -INFINITY) ? 1.f : exp2f(m_b - nb);
      float pa[4], pb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pa[k] = (na == -INFINITY) ? 0.f : exp2f(xa[k] - na);
        pb[k] = (nb == -INFINITY) ? 0.f : exp2f(xb[k] - nb);
      }
      l_a = l_a * alpha_a + ((pa[0] + pa[1]) + (pa[2] + pa[3]));
      l_b = l_b * alpha_b + ((pb[0] + pb[1]) + (pb[2] + pb[3]));
      m_a = na;
      m_b = nb;
      if (!__all_sync(0xffffffffu, alpha_a == 1.f && alpha_b == 1.f)) {  // no row's maximum moved: skip
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) {
          o[nd][0] *= alpha_a;
          o[nd][1] *= alpha_a;
          o[nd][2] *= alpha_b;
          o[nd][3] *= alpha_b;
        }
      }
      // P as A fragments (rows r, r + 8; keys 2 quad (+1) and 8 + 2 quad (+1)), hi and lo parts
      const uint32_t h0 = pack_bf16x2(pa[0], pa[1]), h1 = pack_bf16x2(pb[0], pb[1]);
      const uint32_t h2 = pack_bf16x2(pa[2], pa[3]), h3 = pack_bf16x2(pb[2], pb[3]);
      const uint32_t l0 = pack_bf16x2(pa[0] - bf16_lo(h0), pa[1] - bf16_hi(h0));
      const uint32_t l1 = pack_bf16x2(pb[0] - bf16_lo(h1), pb[1] - bf16_hi(h1));
      const uint32_t l2 = pack_bf16x2(pa[2] - bf16_lo(h2), pa[3] - bf16_hi(h2));
      const uint32_t l3 = pack_bf16x2(pb[2] - bf16_lo(h3), pb[3] - bf16_hi(h3));
      // V fragments hold keys 2 quad (+1) and 8 + 2 quad (+1): zero those at or past the context
      uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
      if (key0 + kPageTokens > ctx) {
        const int k0 = key0 + 2 * quad;
        vm_lo = (k0 < ctx ? 0x0000ffffu : 0u) | (k0 + 1 < ctx ? 0xffff0000u : 0u);
        vm_hi = (k0 + 8 < ctx ? 0x0000ffffu : 0u) | (k0 + 9 < ctx ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(vbase + vrow + (((nd + vchunk) ^ ri) << 4), v0, v1, v2, v3);
        v0 &= vm_lo;
        v1 &= vm_hi;
        v2 &= vm_lo;
        v3 &= vm_hi;
        mma_16816(o[nd], h0, h1, h2, h3, v0, v1);
        mma_16816(o[nd], l0, l1, l2, l3, v0, v1);
        mma_16816(o[nd + 1], h0, h1, h2, h3, v2, v3);
        mma_16816(o[nd + 1], l0, l1, l2, l3, v2, v3);
      }
    }
    // the last warp done with this stage refills it with the page kPfStages ahead
    __syncwarp();
    if (pg + kPfStages < npages && lane == 0 && !aborted) {
      const unsigned done = atomicAdd(&sm.stage_done[st], 1u) + 1u;
      if (done % kPfWarps == 0) {
        pf_issue(a, sm, st, __ldg(table + pg + kPfStages), g, policy);
        atomicMax(&sm.issued, (unsigned long long)(pg + kPfStages + 1));
      }
    }
    if (aborted && lane == 0) sm.any_aborted = 1;
  }

  // ---- write the rows of real query tokens ----
  float la = l_a + __shfl_xor_sync(0xffffffffu, l_a, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  float lb = l_b + __shfl_xor_sync(0xffffffffu, l_b, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  const float ia = la > 0.f ? 1.f / la : 0.f, ib = lb > 0.f ? 1.f / lb : 0.f;
  if (tok_a < n) {
    float *dst = a.out + ((long long)(q0 + tok_a) * kQHeads + hq) * kHeadDim + 2 * quad;
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) *reinterpret_cast<float2 *>(dst + 8 * nd) = make_float2(o[nd][0] * ia, o[nd][1] * ia);
  }
  if (tok_b < n) {
    float *dst = a.out + ((long long)(q0 + tok_b) * kQHeads + hq) * kHeadDim + 2 * quad;
#pragma unroll
    for (int nd = 0; nd < 8; ++nd) *reinterpret_cast<float2 *>(dst + 8 * nd) = make_float2(o[nd][2] * ib, o[nd][3] * ib);
  }
  __syncthreads();
  if (tid == 0 && sm.any_aborted) {
    const long long issued = (long long)sm.issued;
    const long long first = issued > kPfStages ? issued - kPfStages : 0;
    for (long long j = first; j < issued; ++j)
      mbar_wait(&sm.full[int(j % kPfStages)], uint32_t(j / kPfStages) & 1);
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
  if (!pkv::aligned16(q) || (reinterpret_cast<uintptr_t>(out) & 7u) ||
      (reinterpret_cast<uintptr_t>(query_start) & 3u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_ALIGN;
  const long long tiles = (max_query + pkv::kPfTile - 1) / pkv::kPfTile;
  if ((long long)num_seqs * tiles > 0x7fffffffLL) return PKV_ERR_SHAPE;
  rc = pkv::setup_prefill_attributes();
  if (rc != PKV_OK) return rc;
  pkv::PrefillArgs a;
  rc = pkv::pool_tensor_maps(pool, pkv::kPageTokens, &a.tmap_k, &a.tmap_v);
  if (rc != PKV_OK) return rc;
  a.num_pages = pool->num_pages;
  a.q = static_cast<const uint32_t *>(q);
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
  const dim3 grid(unsigned(num_seqs * tiles), unsigned(pkv::kKvHeads));
  pkv::paged_prefill_kernel<<<grid, pkv::kPfThreads, pkv::kPfSmemBytes, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}
