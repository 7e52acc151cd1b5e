// Paged decode attention: one query token per sequence attends over that
// sequence's cached K/V, read page by page through its block table, with an FP32
// online softmax and grouped-query heads.
//
// What is computed (samir-vllm README, "What works so far": direct paged decode
// attention with FP32 online softmax, each query head streams its sequence's
// cached pages, no contiguous gather, no stored scores; "tiny-vllm part 3",
// "Per-head attention scores and GQA": query head h uses K/V head h / 4, scale
// 1/sqrt(64); same page, "causalMask and online softmax": two partial softmax
// states (m, d) combine as m = max(ma, mb), d = da e^(ma-m) + db e^(mb-m) - here
// extended with the weighted-V accumulator so that partial results over disjoint
// token ranges merge exactly):
//
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t[h/4]) V_t[h/4]
//
// GB300 design
//  * Work split: the pages of all sequences form one list (sequence-major); the
//    grid has G CTAs (a multiple of the SM count) and CTA c takes pages
//    [c*T/G, (c+1)*T/G) of the T pages in the list, so every CTA streams the
//    same number of bytes whatever the mix of context lengths.  A sequence
//    covered by one CTA is written out directly; a sequence cut across CTAs
//    leaves one partial state (m, l, acc) per CTA in the workspace, combined by
//    the merge kernel.  The partial of (CTA c, sequence s) lives in slot c + s,
//    unique because the (c, s) pairs of the list form a monotone staircase.
//  * Staging: one producer thread streams each page as two tiled TMA boxes (the
//    K half and the V half: 8 heads x 16 tokens x 128 B rows) into a ring of
//    shared-memory stages guarded by mbarriers.  The boxes land 128-byte
//    swizzled (16-byte chunk c of row r stored at chunk c ^ (r % 8)), so the
//    ldmatrix reads below are free of bank conflicts.
//  * Math on the tensor cores, one warp per K/V head serving its 4 query heads:
//    S[16 x 16] = Q[16 x 64] K^T (rows 0-3 are the group's query heads, rows
//    4-15 zero) as 2 x 4 mma.sync m16n8k16 (bf16 in, fp32 accumulate), K read
//    with ldmatrix; the online softmax (exp2, scale*log2(e) applied to the fp32
//    scores) runs on the accumulator fragments with quad shuffles; the
//    probabilities stay in registers as the A operand of O[16 x 64] += P V
//    (8 n-tiles, V read with ldmatrix.trans).  P is split into bf16 hi + lo
//    parts (two MMAs each) so the weights keep ~16 significant bits.  Tokens
//    past the context in a sequence's last page get score -inf and their V
//    fragments are zeroed, so stale pool bytes (even NaN) never reach the sums.
//  * Every mbarrier wait is bounded (about 2 s); on expiry the CTA reports
//    PKV_DEV_TIMEOUT and stops, after draining its outstanding copies.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>

#include "host_common.h"
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kStages = 3;
constexpr int kConsumerWarps = kKvHeads;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxCtas = 1024;
constexpr int kCtasPerSm = 2;
constexpr int kMinPagesPerCta = 2;
constexpr int kMergeThreads = 256;
constexpr int kBoxRows = kKvHeads * kPageTokens;  // 128 rows of 128 B per K (or V) half page
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
  CUtensorMap tmap_k;  // K halves: dims (64 elems, 128 rows, pages), 128B swizzle
  CUtensorMap tmap_v;  // V halves, same shape
  int num_pages;
  const uint32_t *q;  // [num_seqs][32][64] bf16, as 32 packed pairs per head
  float *out;         // [num_seqs][32][64]
  const int32_t *block_tables;
  long long bt_stride;
  const int32_t *context_lens;
  int num_seqs;
  int max_context;
  float scale_log2;  // scale * log2(e)
  float *part_acc;   // [kMaxCtas + num_seqs][32][64]
  float2 *part_ml;   // [kMaxCtas + num_seqs][32]  (running max in log2 units, sum)
  int2 *seq_info;    // [num_seqs]  (first CTA, last CTA) touching the sequence
  long long *meta;   // [2]: total pages T and CTA count G of the last split pass
  int32_t *status;
};

struct __align__(1024) Smem {
  uint8_t kv[kStages][2][kHalfPageBytes];  // each half 1024-byte aligned (swizzle atom)
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int stage_ok[kStages];
  long long warp_sums[32];
  long long total_pages;
  long long seq0_first;  // global index of the first page of seq0
  int seq0;
  int found;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + slack to align the dynamic base to 1024 B

__device__ __forceinline__ int seq_pages(int ctx, int max_context) {
  return (ctx > 0 && ctx <= max_context) ? (ctx + kPageTokens - 1) / kPageTokens : 0;
}

// Inclusive block-wide prefix sum (all kThreads threads must call).
__device__ long long block_inclusive_scan(long long v, Smem &sm, long long *block_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.warp_sums[warp] = x;
  __syncthreads();
  long long before = 0, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const long long ws = sm.warp_sums[w];
    if (w < warp) before += ws;
    total += ws;
  }
  __syncthreads();
  *block_total = total;
  return x + before;
}

// CTA that owns global page p when T pages are split over G CTAs.
__device__ __forceinline__ int cta_of_page(long long p, long long T, int G) {
  return int(((p + 1) * G - 1) / T);
}

// Walk over the (sequence, local page) pairs of a CTA's page range.
struct Walk {
  int s, lp, n, ctx;
  __device__ void next(const DecodeArgs &a) {
    if (++lp < n) return;
    lp = 0;
    do {
      ++s;
      ctx = (s < a.num_seqs) ? __ldg(a.context_lens + s) : 1;
      n = seq_pages(ctx, a.max_context);
    } while (n == 0 && s < a.num_seqs);
  }
};

// A-operand fragments of Q for the four k-steps: lane < 16 holds query head
// 4g + lane/4, dims 16ks + 2(lane%4) (+1) and 16ks + 8 + 2(lane%4) (+1); lanes
// 16..31 are the zero rows 4..7.
__device__ __forceinline__ void load_q(const DecodeArgs &a, int s, int g, int lane, uint32_t (&qa)[4][2]) {
  if (lane < 16) {
    const uint32_t *row = a.q + ((long long)s * kQHeads + g * kGroup + (lane >> 2)) * (kHeadDim / 2);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qa[ks][0] = __ldg(row + ks * 8 + (lane & 3));
      qa[ks][1] = __ldg(row + ks * 8 + 4 + (lane & 3));
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) qa[ks][0] = qa[ks][1] = 0u;
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) paged_decode_partial_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kConsumerWarps);
    }
    sm.found = 0;
    mbar_init_fence();
  }

  // ---- total pages T, and this CTA's range [pa, pb) ----
  long long mine = 0;
  for (int i = tid; i < a.num_seqs; i += kThreads) {
    const int c = __ldg(a.context_lens + i);
    mine += seq_pages(c, a.max_context);
    if (cta == 0 && (c < 0 || c > a.max_context)) report(a.status, PKV_DEV_BAD_CONTEXT);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) sm.warp_sums[warp] = mine;
  __syncthreads();
  if (tid == 0) {
    long long t = 0;
    for (int w = 0; w < kThreads / 32; ++w) t += sm.warp_sums[w];
    sm.total_pages = t;
    if (cta == 0) {
      a.meta[0] = t;
      a.meta[1] = G;
    }
  }
  __syncthreads();
  const long long T = sm.total_pages;
  const long long pa = (long long)cta * T / G, pb = (long long)(cta + 1) * T / G;
  if (pa >= pb) return;  // nothing assigned (uniform across the CTA)

  // ---- first sequence of the range ----
  long long running = 0;
  for (int base = 0; base < a.num_seqs; base += kThreads) {
    const int i = base + tid;
    const int v = (i < a.num_seqs) ? seq_pages(__ldg(a.context_lens + i), a.max_context) : 0;
    long long chunk_total;
    const long long incl = block_inclusive_scan(v, sm, &chunk_total) + running;
    if (v > 0 && incl - v <= pa && pa < incl) {
      sm.seq0 = i;
      sm.seq0_first = incl - v;
      sm.found = 1;
    }
    __syncthreads();
    if (sm.found) break;
    running += chunk_total;
  }
  const long long count = pb - pa;

  Walk w;
  w.s = sm.seq0;
  w.ctx = __ldg(a.context_lens + w.s);
  w.n = seq_pages(w.ctx, a.max_context);
  w.lp = int(pa - sm.seq0_first);

  if (warp == kConsumerWarps) {
    // ================= producer: one thread streams pages =================
    if (lane != 0) return;
    prefetch_tensormap(&a.tmap_k);
    prefetch_tensormap(&a.tmap_v);
    const uint64_t policy = policy_evict_first();
    long long issued = 0;
    bool ok = true;
    for (long long i = 0; i < count; ++i) {
      const int st = int(i % kStages);
      const uint32_t round = uint32_t(i / kStages);
      if (i >= kStages && !mbar_wait(&sm.empty[st], (round - 1) & 1)) {
        report(a.status, PKV_DEV_TIMEOUT);
        ok = false;
        break;
      }
      const int page = __ldg(a.block_tables + (long long)w.s * a.bt_stride + w.lp);
      if (page >= 0 && page < a.num_pages) {
        sm.stage_ok[st] = 1;
        mbar_arrive_expect_tx(&sm.full[st], 2 * kHalfPageBytes);
        tma_load_3d(sm.kv[st][0], &a.tmap_k, 0, 0, page, &sm.full[st], policy);
        tma_load_3d(sm.kv[st][1], &a.tmap_v, 0, 0, page, &sm.full[st], policy);
      } else {
        report(a.status, PKV_DEV_BAD_PAGE);
        sm.stage_ok[st] = 0;
        mbar_arrive(&sm.full[st]);
      }
      ++issued;
      if (i + 1 < count) w.next(a);
    }
    if (!ok) {
      // Drain: wait (bounded) for the copies still landing in the stages that
      // were issued but possibly not consumed, so none outlives the CTA.
      const long long first = issued > kStages ? issued - kStages : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait(&sm.full[int(i % kStages)], uint32_t(i / kStages) & 1);
    }
    return;
  }

  // ================= consumers: warp g serves K/V head g =================
  const int g = warp;
  const int quad = lane & 3;     // column pair of the accumulator fragments
  const int hrow = lane >> 2;    // fragment row: query head hrow of the group when < 4
  // ldmatrix row addresses (byte offsets inside a stage half), fixed per lane:
  // lane i addresses row i % 8 of matrix i / 8.
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t krow = uint32_t((g * kPageTokens + ((mi >> 1) << 3) + ri) * kRowBytes);  // K: token (mi/2)*8 + ri
  const uint32_t kchunk = uint32_t(mi & 1);                                                 // + 2 ks
  const uint32_t vrow = uint32_t((g * kPageTokens + ((mi & 1) << 3) + ri) * kRowBytes);   // V: token (mi%2)*8 + ri
  const uint32_t vchunk = uint32_t(mi >> 1);                                                // + nd
  uint32_t qa[4][2];
  load_q(a, w.s, g, lane, qa);
  float m_run = -INFINITY, l_run = 0.f;
  float o[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  bool has_first = (w.lp == 0);
  long long gfirst = pa - w.lp;  // global index of the first page of the current sequence

  for (long long i = 0; i < count; ++i) {
    const int st = int(i % kStages);
    if (!mbar_wait(&sm.full[st], uint32_t(i / kStages) & 1)) {
      report(a.status, PKV_DEV_TIMEOUT);
      return;
    }
    const int valid = min(kPageTokens, w.ctx - w.lp * kPageTokens);
    if (sm.stage_ok[st]) {
      const uint32_t kbase = smem_addr(sm.kv[st][0]);
      const uint32_t vbase = smem_addr(sm.kv[st][1]);
      // ---- S = Q K^T: two n-tiles of 8 tokens, four k-steps of 16 dims ----
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t b00, b01, b10, b11;
        ldmatrix_x4(kbase + krow + (((2 * ks + kchunk) ^ ri) << 4), b00, b01, b10, b11);
        mma_16816(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, b00, b01);
        mma_16816(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, b10, b11);
      }
      // ---- online softmax of row hrow (tokens 8nt + 2 quad + j) ----
      float x[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j)
          x[nt][j] = (8 * nt + 2 * quad + j < valid) ? sc[nt][j] * a.scale_log2 : -INFINITY;
      float mx = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = exp2f(m_run - m_new);
      float p[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) p[nt][j] = exp2f(x[nt][j] - m_new);
      l_run = l_run * alpha + ((p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
      m_run = m_new;
      // P as the A operand of P V, split into bf16 hi + lo parts.
      const uint32_t ph0 = pack_bf16x2(p[0][0], p[0][1]);
      const uint32_t ph1 = pack_bf16x2(p[1][0], p[1][1]);
      const uint32_t pl0 = pack_bf16x2(p[0][0] - bf16_lo(ph0), p[0][1] - bf16_hi(ph0));
      const uint32_t pl1 = pack_bf16x2(p[1][0] - bf16_lo(ph1), p[1][1] - bf16_hi(ph1));
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        o[nd][0] *= alpha;
        o[nd][1] *= alpha;
      }
      // V fragments hold tokens 2 quad (+1) and 8 + 2 quad (+1): zero those past the context.
      uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
      if (valid < kPageTokens) {
        const int t0 = 2 * quad;
        vmask_lo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
        vmask_hi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
      }
      // ---- O += P V: eight n-tiles of 8 dims, one k-step of 16 tokens ----
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(vbase + vrow + (((nd + vchunk) ^ ri) << 4), v0, v1, v2, v3);
        v0 &= vmask_lo;
        v1 &= vmask_hi;
        v2 &= vmask_lo;
        v3 &= vmask_hi;
        mma_16816(o[nd], ph0, 0u, ph1, 0u, v0, v1);
        mma_16816(o[nd], pl0, 0u, pl1, 0u, v0, v1);
        mma_16816(o[nd + 1], ph0, 0u, ph1, 0u, v2, v3);
        mma_16816(o[nd + 1], pl0, 0u, pl1, 0u, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[st]);

    const bool seq_end = (w.lp == w.n - 1);
    if (seq_end || i == count - 1) {
      // ---- finish this sequence's share: direct output or a partial state ----
      float lt = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      if (has_first && seq_end) {
        if (hrow < kGroup) {
          float *dst = a.out + ((long long)w.s * kQHeads + g * kGroup + hrow) * kHeadDim + 2 * quad;
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
          for (int nd = 0; nd < 8; ++nd)
            *reinterpret_cast<float2 *>(dst + 8 * nd) = make_float2(o[nd][0] * inv, o[nd][1] * inv);
        }
      } else {
        const long long slot = (long long)cta + w.s;
        if (hrow < kGroup) {
          float *dst = a.part_acc + (slot * kQHeads + g * kGroup + hrow) * kHeadDim + 2 * quad;
#pragma unroll
          for (int nd = 0; nd < 8; ++nd) *reinterpret_cast<float2 *>(dst + 8 * nd) = make_float2(o[nd][0], o[nd][1]);
          if (quad == 0) a.part_ml[slot * kQHeads + g * kGroup + hrow] = make_float2(m_run, lt);
        }
      }
      if (has_first && g == 0 && lane == 0) {
        const long long T_ = sm.total_pages;
        a.seq_info[w.s] = make_int2(cta, cta_of_page(gfirst + w.n - 1, T_, G));
      }
      if (i + 1 < count) {
        w.next(a);
        load_q(a, w.s, g, lane, qa);
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
        has_first = true;
        gfirst = pa + i + 1;
      }
    } else {
      w.next(a);
    }
  }
}

// Combines the partial states of sequences split across CTAs:
//   M = max_c m_c,  L = sum_c l_c 2^(m_c - M),  out = sum_c acc_c 2^(m_c - M) / L.
// Also writes the zero rows of empty or invalid sequences.
__global__ void __launch_bounds__(kMergeThreads) paged_decode_merge_kernel(const DecodeArgs a) {
  const int s = blockIdx.x;
  const int tid = threadIdx.x;
  const int h = tid >> 3, d0 = (tid & 7) * 8;
  float *o = a.out + ((long long)s * kQHeads + h) * kHeadDim + d0;
  const int ctx = __ldg(a.context_lens + s);
  if (ctx <= 0 || ctx > a.max_context) {
    reinterpret_cast<float4 *>(o)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4 *>(o)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int2 info = a.seq_info[s];
  if (info.x == info.y) return;  // written directly by its only CTA
  // CTAs between the first and the last may own no pages at all (more CTAs than
  // pages); they left no partial and are skipped.
  const long long T = a.meta[0];
  const long long G = a.meta[1];
  float M = -INFINITY;
  for (int c = info.x; c <= info.y; ++c) {
    if ((long long)c * T / G == (long long)(c + 1) * T / G) continue;
    M = fmaxf(M, a.part_ml[((long long)c + s) * kQHeads + h].x);
  }
  float r[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
  if (M != -INFINITY) {
    for (int c = info.x; c <= info.y; ++c) {
      if ((long long)c * T / G == (long long)(c + 1) * T / G) continue;
      const long long slot = (long long)c + s;
      const float2 ml = a.part_ml[slot * kQHeads + h];
      const float wgt = exp2f(ml.x - M);
      L += ml.y * wgt;
      const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + (slot * kQHeads + h) * kHeadDim + d0);
      const float4 x0 = src[0], x1 = src[1];
      r[0] += wgt * x0.x; r[1] += wgt * x0.y; r[2] += wgt * x0.z; r[3] += wgt * x0.w;
      r[4] += wgt * x1.x; r[5] += wgt * x1.y; r[6] += wgt * x1.z; r[7] += wgt * x1.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  reinterpret_cast<float4 *>(o)[0] = make_float4(r[0] * inv, r[1] * inv, r[2] * inv, r[3] * inv);
  reinterpret_cast<float4 *>(o)[1] = make_float4(r[4] * inv, r[5] * inv, r[6] * inv, r[7] * inv);
}


struct WorkspaceLayout {
  long long *meta;
  float *part_acc;
  float2 *part_ml;
  int2 *seq_info;
  size_t bytes;
};

// [meta: 16 B][partial accumulators][partial (m, l)][per-sequence CTA span]
WorkspaceLayout layout_workspace(void *base, int num_seqs) {
  const size_t slots = size_t(kMaxCtas) + size_t(num_seqs);
  WorkspaceLayout L;
  uint8_t *p = static_cast<uint8_t *>(base);
  const size_t meta_bytes = 16;
  const size_t acc_bytes = slots * kQHeads * kHeadDim * sizeof(float);
  const size_t ml_bytes = slots * kQHeads * sizeof(float2);
  L.meta = reinterpret_cast<long long *>(p);
  L.part_acc = reinterpret_cast<float *>(p + meta_bytes);
  L.part_ml = reinterpret_cast<float2 *>(p + meta_bytes + acc_bytes);
  L.seq_info = reinterpret_cast<int2 *>(p + meta_bytes + acc_bytes + ml_bytes);
  L.bytes = meta_bytes + acc_bytes + ml_bytes + size_t(num_seqs) * sizeof(int2);
  return L;
}

int auto_ctas(int num_seqs, int max_context) {
  const int sms = device_sm_count();
  const long long upper = (long long)num_seqs * ((max_context + kPageTokens - 1) / kPageTokens);
  long long g = sms > 0 ? (long long)sms * kCtasPerSm : 2 * 148;
  const long long by_work = (upper + kMinPagesPerCta - 1) / kMinPagesPerCta;
  if (by_work < g) g = by_work;
  if (g < 1) g = 1;
  if (g > kMaxCtas) g = kMaxCtas;
  return int(g);
}

int setup_kernel_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(paged_decode_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(kSmemBytes));
  });
  return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

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
// kv_head * 16 + token, row stride 128 B, page stride page_stride_bytes; one box
// is a whole half page (64 x 128 x 1), delivered 128-byte swizzled.
int encode_half_pages(CUtensorMap *map, const void *base, long long page_stride, int num_pages) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return PKV_ERR_CUDA;
  const cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(kBoxRows), cuuint64_t(num_pages)};
  const cuuint64_t strides[2] = {cuuint64_t(kRowBytes), cuuint64_t(page_stride)};
  const cuuint32_t box[3] = {cuuint32_t(kHeadDim), cuuint32_t(kBoxRows), 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

int decode(const pkv_pool *pool, float *out, const void *q, int num_q_heads, const int32_t *block_tables,
           int64_t bt_stride, const int32_t *context_lens, int num_seqs, int max_context, float scale,
           void *workspace, size_t workspace_bytes, int32_t *device_status, int num_ctas, void *stream) {
  int rc = check_pool(pool);
  if (rc != PKV_OK) return rc;
  if (num_q_heads != kQHeads) return PKV_ERR_UNSUPPORTED;
  if (num_seqs < 0 || max_context < 0 || bt_stride < 0 || num_ctas < 0 || num_ctas > kMaxCtas)
    return PKV_ERR_SHAPE;
  if (num_seqs > (1 << 24)) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (out == nullptr || q == nullptr || block_tables == nullptr || context_lens == nullptr || workspace == nullptr)
    return PKV_ERR_NULL;
  if (!isfinite(scale)) return PKV_ERR_SCALE;
  if (!aligned16(q) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(out) & 7u) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_ALIGN;
  const WorkspaceLayout L = layout_workspace(workspace, num_seqs);
  if (workspace_bytes < L.bytes) return PKV_ERR_WORKSPACE;
  rc = setup_kernel_attributes();
  if (rc != PKV_OK) return rc;

  DecodeArgs a;
  rc = encode_half_pages(&a.tmap_k, pool->k_base, pool->page_stride_bytes, pool->num_pages);
  if (rc != PKV_OK) return rc;
  rc = encode_half_pages(&a.tmap_v, pool->v_base, pool->page_stride_bytes, pool->num_pages);
  if (rc != PKV_OK) return rc;
  a.num_pages = pool->num_pages;
  a.q = static_cast<const uint32_t *>(q);
  a.out = out;
  a.block_tables = block_tables;
  a.bt_stride = bt_stride;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.max_context = max_context;
  a.scale_log2 = scale * kLog2e;
  a.part_acc = L.part_acc;
  a.part_ml = L.part_ml;
  a.seq_info = L.seq_info;
  a.meta = L.meta;
  a.status = device_status;

  const int G = num_ctas > 0 ? num_ctas : auto_ctas(num_seqs, max_context);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  paged_decode_partial_kernel<<<G, kThreads, kSmemBytes, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_LAUNCH;
  // A single CTA covers every sequence whole and writes the output itself, but
  // sequences with no pages still need their zero rows from the merge kernel.
  paged_decode_merge_kernel<<<num_seqs, kMergeThreads, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_LAUNCH;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim) {
  if (num_seqs < 0 || num_q_heads != pkv::kQHeads || head_dim != pkv::kHeadDim) return 0;
  return pkv::layout_workspace(nullptr, num_seqs).bytes;
}

extern "C" int pkv_decode_max_ctas(void) { return pkv::kMaxCtas; }

extern "C" int pkv_decode_plan(int num_seqs, int max_context, int *num_ctas, int *launches) {
  if (num_seqs < 0 || max_context < 0) return PKV_ERR_SHAPE;
  const int g = num_seqs == 0 ? 0 : pkv::auto_ctas(num_seqs, max_context);
  if (num_ctas) *num_ctas = g;
  if (launches) *launches = num_seqs == 0 ? 0 : 2;
  return PKV_OK;
}

extern "C" int pkv_paged_decode_attention(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                          const int32_t *block_tables, int64_t block_table_stride,
                                          const int32_t *context_lens, int num_seqs, int max_context, float scale,
                                          void *workspace, size_t workspace_bytes, int32_t *device_status,
                                          void *stream) {
  return pkv::decode(pool, out, q, num_q_heads, block_tables, block_table_stride, context_lens, num_seqs,
                     max_context, scale, workspace, workspace_bytes, device_status, 0, stream);
}

extern "C" int pkv_paged_decode_attention_ctas(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                               const int32_t *block_tables, int64_t block_table_stride,
                                               const int32_t *context_lens, int num_seqs, int max_context,
                                               float scale, void *workspace, size_t workspace_bytes,
                                               int32_t *device_status, int num_ctas, void *stream) {
  return pkv::decode(pool, out, q, num_q_heads, block_tables, block_table_stride, context_lens, num_seqs,
                     max_context, scale, workspace, workspace_bytes, device_status, num_ctas, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  The workspace of pkv_paged_decode_attention lives in
// a fixed device array of this file, sized for PKV_NOALLOC_MAX_SEQS sequences,
// for callers that cannot allocate device memory.  Its device address is looked
// up once per device (cudaGetSymbolAddress on the first call with that device
// current); the call then follows the regular path with that address as the
// workspace.  No value in the array needs to start at zero: every partial state,
// span and total the merge reads is written earlier in the same call.
namespace pkv {
namespace {

constexpr size_t kNoallocScratchBytes =
    16 + (size_t(kMaxCtas) + PKV_NOALLOC_MAX_SEQS) * (size_t(kQHeads) * kHeadDim * sizeof(float) +
                                                      size_t(kQHeads) * sizeof(float2)) +
    size_t(PKV_NOALLOC_MAX_SEQS) * sizeof(int2);

}  // namespace
}  // namespace pkv

static __device__ __align__(256) unsigned char pkv_noalloc_scratch[pkv::kNoallocScratchBytes];

namespace pkv {
namespace {

// Device address of pkv_noalloc_scratch on the current device, or nullptr.
void *noalloc_scratch_address() {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, pkv_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_decode_attention_noalloc(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                                  const int32_t *block_tables, int64_t block_table_stride,
                                                  const int32_t *context_lens, int num_seqs, int max_context,
                                                  float scale, int32_t *device_status, void *stream) {
  if (num_seqs > PKV_NOALLOC_MAX_SEQS) return PKV_ERR_NOALLOC_LIMIT;
  if (num_seqs <= 0) {
    return num_seqs < 0 ? PKV_ERR_SHAPE : PKV_OK;
  }
  const size_t need = pkv::layout_workspace(nullptr, num_seqs).bytes;
  if (need > pkv::kNoallocScratchBytes) return PKV_ERR_NOALLOC_LIMIT;
  void *scratch = pkv::noalloc_scratch_address();
  if (scratch == nullptr) return PKV_ERR_CUDA;
  return pkv::decode(pool, out, q, num_q_heads, block_tables, block_table_stride, context_lens, num_seqs,
                     max_context, scale, scratch, pkv::kNoallocScratchBytes, device_status, 0, stream);
}
