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
//    grid has G CTAs (two per SM, or one per SM for small batches) and, from the
//    lengths it reads on the device,
//    the kernel picks how many of them (Gu) share the T pages: CTA c takes pages
//    [c*T/Gu, (c+1)*T/Gu), so every CTA streams the same number of bytes
//    whatever the mix of context lengths.  Equal-length batches are split along
//    sequence boundaries instead (a cut costs a merge), and no CTA gets fewer
//    than 4 pages unless the caller fixes the count.  A sequence
//    covered by one CTA is written out directly; a sequence cut across CTAs
//    leaves one partial state (m, l, acc) per CTA in the workspace, and for each
//    group of 4 query heads the last warp to finish (an atomic ticket on a
//    counter, no waiting, no CTA-wide barrier) merges them with the rule above:
//    one launch per call.  The partial of (CTA c, sequence s) lives in slot
//    c + s, unique because the (c, s) pairs of the list form a monotone
//    staircase; the ticket counters of s live in slot (first CTA of s) + s and
//    are reset by the merging warps, so a zeroed workspace stays valid across
//    calls of any batch size.  Sequences with no
//    pages (context 0 or invalid) get zero rows from CTA s % G.  Small grids
//    start their block-table and query lines toward L2 at entry, as the lengths
//    are read.
//  * Small grids (no more CTAs than can be resident in clusters of 8 at one CTA
//    per SM) are launched in thread-block clusters of 8 consecutive CTAs, and
//    the first merge level stays on chip: the CTAs of a cluster that hold parts
//    of a cut sequence push each head group's partial state into the shared
//    memory of the cluster CTA that merges that head group (distributed shared
//    memory stores), one cluster barrier makes them visible, and the merge reads
//    local shared memory.  Only a sequence cut across clusters still meets in the
//    workspace, one state per cluster, behind the same atomic tickets.
//  * Staging: each page arrives as two tiled TMA boxes (its K half and its V
//    half: 8 heads x 16 tokens x 128 B rows, 16 KiB each, contiguous in the
//    pool) into a ring of shared-memory stages, each with an mbarrier: three
//    stages when two CTAs share an SM, six when the grid has at most one CTA per
//    SM (the same bytes in flight per SM, and a CTA of a small batch has all of
//    its pages requested at once).  There is no producer warp: the CTA has one
//    warp per K/V head, and the last warp to finish with a stage (a per-stage
//    counter in shared memory; nobody waits) refills it with the page a ring
//    length ahead.  The boxes land 128-byte
//    swizzled (16-byte chunk c of row r stored at chunk c ^ (r % 8)), so the
//    ldmatrix reads below are free of bank conflicts.
//  * Math on the tensor cores, one warp per K/V head serving its 4 query heads:
//    S[16 x 16] = Q[16 x 64] K^T (rows 0-3 are the group's query heads, rows
//    4-15 zero) as 2 x 4 mma.sync m16n8k16 (bf16 in, fp32 accumulate), K read
//    with ldmatrix; the online softmax (exp2, scale*log2(e) applied to the fp32
//    scores) runs on the accumulator fragments with quad shuffles; the
//    probabilities stay in registers as the A operand of O[16 x 64] += P V
//    (8 n-tiles, V read with ldmatrix.trans).  P is split into bf16 hi + lo
//    parts so the weights keep ~16 significant bits: the hi part fills A rows
//    0-7 and the lo part rows 8-15, so one MMA per n-tile yields both products
//    (accumulator halves c0/c1 and c2/c3, summed when the sequence ends).  Tokens
//    past the context in a sequence's last page get score -inf and their V
//    fragments are zeroed, so stale pool bytes (even NaN) never reach the sums.
//  * Every mbarrier wait is bounded (about 2 s); on expiry the warp reports
//    PKV_DEV_TIMEOUT, stops waiting, computing and refilling, and walks on to the
//    end so that all warps still meet at the same named barriers; then warp 0
//    waits, again bounded, for any copy still in flight.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>

#include "host_common.h"
#include "pkv_device.cuh"

namespace pkv {
namespace {

constexpr int kStagesShared = 3;  // ring stages when two CTAs share an SM
constexpr int kStagesAlone = 6;   // ring stages when the grid has at most one CTA per SM
constexpr int kClusterCtas = 8;   // CTAs per cluster when the small-grid kernel merges on chip
constexpr int kWarps = kKvHeads;          // one warp per K/V head
constexpr int kThreads = kWarps * 32;
constexpr int kMaxCtas = 1024;
constexpr int kCtasPerSm = 2;
constexpr int kMinPagesPerCta = 4;  // least pages a CTA is given (unless the caller fixes the split)
constexpr int kMergeOneLevel = 12;  // a sequence cut into at most this many parts is merged in one pass
constexpr int kMergeGroup = 8;      // a longer one merges groups of this many consecutive parts first
constexpr int kMergeBatch = 4;      // partial states read at once by a merging warp
constexpr int kHeadRowsBytes = kPageTokens * kRowBytes;  // one head's K (or V) rows of a page: 2 KiB
constexpr float kLog2e = 1.4426950408889634f;

// One workspace slot: the partial state of one (CTA, sequence) pair, plus the
// ticket counter used when this slot is a sequence's first.
struct Slot {
  float acc[kQHeads][kHeadDim];  // un-normalised sum of p * V
  float2 ml[kQHeads];            // (running max in log2 units, sum of p)
  int counter[kWarps];           // per head group: parts of the sequence (or of a merge group) done; 0 between calls
  int counter2[kWarps];          // per head group: merge groups of the sequence done (long sequences); 0 between calls
};

// Cluster merges: one head group's partial state of one part of a sequence, as the CTA that
// holds the part pushes it into the shared memory of the CTA that merges that head group.
struct GroupState {
  float acc[kGroup][kHeadDim];  // un-normalised sum of p * V of query heads 4g .. 4g+3
  float2 ml[kGroup];            // (running max in log2 units, sum of p)
};
// A sequence held by p <= kClusterCtas CTAs of a cluster has its head group g merged by the
// (g mod p)-th of those CTAs, which so receives p parts of at most ceil(kWarps / p) head
// groups: at most 14 states (p = 7).
constexpr int kRecvSlots = 14;
struct RecvArea {
  GroupState slot[kRecvSlots];  // slot k * ceil(kWarps / p) + g / p: part k, head group g
};

struct DecodeArgs {
  CUtensorMap tmap_k;  // K halves: dims (64 elems, 128 rows = head*16 + token, pages), 128B swizzle
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
  Slot *slots;       // [kMaxCtas + num_seqs] partial states and ticket counters
  int32_t *status;
  int split_ctas;    // > 0: split over exactly min(split_ctas, T) CTAs (the caller chose the count)
  // Fused append (pkv_decode_step), else null: sequence s's new token (position ctx-1)
  // goes to slot_mapping[s]; its rows replace the stale ones of the last page in shared
  // memory and are written to the pool by the CTA that holds that page.
  const uint4 *k_new;  // [num_seqs][8][64] bf16, 8 uint4 per head row
  const uint4 *v_new;
  const int32_t *slot_mapping;
  uint8_t *k_pool;     // pool bases for the write
  uint8_t *v_pool;
  long long page_stride;
  long long num_slots;  // num_pages * 16
};

template <int kStages>
struct __align__(1024) SmemT {
  uint8_t kv[kStages][2][kHalfPageBytes];  // [stage][K|V] boxes of [head][token][128 B], 1024-byte aligned
  uint64_t full[kStages];
  int stage_ok[kStages];
  unsigned stage_done[kStages];  // warps done with the stage, counted over all rounds
  unsigned long long issued;     // pages issued so far (for the drain after a timeout)
  int any_aborted;
  long long warp_sums[32];
  int warp_n[32], warp_pmin[32], warp_pmax[32];
  long long total_pages;
  int used_ctas;         // CTAs the pages are split over (<= gridDim.x)
  long long seq0_first;  // global index of the first page of seq0
  int seq0;
  int found;
};
// Dynamic shared memory of a kernel instance: the ring and bookkeeping, then (cluster merges)
// two receive areas, plus slack to align the base to 1024 B.
template <int kStages, bool kCluster>
constexpr size_t smem_bytes() { return sizeof(SmemT<kStages>) + (kCluster ? 2 * sizeof(RecvArea) : 0) + 1024; }

__device__ __forceinline__ int seq_pages(int ctx, int max_context) {
  return (ctx > 0 && ctx <= max_context) ? (ctx + kPageTokens - 1) / kPageTokens : 0;
}

// Inclusive block-wide prefix sum (all kThreads threads must call).
template <class Smem>
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

// How many of the G launched CTAs share the T pages of n sequences (pmin .. pmax
// pages each).  Every choice is at most min(G, T), so no CTA is left without a page.
//  * no pages at all: 0 (every CTA only zeroes the rows of empty sequences).
//  * split > 0: the caller fixed the count.
//  * equal-length batches: split along sequence boundaries, so that no CTA holds
//    the end of one sequence and the start of the next: k CTAs per sequence
//    when n <= G (k >= 1, at least kMinPagesPerCta pages each), else the largest
//    divisor of n not above G (whole sequences per CTA) when that keeps at least
//    half of the CTAs busy.
//  * otherwise an even split with at least kMinPagesPerCta pages per CTA.
__device__ int effective_ctas(int G, long long T, int n, int pmin, int pmax, int split) {
  if (T <= 0) return 0;
  if (split > 0) return int(T < split ? T : split);
  const long long cap = T < G ? T : G;
  if (n > 0 && pmin == pmax) {
    if (n <= G) {
      int k = G / n;
      const int by_pages = pmin / kMinPagesPerCta;
      if (k > by_pages) k = by_pages;
      if (k < 1) k = 1;
      return n * k;
    }
    const int k0 = (n + G - 1) / G;
    if (k0 <= 64) {
      for (int k = k0; k <= 2 * k0; ++k)
        if (n % k == 0 && n / k >= G / 2) return n / k;
    }
  }
  long long g = (T + kMinPagesPerCta - 1) / kMinPagesPerCta;
  if (g > cap) g = cap;
  return int(g < 1 ? 1 : g);
}

// Start the copy of the page the walk points at into stage st (or mark the stage
// empty when the page id is invalid).  One thread calls this.
template <class Smem>
__device__ __forceinline__ void issue_page(const DecodeArgs &a, Smem &sm, int st, const Walk &w, uint64_t policy) {
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
}

// Warp g's share of finishing sequence s, cut across CTAs c_first .. c_last (its pages
// are the global pages gfirst .. gfirst + n - 1), once this CTA's partial state is
// stored: a ticket on a (merge group, head group) counter - an acquire-release atomic
// that publishes the lanes' partial stores (ordered before it by __syncwarp) and, for
// the last ticket, makes the other parts visible.  ticket_of() takes the ticket;
// merge_if_last() lets the warp holding the last ticket merge the partial states of
// query heads 4g .. 4g+3 with
//   M = max_c m_c,  L = sum_c l_c 2^(m_c - M),  out = sum_c acc_c 2^(m_c - M) / L
// (one pass, rescaling as the running maximum grows) and reset the counter.  A sequence
// in at most kMergeOneLevel parts is merged at once.  A longer one is merged in two levels,
// so that its first merges overlap its other parts' streaming: the parts of each group of
// kMergeGroup consecutive CTAs are merged into the group's first slot, and the warp that
// finishes the last group merges the group results.  The two halves of a ticket may be
// apart: a warp can take the ticket, stream more pages, and only then look at it.

// First-level merge group [lo, hi] of part c of a sequence cut across c_first .. c_last.
__device__ __forceinline__ void merge_group(int c, int c_first, int c_last, int &lo, int &hi) {
  if (c_last - c_first < kMergeOneLevel) {
    lo = c_first;
    hi = c_last;
    return;
  }
  lo = c_first + (c - c_first) / kMergeGroup * kMergeGroup;
  hi = min(lo + kMergeGroup - 1, c_last);
}

__device__ __forceinline__ int ticket_of(const DecodeArgs &a, int s, long long gfirst, int n, int g, int lane,
                                         long long T, int Gu, int cta) {
  __syncwarp();
  int ticket = 0;
  if (lane == 0) {
    int lo, hi;
    merge_group(cta, cta_of_page(gfirst, T, Gu), cta_of_page(gfirst + n - 1, T, Gu), lo, hi);
    ticket = atomic_add_acq_rel_gpu(&a.slots[(long long)lo + s].counter[g], 1);
  }
  return ticket;  // meaningful in lane 0
}

// Merge of `count` partial states for this lane's query head h and dims d0 .. d0 + 7:
// the running maximum M, sum L and accumulator r.  read(k, ml, x0, x1) loads part k's
// (m, l) and accumulator dims d0 .. d0 + 7.  The parts are read kBatch at a time, every
// load of a batch issued before the first is used, so a batch costs one round trip; the
// batch's maximum rescales the running state once.  (Eight at a time where the warp has
// the registers to spare: the clusters' states after the page loop.)
template <int kBatch = kMergeBatch, class Read>
__device__ __forceinline__ void merge_states(int count, Read read, float &M, float &L, float (&r)[8]) {
  M = -INFINITY;
  L = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = 0.f;
  for (int k0 = 0; k0 < count; k0 += kBatch) {
    float2 ml[kBatch];
    float4 x0[kBatch], x1[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (k0 + j < count) {
        read(k0 + j, ml[j], x0[j], x1[j]);
      } else {
        ml[j] = make_float2(-INFINITY, 0.f);
        x0[j] = x1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // a part whose pages were all invalid (or a padding entry) has m = -inf and weight 0
    float m_new = M;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) m_new = fmaxf(m_new, ml[j].x);
    const float keep = (m_new == -INFINITY) ? 1.f : exp2f(M - m_new);
    L *= keep;
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] *= keep;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float wgt = (ml[j].x == -INFINITY) ? 0.f : exp2f(ml[j].x - m_new);
      L += ml[j].y * wgt;
      r[0] += wgt * x0[j].x; r[1] += wgt * x0[j].y; r[2] += wgt * x0[j].z; r[3] += wgt * x0[j].w;
      r[4] += wgt * x1[j].x; r[5] += wgt * x1[j].y; r[6] += wgt * x1[j].z; r[7] += wgt * x1[j].w;
    }
    M = m_new;
  }
}

// merge_states over the workspace slots first + k * stride + s, k < count (L2 reads).
__device__ __forceinline__ void merge_parts(const DecodeArgs &a, int s, int first, int count, int stride, int h,
                                            int d0, float &M, float &L, float (&r)[8]) {
  merge_states(
      count,
      [&](int k, float2 &ml, float4 &x0, float4 &x1) {
        const Slot &part = a.slots[(long long)first + (long long)k * stride + s];
        ml = __ldcg(&part.ml[h]);
        x0 = __ldcg(reinterpret_cast<const float4 *>(&part.acc[h][d0]));
        x1 = __ldcg(reinterpret_cast<const float4 *>(&part.acc[h][d0 + 4]));
      },
      M, L, r);
}

// Writes the merged rows of query head h, dims d0 .. d0 + 7 of sequence s.
__device__ __forceinline__ void write_merged(const DecodeArgs &a, int s, int h, int d0, float L, const float (&r)[8]) {
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float4 *out = reinterpret_cast<float4 *>(a.out + ((long long)s * kQHeads + h) * kHeadDim + d0);
  out[0] = make_float4(r[0] * inv, r[1] * inv, r[2] * inv, r[3] * inv);
  out[1] = make_float4(r[4] * inv, r[5] * inv, r[6] * inv, r[7] * inv);
}

__device__ __forceinline__ void merge_if_last(const DecodeArgs &a, int s, long long gfirst, int n, int g, int lane,
                                              long long T, int Gu, int ticket, int cta) {
  const int c_first = cta_of_page(gfirst, T, Gu);
  const int c_last = cta_of_page(gfirst + n - 1, T, Gu);
  int lo, hi;
  merge_group(cta, c_first, c_last, lo, hi);
  int last = 0;
  if (lane == 0) {
    last = (ticket == hi - lo);  // every CTA in the group owns pages of the sequence
    if (last) atomicExch(&a.slots[(long long)lo + s].counter[g], 0);  // ready for the next call
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __syncwarp();  // lane 0's acquire comes before every lane's reads of the partial states
  // lane -> query head 4g + lane/8, dims 8 (lane%8) .. +7
  const int h = g * kGroup + (lane >> 3), d0 = (lane & 7) * 8;
  float M, L, r[8];
  merge_parts(a, s, lo, hi - lo + 1, 1, h, d0, M, L, r);
  if (c_last - c_first >= kMergeOneLevel) {
    // first level done: the group's merged state replaces its first part, then the
    // second-level ticket (lane 0's release covers every lane's stores after __syncwarp)
    Slot &dst = a.slots[(long long)lo + s];
    __stcg(reinterpret_cast<float4 *>(&dst.acc[h][d0]), make_float4(r[0], r[1], r[2], r[3]));
    __stcg(reinterpret_cast<float4 *>(&dst.acc[h][d0 + 4]), make_float4(r[4], r[5], r[6], r[7]));
    if ((lane & 7) == 0) __stcg(&dst.ml[h], make_float2(M, L));
    __syncwarp();
    const int groups = (c_last - c_first) / kMergeGroup + 1;
    int last2 = 0;
    if (lane == 0) {
      last2 = atomic_add_acq_rel_gpu(&a.slots[(long long)c_first + s].counter2[g], 1) == groups - 1;
      if (last2) atomicExch(&a.slots[(long long)c_first + s].counter2[g], 0);
    }
    last2 = __shfl_sync(0xffffffffu, last2, 0);
    if (!last2) return;
    __syncwarp();
    merge_parts(a, s, c_first, groups, kMergeGroup, h, d0, M, L, r);
  }
  write_merged(a, s, h, d0, L, r);
}

// Cluster merges (launches with clusters of kClusterCtas consecutive CTAs; CTA c has cluster
// rank c % kClusterCtas).  Sequence s (pages gfirst .. gfirst + n - 1, cut across CTAs
// c_first .. c_last) has parts in CTAs lo .. hi of a cluster, p = hi - lo + 1 of them.  Head
// group g of these parts is merged by warp g of CTA lo + g % p: the CTA holding part k
// pushes it into that CTA's receive area (area 1 when s reaches the end of the receiving
// CTA's range, else area 0: a CTA receives for at most its first and its last segment),
// slot k * ceil(kWarps / p) + g / p.
struct ClusterPlan {
  int c_first, c_last, cl0, lo, p;
  int recv;  // CTA that merges this warp's head group
  int slot;  // its receive slot for part 0 (part k: + k * qmax)
  int qmax;
  int area;  // receive area of s in CTA recv
};

__device__ __forceinline__ ClusterPlan cluster_plan(long long gfirst, int n, int g, long long T, int Gu, int cta) {
  ClusterPlan c;
  c.c_first = cta_of_page(gfirst, T, Gu);
  c.c_last = cta_of_page(gfirst + n - 1, T, Gu);
  c.cl0 = cta - cta % kClusterCtas;
  c.lo = max(c.c_first, c.cl0);
  c.p = min(c.c_last, c.cl0 + kClusterCtas - 1) - c.lo + 1;
  c.recv = c.lo + g % c.p;
  c.qmax = (kWarps + c.p - 1) / c.p;
  c.slot = g / c.p;
  c.area = gfirst + n - 1 >= (long long)(c.recv + 1) * T / Gu - 1 ? 1 : 0;
  return c;
}

// After the cluster barrier that follows every push: if this CTA merges head group g of s,
// warp g merges the p parts from its receive area.  When s lies in this cluster alone the
// rows are written out; otherwise the cluster's state goes to workspace slot lo + s, and the
// warp that takes the last ticket on a counter of slot c_first + s merges the clusters'
// states from the workspace, as the two-level merge does.
__device__ __forceinline__ void cluster_merge(const DecodeArgs &a, const RecvArea *recv, int s, long long gfirst,
                                              int n, int g, int lane, long long T, int Gu, int cta) {
  const ClusterPlan c = cluster_plan(gfirst, n, g, T, Gu, cta);
  if (cta != c.recv) return;  // another CTA of this cluster merges this head group
  const int hl = lane >> 3, h = g * kGroup + hl, d0 = (lane & 7) * 8;
  float M, L, r[8];
  merge_states(
      c.p,
      [&](int k, float2 &ml, float4 &x0, float4 &x1) {
        const GroupState &gs = recv[c.area].slot[k * c.qmax + c.slot];
        ml = gs.ml[hl];
        x0 = *reinterpret_cast<const float4 *>(&gs.acc[hl][d0]);
        x1 = *reinterpret_cast<const float4 *>(&gs.acc[hl][d0 + 4]);
      },
      M, L, r);
  if (c.c_first >= c.cl0 && c.c_last < c.cl0 + kClusterCtas) {
    write_merged(a, s, h, d0, L, r);
    return;
  }
  // this cluster's state, then the ticket (lane 0's release covers every lane's stores after __syncwarp)
  Slot &dst = a.slots[(long long)c.lo + s];
  __stcg(reinterpret_cast<float4 *>(&dst.acc[h][d0]), make_float4(r[0], r[1], r[2], r[3]));
  __stcg(reinterpret_cast<float4 *>(&dst.acc[h][d0 + 4]), make_float4(r[4], r[5], r[6], r[7]));
  if ((lane & 7) == 0) __stcg(&dst.ml[h], make_float2(M, L));
  __syncwarp();
  const int k0 = c.c_first / kClusterCtas, k1 = c.c_last / kClusterCtas;
  int last = 0;
  if (lane == 0) {
    last = atomic_add_acq_rel_gpu(&a.slots[(long long)c.c_first + s].counter[g], 1) == k1 - k0;
    if (last) atomicExch(&a.slots[(long long)c.c_first + s].counter[g], 0);  // ready for the next call
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __syncwarp();  // lane 0's acquire comes before every lane's reads of the clusters' states
  merge_states<8>(
      k1 - k0 + 1,
      [&](int k, float2 &ml, float4 &x0, float4 &x1) {
        const Slot &part = a.slots[(long long)(k == 0 ? c.c_first : (k0 + k) * kClusterCtas) + s];
        ml = __ldcg(&part.ml[h]);
        x0 = __ldcg(reinterpret_cast<const float4 *>(&part.acc[h][d0]));
        x1 = __ldcg(reinterpret_cast<const float4 *>(&part.acc[h][d0 + 4]));
      },
      M, L, r);
  write_merged(a, s, h, d0, L, r);
}

template <int kStages, bool kCluster>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) paged_decode_partial_kernel(const __grid_constant__ DecodeArgs a) {
  using Smem = SmemT<kStages>;
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  // cluster merges: the partial states other CTAs of the cluster push to this one
  RecvArea *recv = reinterpret_cast<RecvArea *>(reinterpret_cast<uint8_t *>(&sm) + sizeof(Smem));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  // Launched with overlap (PKV_OVERLAP_PREVIOUS), the next kernel may start its own set-up
  // now; this one reads the lengths, tables and pool pages at once, and q, the new rows and
  // every global write wait (griddep_wait) until the kernel before it has completed.
  griddep_launch_dependents();
  // cluster merges: no CTA writes into another's shared memory before every CTA of the cluster
  // has started (this arrival, and the wait before the page loop)
  if constexpr (kCluster) cluster_arrive_relaxed();

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      sm.stage_done[i] = 0;
    }
    sm.found = 0;
    sm.seq0 = 0;
    sm.seq0_first = 0;
    sm.issued = 0;
    sm.any_aborted = 0;
    mbar_init_fence();
  }

  // Small grids: the block-table entries are read right after the lengths, so start their
  // lines toward L2 now, spread over the CTAs (each row's first ceil(max_context / 16)
  // entries, and no byte outside them).  (Large grids measured no gain from it.)
  if (kStages == kStagesAlone && tid < 4) {
    const long long row_bytes = (long long)((a.max_context + kPageTokens - 1) / kPageTokens) * 4;
    const long long per_row = (row_bytes + 127) / 128 + 1;
    const long long idx = cta + (long long)tid * G;
    if (row_bytes > 0 && idx < (long long)a.num_seqs * per_row) {
      const long long s = idx / per_row, k = idx % per_row;
      const long long off = k * 128 < row_bytes - 4 ? k * 128 : row_bytes - 4;
      prefetch_l2(reinterpret_cast<const uint8_t *>(a.block_tables + s * a.bt_stride) + off);
    }
  }

  // ... and the query rows, read right after griddep_wait: a prefetch into L2 brings nothing
  // into this SM, so those loads still see whatever the kernel before this one wrote.
  if (kStages == kStagesAlone && tid >= 32 && tid < 40) {
    const long long idx = cta + (long long)(tid - 32) * G;  // 128-byte lines, 32 per sequence
    if (idx < (long long)a.num_seqs * (kQHeads * kHeadDim * 2 / 128))
      prefetch_l2(reinterpret_cast<const uint8_t *>(a.q) + idx * 128);
  }

  // ---- total pages T, and this CTA's range [pa, pb) ----
  // Per thread: pages, sequences with pages, and the least and most pages of one sequence.
  long long mine = 0;
  int n_mine = 0, pmin = 0x7fffffff, pmax = 0;
  bool bad_context = false;  // reported after griddep_wait, like every global write
  for (int i = tid; i < a.num_seqs; i += kThreads) {
    const int c = __ldg(a.context_lens + i);
    const int p = seq_pages(c, a.max_context);
    mine += p;
    if (p > 0) {
      ++n_mine;
      pmin = min(pmin, p);
      pmax = max(pmax, p);
    }
    if (cta == 0 && (c < 0 || c > a.max_context)) bad_context = true;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
    n_mine += __shfl_xor_sync(0xffffffffu, n_mine, o);
    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
  }
  if (lane == 0) {
    sm.warp_sums[warp] = mine;
    sm.warp_n[warp] = n_mine;
    sm.warp_pmin[warp] = pmin;
    sm.warp_pmax[warp] = pmax;
  }
  __syncthreads();
  if (tid == 0) {
    long long t = 0;
    int n = 0, lo = 0x7fffffff, hi = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      t += sm.warp_sums[w];
      n += sm.warp_n[w];
      lo = min(lo, sm.warp_pmin[w]);
      hi = max(hi, sm.warp_pmax[w]);
    }
    sm.total_pages = t;
    sm.used_ctas = effective_ctas(G, t, n, lo, hi, a.split_ctas);
  }
  __syncthreads();
  const long long T = sm.total_pages;
  // zero rows of the sequences that have no pages, spread over all launched CTAs
  auto zero_empty_rows = [&]() {
    for (int s = cta; s < a.num_seqs; s += G) {
      if (seq_pages(__ldg(a.context_lens + s), a.max_context) == 0) {
        float4 *row = reinterpret_cast<float4 *>(a.out + (long long)s * kQHeads * kHeadDim);
        for (int k = tid; k < kQHeads * kHeadDim / 4; k += kThreads) row[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  // The pages are split over Gu <= min(G, T) CTAs, so every CTA below Gu owns at least one page.
  const int Gu = sm.used_ctas;
  if (cta >= Gu) {
    griddep_wait();
    if (bad_context) report(a.status, PKV_DEV_BAD_CONTEXT);
    zero_empty_rows();
    if constexpr (kCluster) {
      // the cluster barriers of the CTAs that hold pages: the start, and after every push
      cluster_wait();
      cluster_sync();
    }
    return;
  }
  const long long pa = (long long)cta * T / Gu, pb = (long long)(cta + 1) * T / Gu;

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

  // ================= warp g: K/V head g, query heads 4g .. 4g+3 =================
  const int g = warp;
  Walk w;  // page being computed
  w.s = sm.seq0;
  w.ctx = __ldg(a.context_lens + w.s);
  w.n = seq_pages(w.ctx, a.max_context);
  w.lp = int(pa - sm.seq0_first);
  Walk wi = w;  // page to issue next (kStages ahead of w once the ring is full)
  const uint64_t policy = policy_evict_first();
  const long long first_fill = count < kStages ? count : kStages;
  if (tid == 0) {
    prefetch_tensormap(&a.tmap_k);
    prefetch_tensormap(&a.tmap_v);
  }
  for (long long j = 0; j < first_fill; ++j) {
    if (tid == 0) issue_page(a, sm, int(j), wi, policy);
    if (j + 1 < count) wi.next(a);
  }
  if (tid == 0) atomicMax(&sm.issued, (unsigned long long)first_fill);
  // the first pages are on their way; what follows reads q and the new rows and writes
  griddep_wait();
  if (bad_context) report(a.status, PKV_DEV_BAD_CONTEXT);
  zero_empty_rows();
  if constexpr (kCluster) cluster_wait();  // every CTA of the cluster has started

  const int quad = lane & 3;     // column pair of the accumulator fragments
  const int hrow = lane >> 2;    // fragment row: query head hrow of the group when < 4
  // ldmatrix row addresses inside a 2 KiB box (lane i addresses row i % 8 of matrix i / 8)
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t krow = uint32_t((((mi >> 1) << 3) + ri) * kRowBytes);  // K: token (mi/2)*8 + ri
  const uint32_t kchunk = uint32_t(mi & 1);                             // + 2 ks
  const uint32_t vrow = uint32_t((((mi & 1) << 3) + ri) * kRowBytes);   // V: token (mi%2)*8 + ri
  const uint32_t vchunk = uint32_t(mi >> 1);                            // + nd
  uint32_t qa[4][2];
  load_q(a, w.s, g, lane, qa);
  float m_run = -INFINITY, l_run = 0.f;
  float o[8][4];
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  bool has_first = (w.lp == 0);
  long long gfirst = pa - w.lp;  // global index of the first page of the current sequence
  bool aborted = false;          // a wait gave up: stop waiting, computing and issuing, keep walking
  struct Pending {
    int s, n, ticket;
    long long gfirst;
  } pend0 = {-1, 0, 0, 0}, pend1 = {-1, 0, 0, 0};  // cut segments whose merge check waits for the end

  for (long long i = 0; i < count; ++i) {
    const int st = int(i % kStages);
    if (!aborted && !mbar_wait(&sm.full[st], uint32_t(i / kStages) & 1)) {
      report(a.status, PKV_DEV_TIMEOUT);
      aborted = true;
    }
    const int valid = min(kPageTokens, w.ctx - w.lp * kPageTokens);
    if (a.slot_mapping != nullptr && w.lp == w.n - 1 && !aborted) {
      // Fused append: the new token is the last of this page, so its slot must be
      // page * 16 + (ctx - 1) % 16 for this page's block-table entry.  Any other slot is
      // reported and ignored (the cached row is attended as it is, nothing is stored).
      // Lanes 0-7 move its K row of head g (16 B each), lanes 8-15 its V row, into the
      // stage (swizzled position) and the pool.
      const long long slot = __ldg(a.slot_mapping + w.s);
      if (slot >= 0) {
        const long long page = __ldg(a.block_tables + (long long)w.s * a.bt_stride + w.lp);
        const int r = valid - 1;
        const bool ok = slot == page * kPageTokens + r && slot < a.num_slots;
        if (ok && lane < 16) {
          const int c = lane & 7, is_v = lane >> 3;
          const uint4 x = __ldg((is_v ? a.v_new : a.k_new) + ((long long)w.s * kKvHeads + g) * 8 + c);
          if (sm.stage_ok[st]) {
            uint8_t *row = sm.kv[st][is_v] + (g * kPageTokens + r) * kRowBytes;
            *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) = x;
          }
          uint8_t *dst = (is_v ? a.v_pool : a.k_pool) + page * a.page_stride +
                         (long long)(g * kPageTokens + r) * kRowBytes + c * 16;
          *reinterpret_cast<uint4 *>(dst) = x;
          fence_proxy_async_smem();  // these generic stores precede the stage's next TMA refill
        } else if (!ok && g == 0 && lane == 0) {
          report(a.status, PKV_DEV_BAD_SLOT);
        }
      }
      __syncwarp();
    }
    if (!aborted && sm.stage_ok[st]) {
      const uint32_t kbase = smem_addr(sm.kv[st][0]) + g * kHeadRowsBytes;
      const uint32_t vbase = smem_addr(sm.kv[st][1]) + g * kHeadRowsBytes;
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
        o[nd][2] *= alpha;
        o[nd][3] *= alpha;
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
        // A rows 0-7 carry P_hi and rows 8-15 P_lo: c0/c1 gather P_hi V, c2/c3 P_lo V.
        mma_16816(o[nd], ph0, pl0, ph1, pl1, v0, v1);
        mma_16816(o[nd + 1], ph0, pl0, ph1, pl1, v2, v3);
      }
    }
    // ---- the last warp done with this stage refills it with the page kStages ahead ----
    // Every ldmatrix result of this stage has been consumed by an instruction above,
    // so the warp's reads are complete once all lanes reach this point.
    __syncwarp();
    if (i + kStages < count) {
      if (lane == 0 && !aborted) {
        if (a.slot_mapping != nullptr && w.lp == w.n - 1) __threadfence_block();  // after the fused-append stores
        const unsigned done = atomicAdd(&sm.stage_done[st], 1u) + 1u;
        if (done % kWarps == 0) {
          issue_page(a, sm, st, wi, policy);
          atomicMax(&sm.issued, (unsigned long long)(i + kStages + 1));
        }
      }
      wi.next(a);
      // the walk ahead entered a new sequence: bring this warp's query rows of it into L2
      if (wi.lp == 0 && lane < kGroup && wi.s < a.num_seqs)
        prefetch_l2(a.q + ((long long)wi.s * kQHeads + g * kGroup + lane) * (kHeadDim / 2));
    }
    if (aborted && lane == 0) sm.any_aborted = 1;

    const bool seq_end = (w.lp == w.n - 1);
    if (seq_end || i == count - 1) {
      // ---- finish this sequence's share: direct output, or a partial state and maybe the merge ----
      float lt = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      if (has_first && seq_end) {
        if (hrow < kGroup) {
          float *dst = a.out + ((long long)w.s * kQHeads + g * kGroup + hrow) * kHeadDim + 2 * quad;
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
          for (int nd = 0; nd < 8; ++nd)
            *reinterpret_cast<float2 *>(dst + 8 * nd) =
                make_float2((o[nd][0] + o[nd][2]) * inv, (o[nd][1] + o[nd][3]) * inv);
        }
      } else {
        // the partial state: into the workspace slot cta + s, or (cluster merges) pushed into
        // the receive area of the CTA that merges this head group
        if (hrow < kGroup) {
          if constexpr (kCluster) {
            const ClusterPlan c = cluster_plan(gfirst, w.n, g, T, Gu, cta);
            GroupState &dst = recv[c.area].slot[(cta - c.lo) * c.qmax + c.slot];  // its address in CTA c.recv
            const uint32_t rank = uint32_t(c.recv - c.cl0);
            const uint32_t acc = cluster_map(smem_addr(&dst.acc[hrow][2 * quad]), rank);
#pragma unroll
            for (int nd = 0; nd < 8; ++nd)
              st_cluster_f2(acc + 32u * nd, make_float2(o[nd][0] + o[nd][2], o[nd][1] + o[nd][3]));
            if (quad == 0) st_cluster_f2(cluster_map(smem_addr(&dst.ml[hrow]), rank), make_float2(m_run, lt));
          } else {
            Slot &mine = a.slots[(long long)cta + w.s];
            float *acc = &mine.acc[g * kGroup + hrow][2 * quad];
#pragma unroll
            for (int nd = 0; nd < 8; ++nd)
              *reinterpret_cast<float2 *>(acc + 8 * nd) = make_float2(o[nd][0] + o[nd][2], o[nd][1] + o[nd][3]);
            if (quad == 0) mine.ml[g * kGroup + hrow] = make_float2(m_run, lt);
          }
        }
        // The ticket is looked at after the loop, so that its round trip (and a merge) do not
        // stall the pages that follow.  A range holds at most two cut segments: its first
        // (begun in an earlier range) and its last (going on in a later one).
        int ticket = 0;
        if constexpr (!kCluster) ticket = ticket_of(a, w.s, gfirst, w.n, g, lane, T, Gu, cta);
        Pending &p = pend0.s < 0 ? pend0 : pend1;
        p.s = w.s;
        p.gfirst = gfirst;
        p.n = w.n;
        p.ticket = ticket;
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
  if constexpr (kCluster) {
    cluster_sync();  // every push of the cluster has landed
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
      const Pending p = k == 0 ? pend0 : pend1;
      if (p.s >= 0) cluster_merge(a, recv, p.s, p.gfirst, p.n, g, lane, T, Gu, cta);
    }
  } else {
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
      const Pending p = k == 0 ? pend0 : pend1;
      if (p.s >= 0) merge_if_last(a, p.s, p.gfirst, p.n, g, lane, T, Gu, p.ticket, cta);
    }
  }
  named_barrier_sync(1, kThreads);
  if (tid == 0 && sm.any_aborted) {
    // Copies issued for pages nobody consumed: wait (bounded) so none lands after exit.
    const long long issued = (long long)sm.issued;
    const long long first = issued > kStages ? issued - kStages : 0;
    for (long long j = first; j < issued; ++j) mbar_wait(&sm.full[int(j % kStages)], uint32_t(j / kStages) & 1);
  }
}

// The workspace is an array of kMaxCtas + num_seqs slots.  Slot positions do not
// depend on num_seqs, so the ticket counters (zero between calls) stay valid when
// the batch size changes.
size_t workspace_bytes(int num_seqs) { return (size_t(kMaxCtas) + size_t(num_seqs)) * sizeof(Slot); }

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

// The three kernel instances: two CTAs per SM with the shallow ring; one CTA per SM with the
// deep ring; the same in clusters of kClusterCtas that merge cut sequences on chip.
using KernelFn = void (*)(DecodeArgs);
constexpr KernelFn kKernelShared = paged_decode_partial_kernel<kStagesShared, false>;
constexpr KernelFn kKernelAlone = paged_decode_partial_kernel<kStagesAlone, false>;
constexpr KernelFn kKernelCluster = paged_decode_partial_kernel<kStagesAlone, true>;

int setup_kernel_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(kKernelShared, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(smem_bytes<kStagesShared, false>()));
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(kKernelAlone, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes<kStagesAlone, false>()));
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(kKernelCluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes<kStagesAlone, true>()));
  });
  return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Most CTAs of the clustered instance resident at once on the current device (a multiple of
// kClusterCtas), 0 when it cannot be determined.
int cluster_capacity() {
  static std::mutex mu;
  static int cap[64];
  static bool known[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!known[dev]) {
    if (setup_kernel_attributes() != PKV_OK) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterCtas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<kStagesAlone, true>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kKernelCluster, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cap[dev] = n > 0 ? n * kClusterCtas : 0;
    known[dev] = true;
  }
  return cap[dev];
}

// Kernel instance and grid for a split over G CTAs: clusters when there is more than one CTA
// and every cluster of the grid can be resident at once (a grid the kernel sizes itself that
// would fit the SMs but not the clusters is cut to the cluster capacity), else one CTA per SM
// with the deep ring when G fits the SMs, else two CTAs per SM.
struct LaunchChoice {
  KernelFn kernel;
  size_t smem;
  int grid;
  int cluster;  // CTAs per cluster, 1 without
};

LaunchChoice choose_launch(int G, bool caller_chose) {
  const int cap = cluster_capacity();
  if (!caller_chose && G > cap && G <= device_sm_count()) G = cap;
  if (G >= 2 && G <= cap) {
    const int grid = (G + kClusterCtas - 1) / kClusterCtas * kClusterCtas;
    return {kKernelCluster, smem_bytes<kStagesAlone, true>(), grid, kClusterCtas};
  }
  if (G <= device_sm_count()) return {kKernelAlone, smem_bytes<kStagesAlone, false>(), G, 1};
  return {kKernelShared, smem_bytes<kStagesShared, false>(), G, 1};
}

int decode(const pkv_pool *pool, float *out, const void *q, int num_q_heads, const int32_t *block_tables,
           int64_t bt_stride, const int32_t *context_lens, int num_seqs, int max_context, float scale,
           void *workspace, size_t workspace_bytes, int32_t *device_status, int num_ctas, void *stream,
           const void *k_new = nullptr, const void *v_new = nullptr, const int32_t *slot_mapping = nullptr,
           unsigned flags = 0) {
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
  if (workspace_bytes < pkv::workspace_bytes(num_seqs)) return PKV_ERR_WORKSPACE;
  rc = setup_kernel_attributes();
  if (rc != PKV_OK) return rc;

  DecodeArgs a;
  rc = pool_tensor_maps(pool, kKvHeads * kPageTokens, &a.tmap_k, &a.tmap_v);
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
  a.slots = static_cast<Slot *>(workspace);
  a.status = device_status;

  a.split_ctas = num_ctas;
  a.k_new = static_cast<const uint4 *>(k_new);
  a.v_new = static_cast<const uint4 *>(v_new);
  a.slot_mapping = slot_mapping;
  a.k_pool = static_cast<uint8_t *>(pool->k_base);
  a.v_pool = static_cast<uint8_t *>(pool->v_base);
  a.page_stride = pool->page_stride_bytes;
  a.num_slots = (long long)pool->num_pages * pool->page_tokens;
  const LaunchChoice lc = num_ctas > 0 ? choose_launch(num_ctas, true) : choose_launch(auto_ctas(num_seqs, max_context), false);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(lc.grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = lc.smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  if (lc.cluster > 1) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = unsigned(lc.cluster);
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (flags & PKV_OVERLAP_PREVIOUS) {
    // programmatic stream serialization: the kernel may start while the previous kernel on
    // the stream finishes (see griddep_launch_dependents / griddep_wait in the kernel)
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = unsigned(n_attr);
  if (cudaLaunchKernelEx(&cfg, lc.kernel, a) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_LAUNCH;
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim) {
  if (num_seqs < 0 || num_q_heads != pkv::kQHeads || head_dim != pkv::kHeadDim) return 0;
  return pkv::workspace_bytes(num_seqs);
}

extern "C" int pkv_decode_max_ctas(void) { return pkv::kMaxCtas; }

extern "C" int pkv_decode_plan(int num_seqs, int max_context, int *num_ctas, int *launches) {
  if (num_seqs < 0 || max_context < 0) return PKV_ERR_SHAPE;
  const int g = num_seqs == 0 ? 0 : pkv::choose_launch(pkv::auto_ctas(num_seqs, max_context), false).grid;
  if (num_ctas) *num_ctas = g;
  if (launches) *launches = num_seqs == 0 ? 0 : 1;
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

extern "C" int pkv_decode_step(const pkv_pool *pool, const void *k_new, const void *v_new,
                               const int32_t *slot_mapping, float *out, const void *q, int num_q_heads,
                               const int32_t *block_tables, int64_t block_table_stride, const int32_t *context_lens,
                               int num_seqs, int max_context, float scale, void *workspace, size_t workspace_bytes,
                               int32_t *device_status, void *stream) {
  return pkv_decode_step_ex(pool, k_new, v_new, slot_mapping, out, q, num_q_heads, block_tables, block_table_stride,
                            context_lens, num_seqs, max_context, scale, workspace, workspace_bytes, device_status, 0u,
                            stream);
}

extern "C" int pkv_decode_step_ex(const pkv_pool *pool, const void *k_new, const void *v_new,
                                  const int32_t *slot_mapping, float *out, const void *q, int num_q_heads,
                                  const int32_t *block_tables, int64_t block_table_stride, const int32_t *context_lens,
                                  int num_seqs, int max_context, float scale, void *workspace, size_t workspace_bytes,
                                  int32_t *device_status, unsigned flags, void *stream) {
  if (flags & ~unsigned(PKV_OVERLAP_PREVIOUS)) return PKV_ERR_SHAPE;
  if (num_seqs > 0 && (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr)) return PKV_ERR_NULL;
  if (num_seqs > 0 && (!pkv::aligned16(k_new) || !pkv::aligned16(v_new) ||
                       (reinterpret_cast<uintptr_t>(slot_mapping) & 3u)))
    return PKV_ERR_ALIGN;
  return pkv::decode(pool, out, q, num_q_heads, block_tables, block_table_stride, context_lens, num_seqs,
                     max_context, scale, workspace, workspace_bytes, device_status, 0, stream, k_new, v_new,
                     slot_mapping, flags);
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
// for callers that cannot allocate device memory.  On the first call with a
// device current, its device address is looked up (cudaGetSymbolAddress) and the
// array is cleared once on the caller's stream, ahead of that call's kernel (the
// ticket counters must start at zero; every completed call leaves them at zero
// again).  The call then follows the regular path with that address as the
// workspace.
namespace pkv {
namespace {

constexpr size_t kNoallocScratchBytes = (size_t(kMaxCtas) + PKV_NOALLOC_MAX_SEQS) * sizeof(Slot);

}  // namespace
}  // namespace pkv

static __device__ __align__(256) unsigned char pkv_noalloc_scratch[pkv::kNoallocScratchBytes];

namespace pkv {
namespace {

// Device address of pkv_noalloc_scratch on the current device, or nullptr.  The first
// call per device enqueues the clear on `stream`, so the kernel enqueued after it on the
// same stream sees a zeroed array whatever kind of stream it is (a non-blocking stream
// is not ordered after work on the legacy default stream).
void *noalloc_scratch_address(cudaStream_t stream) {
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
    if (cudaMemsetAsync(p, 0, kNoallocScratchBytes, stream) != cudaSuccess) {
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
  void *scratch = pkv::noalloc_scratch_address(static_cast<cudaStream_t>(stream));
  if (scratch == nullptr) return PKV_ERR_CUDA;
  return pkv::decode(pool, out, q, num_q_heads, block_tables, block_table_stride, context_lens, num_seqs,
                     max_context, scale, scratch, pkv::kNoallocScratchBytes, device_status, 0, stream);
}
