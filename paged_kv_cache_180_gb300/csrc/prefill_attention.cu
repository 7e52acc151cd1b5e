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
//  * Tile: 32 query tokens of a sequence against one K/V head g.  Its 128 rows
//    (row = 4 * token + head in group) share every K/V row loaded: M = 128.  The
//    grid is persistent (two CTAs per SM); the tiles are numbered latest-first (the
//    longest causal spans start first) and dealt to the CTAs in a snake, forward on even
//    rounds and backward on odd ones, which evens out the CTAs' key blocks.
//  * Keys in blocks of 64 (4 pages).  S = Q K^T is 4 tcgen05.mma (M 128, N 64,
//    K 16; Q and K K-major, 128-byte swizzled) into one of two TMEM S buffers, so
//    S of block j + 1 runs while the softmax works on block j.  P, as bf16 hi + lo
//    halves (the weights keep ~16 significant bits), is stored back over its own S
//    and read by O += P V as the TMEM A operand: 8 tcgen05.mma of N 80, B being V
//    (MN-major, 128-byte swizzled) followed by 16 columns of a constant "ones" atom,
//    so O's column 64 accumulates the row sum of exactly the weights used.
//  * Warp roles: warps 0-3 own one row each per thread (TMEM lane = row): they read
//    S, mask, keep the row's reference maximum, write P, and finally read O, divide
//    and store.  Warp 4 loads by tiled TMA: the next tile's Q (one 16 KiB box of 32
//    query rows x 4 heads; two Q buffers) and head g's K and V rows of each page
//    (2 KiB boxes) into a 4-stage ring; pages past the query span come from a
//    coordinate outside the pool, which TMA fills with zeros.  Warp 5 owns the TMEM
//    allocation and issues the MMAs from one thread (S of block j, then P V of block
//    j - 1), completion signalled by tcgen05.commit.
//  * Online softmax in the exp2 domain with a lazily moved maximum: a row's
//    reference moves only when a block's maximum exceeds it by more than 8 (a
//    factor 256), and only then is the row of O (with its sum column) rescaled in
//    TMEM, after the previous P V completed.  The final division uses the same
//    reference, so the result is the exact softmax up to rounding.  A negative
//    scale takes the reference from -s.
//  * Masks: keys after a row's position and the keys of invalid pages get weight 0;
//    V rows at or past the context in a sequence's last page are zeroed in shared
//    memory so stale pool bytes (even NaN) never reach O.
//  * The P-ready and P V-done barriers exist per P buffer: with a single barrier a
//    softmax warp already on the next block could complete a phase for a slower warp.
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

constexpr int kPfTok = 32;                             // query tokens per tile
constexpr int kPfRows = kPfTok * kGroup;               // M = 128
constexpr int kPfKeys = 64;                            // keys per block
constexpr int kPfPagesPerBlock = kPfKeys / kPageTokens;
constexpr int kPfStages = 4;                           // K/V blocks in flight
constexpr int kPfThreads = 192;                        // warps 0-3 softmax, 4 loads, 5 MMA
constexpr int kPfCtasPerSm = 2;
constexpr int kPfMaxTiles = 64;                        // tiles one CTA walks (its tile table in shared memory)
constexpr int kPfBox = kPageTokens * kRowBytes;        // one head's rows of one page: 2 KiB
constexpr int kPfTileBytes = kPfKeys * kRowBytes;      // K (or V) of one block: 8 KiB
constexpr uint32_t kPfTmemCols = 256;
constexpr uint32_t kColS = 0;                          // S buffers at columns 0 and 64
constexpr uint32_t kColO = 128;                        // O: columns 128 .. 191, row sum l at 192 (193 .. 207 zero)
constexpr int kPvN = kHeadDim + 16;                    // P V's N: V's 64 columns and 16 of the ones atom
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;                    // move a row's reference max when exceeded by more

constexpr uint32_t kIdescS = idesc_bf16(kPfRows, kPfKeys, false);   // B = K rows (K-major)
constexpr uint32_t kIdescPV = idesc_bf16(kPfRows, kPvN, true);  // B = [V | ones] (MN-major)

struct PrefillArgs {
  CUtensorMap tmap_k;  // boxes of one head's 16 rows of one page
  CUtensorMap tmap_v;
  CUtensorMap tmap_q;  // boxes of 32 query rows x one group's 4 heads (rows past num_q_rows read as zeros)
  int num_pages;
  float *out;      // [total][32][64]
  const int32_t *query_start;
  const int32_t *block_tables;
  long long bt_stride;
  const int32_t *context_lens;
  int num_seqs;
  int num_q_rows;
  int max_context;
  int tiles_per_seq;
  int num_tiles;  // num_seqs * tiles_per_seq * 8
  float scale_log2;   // |scale| * log2(e)
  float move_thresh;  // scores (unscaled) by which a block's max must pass the reference to move it
  int neg;            // scale < 0: a row's reference is the max of -s (the min of s)
  int32_t *status;
};

// One work tile: 32 query tokens of sequence s (from t0) against K/V head g.
struct PfTile {
  int s, g, t0, n, q0, ctx, nblocks, npages;
  int run;      // has queries and a valid context
  int invalid;  // has queries, invalid context: its rows are zeroed
};

struct __align__(1024) PfSmem {
  uint8_t q[2][kPfRows * kRowBytes];       // two tiles' Q, row = 4 * token + head, 128-byte swizzled
  uint8_t k[kPfStages][kPfTileBytes];      // 64 keys x 128 B per stage
  uint8_t v[kPfStages][kPfTileBytes];
  uint8_t ones[kPfTileBytes];              // the second MN atom of P V's B: 1 in column 0 of every key row
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t kv_full[kPfStages];
  uint64_t kv_empty[kPfStages];
  uint64_t s_full[2];
  uint64_t s_free[2];  // the P V that read a buffer's P is done: S may be written again
  uint64_t p_full[2];  // per P buffer: every softmax thread wrote its row of P (one barrier per
                       // buffer, so a thread already on the next block cannot complete this phase)
  uint64_t p_free[2];  // per P buffer: the P V of a block done (O, and everything before, may be read);
                       // per buffer so that the phase waited for is never two behind
  uint64_t mma_done;
  int kv_bad[kPfStages];  // per stage: bit pp set when page pp of the block is invalid (loaded as zeros)
  PfTile tiles[kPfMaxTiles];  // this CTA's tiles in walking order, read once from global memory
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kPfSmemBytes = sizeof(PfSmem) + 1024;

// Tile ti of the grid-wide list: latest token tiles first, then sequence, then K/V head.
__device__ __forceinline__ PfTile pf_tile(const PrefillArgs &a, int ti) {
  PfTile t;
  const int per_rank = a.num_seqs * kKvHeads;
  const int rank = ti / per_rank, rem = ti % per_rank;
  t.s = rem / kKvHeads;
  t.g = rem % kKvHeads;
  t.t0 = (a.tiles_per_seq - 1 - rank) * kPfTok;
  t.q0 = __ldg(a.query_start + t.s);
  t.n = __ldg(a.query_start + t.s + 1) - t.q0;
  t.ctx = __ldg(a.context_lens + t.s);
  const bool has = t.n > 0 && t.t0 < t.n;
  t.invalid = has && (t.ctx < 0 || t.ctx > a.max_context || t.n > t.ctx || t.q0 < 0 || t.q0 + t.n > a.num_q_rows);
  t.run = has && !t.invalid;
  const int last_pos = t.run ? t.ctx - t.n + min(t.t0 + kPfTok, t.n) - 1 : 0;
  t.nblocks = last_pos / kPfKeys + 1;
  t.npages = last_pos / kPageTokens + 1;  // pages holding keys 0 .. last_pos
  return t;
}

// Bounded wait that gives up at once when another role has already aborted.
// Returns true when the phase completed.
__device__ __forceinline__ bool pf_wait(PfSmem &sm, uint64_t *bar, uint32_t parity, int32_t *status) {
  if (*reinterpret_cast<volatile int *>(&sm.abort)) return false;
  if (mbar_wait(bar, parity)) return true;
  *reinterpret_cast<volatile int *>(&sm.abort) = 1;
  report(status, PKV_DEV_TIMEOUT);
  return false;
}

template <bool kMin>
__device__ __forceinline__ float ext3(float a, float b, float c) {
  return kMin ? min3f(a, b, c) : max3f(a, b, c);
}

// Largest (kMin: smallest) of 64 values: a tree of three-input max (32 instructions, 4 deep).
template <bool kMin>
__device__ __forceinline__ float extreme64(const float (&x)[64]) {
  float m[22];
#pragma unroll
  for (int i = 0; i < 21; ++i) m[i] = ext3<kMin>(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  m[21] = x[63];
  float n[8];
#pragma unroll
  for (int i = 0; i < 7; ++i) n[i] = ext3<kMin>(m[3 * i], m[3 * i + 1], m[3 * i + 2]);
  n[7] = m[21];
  const float a = ext3<kMin>(n[0], n[1], n[2]), b = ext3<kMin>(n[3], n[4], n[5]);
  const float c = kMin ? fminf(n[6], n[7]) : fmaxf(n[6], n[7]);
  return ext3<kMin>(a, b, c);
}

// max over the keys whose bit in `valid` is set of sigma * s, sigma = -1 when neg.
__device__ __forceinline__ float signed_max(const float (&sv)[64], bool masked, uint64_t valid, bool neg) {
  if (!masked) return neg ? -extreme64<true>(sv) : extreme64<false>(sv);
  float xm[64];
  const float off = neg ? INFINITY : -INFINITY;
#pragma unroll
  for (int c = 0; c < 64; ++c) xm[c] = (valid >> c) & 1 ? sv[c] : off;
  return neg ? -extreme64<true>(xm) : extreme64<false>(xm);
}

// P = 2^((s - m) * c) for the 64 keys of a block as bf16 hi + lo parts, keys 2i and
// 2i + 1 packed in word i; with kMasked, keys whose bit in `valid` is clear get 0.
template <bool kMasked>
__device__ __forceinline__ void block_probs(const float (&sv)[64], uint64_t valid, float m, float2 c2,
                                            uint32_t (&hi)[32], uint32_t (&lo)[32]) {
  // exponent arguments (s - m) c as one packed fused multiply-add: s c + (-m c)
  const float2 mc = make_float2(-m * c2.x, -m * c2.y);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float2 e = fma_f32x2(make_float2(sv[2 * i], sv[2 * i + 1]), c2, mc);
    float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
    if (kMasked) {
      p0 = (valid >> (2 * i)) & 1 ? p0 : 0.f;
      p1 = (valid >> (2 * i + 1)) & 1 ? p1 : 0.f;
    }
    hi[i] = pack_bf16x2(p0, p1);
    const float2 r = sub_f32x2(make_float2(p0, p1), make_float2(bf16_lo(hi[i]), bf16_hi(hi[i])));
    lo[i] = pack_bf16x2(r.x, r.y);
  }
}

// Persistent: each CTA walks its tiles of the snake order (at most kPfMaxTiles;
// their descriptors are read from global memory once, in parallel, into shared memory).
// Every role walks the same table and skips the same tiles, so their running block
// counters agree.  The loader fetches the next tile's Q and block-table entries while the
// current tile computes; the MMA warp starts the next tile's S during the current one's
// last blocks; the softmax warps finish a tile (read O, divide, store) only after writing
// P for the next tile's first block, so the wait for the last P V overlaps useful work.
__global__ void __launch_bounds__(kPfThreads, kPfCtasPerSm) paged_prefill_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  PfSmem &sm = *reinterpret_cast<PfSmem *>(smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Tile k of this CTA: k * G + c on even rounds and k * G + (G - 1 - c) on odd ones, a snake
  // over the latest-first list that evens out the CTAs' key blocks.
  const int G = int(gridDim.x), c = int(blockIdx.x);
  auto tile_index = [&](int k) { return k * G + ((k & 1) ? G - 1 - c : c); };
  int nt = 0;  // <= kPfMaxTiles
  while (nt < kPfMaxTiles && tile_index(nt) < a.num_tiles) ++nt;

  if (tid < nt) sm.tiles[tid] = pf_tile(a, tile_index(tid));
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 1);
    }
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&sm.kv_full[i], 1);
      mbar_init(&sm.kv_empty[i], 1);
    }
    mbar_init(&sm.p_full[0], kPfRows);
    mbar_init(&sm.p_full[1], kPfRows);
    mbar_init(&sm.p_free[0], 1);
    mbar_init(&sm.p_free[1], 1);
    mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    mbar_init_fence();
  }
  if (tid < kPfRows) {
    // ones block: key row r (of 64) holds bf16 1.0 in element 0 (its 128-byte-swizzled position)
    for (int i = tid; i < kPfKeys * 8; i += kPfRows) {
      const int r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4 *>(sm.ones + r * kRowBytes + ((c ^ (r & 7)) << 4)) =
          make_uint4(c == 0 ? 0x3f80u : 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (warp == 5) tmem_alloc(&sm.tmem_base, kPfTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // index of the first running tile at or after k
  auto next_run = [&](int k) {
    while (k < nt && !sm.tiles[k].run) ++k;
    return k;
  };

  if (warp == 4) {
    // ================= loader: Q tiles and K/V blocks (tiled TMA) =================
    const uint64_t policy = policy_evict_last();
    const uint64_t policy_q = policy_evict_first();  // each query row is read by one tile
    if (lane == 0) {
      prefetch_tensormap(&a.tmap_k);
      prefetch_tensormap(&a.tmap_v);
      prefetch_tensormap(&a.tmap_q);
    }
    // block-table entries of a tile's first 128 pages: page lp sits in lane lp % 32, slot lp / 32
    auto load_entries = [&](const PfTile &t, int (&e)[4]) {
      const int32_t *table = a.block_tables + (long long)t.s * a.bt_stride;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int lp = lane + 32 * k;
        e[k] = lp < t.npages ? __ldg(table + lp) : -1;
      }
    };
    // Q of tile t into buffer qb: one tiled TMA box of 32 query rows x the group's 4 heads,
    // landing as rows 4 * token + head, 128-byte swizzled (rows past num_q_rows read as zeros;
    // padding rows past n are the next sequence's queries: computed, never written)
    auto load_q = [&](const PfTile &t, int qb) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full[qb], kPfRows * kRowBytes);
        tma_load_3d(sm.q[qb], &a.tmap_q, 0, t.g * kGroup, t.q0 + t.t0, &sm.q_full[qb], policy_q);
      }
      __syncwarp();
    };
    long long gb = 0;  // K/V blocks issued so far
    int lt = 0;        // running tiles started so far
    bool ok = true;
    int k = next_run(0);
    int ent[4] = {-1, -1, -1, -1};
    if (k < nt) {
      load_entries(sm.tiles[k], ent);
      load_q(sm.tiles[k], 0);
    }
    // launched with overlap (PKV_OVERLAP_PREVIOUS), the kernel before this one (the append of
    // the prompt's K/V) may still be running: the pages are read only once it has completed
    griddep_wait();
    while (ok && k < nt) {
      const PfTile t = sm.tiles[k];
      const int kn = next_run(k + 1);
      int ent_next[4] = {-1, -1, -1, -1};
      if (kn < nt) load_entries(sm.tiles[kn], ent_next);  // in flight while this tile's blocks go out
      const int32_t *table = a.block_tables + (long long)t.s * a.bt_stride;
      for (int j = 0; j < t.nblocks; ++j, ++gb) {
        const int st = int(gb % kPfStages);
        if (gb >= kPfStages) {
          const bool w = pf_wait(sm, &sm.kv_empty[st], uint32_t(gb / kPfStages - 1) & 1, a.status);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
        }
        int page[kPfPagesPerBlock], bad = 0;
#pragma unroll
        for (int pp = 0; pp < kPfPagesPerBlock; ++pp) {
          const int lp = j * kPfPagesPerBlock + pp;
          int e;
          if (lp < 128) {
            const int q = lp >> 5;
            e = __shfl_sync(0xffffffffu, q == 0 ? ent[0] : q == 1 ? ent[1] : q == 2 ? ent[2] : ent[3], lp & 31);
          } else {
            e = lp < t.npages ? __ldg(table + lp) : -1;
          }
          page[pp] = -1;  // outside the pool: TMA fills the box with zeros
          if (lp < t.npages) {
            if (e >= 0 && e < a.num_pages)
              page[pp] = e;
            else
              bad |= 1 << pp;
          }
        }
        if (lane == 0) {
          if (bad) report(a.status, PKV_DEV_BAD_PAGE);
          sm.kv_bad[st] = bad;
          mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kPfTileBytes);
#pragma unroll
          for (int pp = 0; pp < kPfPagesPerBlock; ++pp) {
            tma_load_3d(sm.k[st] + pp * kPfBox, &a.tmap_k, 0, t.g * kPageTokens, page[pp], &sm.kv_full[st], policy);
            tma_load_3d(sm.v[st] + pp * kPfBox, &a.tmap_v, 0, t.g * kPageTokens, page[pp], &sm.kv_full[st], policy);
          }
        }
        __syncwarp();
        if (j == min(1, t.nblocks - 1) && kn < nt) {
          // the next tile's Q, once the tile before this one released its buffer
          const int qb = (lt + 1) & 1;
          if (lt + 1 >= 2) {
            const bool w = pf_wait(sm, &sm.q_empty[qb], uint32_t((lt + 1) / 2 - 1) & 1, a.status);
            if (!__all_sync(0xffffffffu, w)) {
              ok = false;
              break;
            }
          }
          load_q(sm.tiles[kn], qb);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) ent[q] = ent_next[q];
      k = kn;
      ++lt;
    }
    // every copy issued has landed before the CTA exits
    if (lane == 0)
      for (long long j = gb > kPfStages ? gb - kPfStages : 0; j < gb; ++j)
        mbar_wait(&sm.kv_full[int(j % kPfStages)], uint32_t(j / kPfStages) & 1);
    __syncwarp();
  } else if (warp == 5) {
    // ================= MMA issuer (one thread issues, the warp waits) =================
    long long gb = 0;          // blocks whose S was issued
    long long pend = -1;       // block whose P V is still to issue
    bool pend_first = false;   // ... and whether it starts its tile (O is overwritten, not accumulated)
    int lt = 0;
    bool ok = true;
    auto issue_pv = [&]() {
      bool w = pf_wait(sm, &sm.p_full[pend & 1], uint32_t(pend >> 1) & 1, a.status);
      if (!__all_sync(0xffffffffu, w)) return false;
      tc_fence_after();
      if (lane == 0) {
        const int st = int(pend % kPfStages), b = int(pend & 1);
        const uint32_t vb = smem_addr(sm.v[st]);
        const uint32_t pa = tmem + kColS + b * kPfKeys;  // P hi in its 32 first columns, P lo in the next 32
        const uint32_t to_ones = smem_addr(sm.ones) - vb;  // stride to the second (ones) MN atom
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_tmem_a(tmem + kColO, pa + kk * 8, sw128_desc(vb + kk * 2048, to_ones, 1024), kIdescPV,
                        (pend_first && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_tmem_a(tmem + kColO, pa + 32 + kk * 8, sw128_desc(vb + kk * 2048, to_ones, 1024), kIdescPV, 1u);
        tc_commit(&sm.p_free[b]);
        tc_commit(&sm.kv_empty[st]);
        tc_commit(&sm.s_free[b]);
      }
      __syncwarp();
      pend = -1;
      return true;
    };
    for (int k = next_run(0); ok && k < nt; k = next_run(k + 1)) {
      const PfTile t = sm.tiles[k];
      const int qb = lt & 1;
      bool w = pf_wait(sm, &sm.q_full[qb], uint32_t(lt / 2) & 1, a.status);
      if (!__all_sync(0xffffffffu, w)) break;
      const uint32_t q_base = smem_addr(sm.q[qb]);
      for (int j = 0; j < t.nblocks; ++j, ++gb) {
        const int st = int(gb % kPfStages), b = int(gb & 1);
        w = pf_wait(sm, &sm.kv_full[st], uint32_t(gb / kPfStages) & 1, a.status);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        // V rows at or past the context (stale pool bytes) in this block become zeros
        const int z0 = max(t.ctx, j * kPfKeys), z1 = min(t.npages * kPageTokens, (j + 1) * kPfKeys);
        if (z0 < z1) {
          uint8_t *vt = sm.v[st];
          for (int idx = lane; idx < (z1 - z0) * 8; idx += 32)
            *reinterpret_cast<uint4 *>(vt + (z0 - j * kPfKeys + idx / 8) * kRowBytes + (idx % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (gb >= 2) {
          w = pf_wait(sm, &sm.s_free[b], uint32_t(gb / 2 - 1) & 1, a.status);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kb = smem_addr(sm.k[st]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(tmem + kColS + b * kPfKeys, sw128_desc(q_base + kk * 32, 16, 1024),
                   sw128_desc(kb + kk * 32, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          tc_commit(&sm.s_full[b]);
          if (j == t.nblocks - 1) tc_commit(&sm.q_empty[qb]);  // the tile's last read of its Q
        }
        __syncwarp();
        if (pend >= 0 && !issue_pv()) {
          ok = false;
          break;
        }
        pend = gb;
        pend_first = (j == 0);
      }
      ++lt;
    }
    if (ok && pend >= 0) issue_pv();
    // every MMA issued has completed before the tensor memory is freed
    if (lane == 0) {
      tc_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0);
    }
    __syncwarp();
  } else {
    // ================= softmax warps: thread = row = 4 * token + head =================
    griddep_wait();  // the first global write below comes after the kernel before this one
    const int r = tid, tok = r >> 2, hh = r & 3;
    const uint32_t lane_base = tmem + (uint32_t(32 * warp) << 16);
    long long gb = 0;
    bool ok = true;
    // the tile whose O is still to be read, divided and stored
    bool fin = false;
    int fin_q0 = 0, fin_t0 = 0, fin_n = 0, fin_g = 0;
    auto finish = [&]() {
      // wait for the tile's last P V (global block gb - 1); O, and its row-sum column, are final
      const bool w = pf_wait(sm, &sm.p_free[(gb - 1) & 1], uint32_t((gb - 1) >> 1) & 1, a.status);
      if (!__all_sync(0xffffffffu, w)) return false;
      tc_fence_after();
      const float l_sum = __uint_as_float(tmem_ld1(lane_base + kColO + kHeadDim));
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      float *dst = a.out + ((long long)(fin_q0 + fin_t0 + tok) * kQHeads + fin_g * kGroup + hh) * kHeadDim;
      const bool wide = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        tmem_ld32(lane_base + kColO + 32 * half, o);
        if (fin_t0 + tok < fin_n) {
          if (wide) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              const float v[8] = {__uint_as_float(o[c]) * inv,     __uint_as_float(o[c + 1]) * inv,
                                  __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv,
                                  __uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv,
                                  __uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv};
              st_global_v8(dst + 32 * half + c, v);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4 *>(dst + 32 * half + c) =
                  make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                              __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
          }
        }
      }
      fin = false;
      return true;
    };
    for (int k = 0; ok && k < nt; ++k) {
      const PfTile t = sm.tiles[k];
      if (t.invalid) {
        // invalid sequence: zero this tile's rows (its tokens, query heads 4g .. 4g+3)
        if (t.t0 == 0 && t.g == 0 && tid == 0) report(a.status, PKV_DEV_BAD_CONTEXT);
        const int rows = min(kPfTok, t.n - t.t0) * kGroup * kHeadDim;
        for (int i = tid; i < rows; i += kPfRows) {
          const long long row = (long long)t.q0 + t.t0 + i / (kGroup * kHeadDim);
          if (row >= 0 && row < a.num_q_rows)
            a.out[(row * kQHeads + t.g * kGroup) * kHeadDim + i % (kGroup * kHeadDim)] = 0.f;
        }
        continue;
      }
      if (!t.run) continue;
      const int pos = t.ctx - t.n + min(t.t0 + tok, t.n - 1);
      // reference max of the row's sigma * s (sigma = sign of scale): the exponents are
      // |scale| log2(e) (sigma s - m) = (sigma |scale| log2(e)) (s - sigma m)
      float m_ref = -INFINITY;
      const float sig = a.neg ? -1.f : 1.f;
      const float2 c2 = make_float2(sig * a.scale_log2, sig * a.scale_log2);
      for (int j = 0; j < t.nblocks; ++j, ++gb) {
        const int b = int(gb & 1), st = int(gb % kPfStages);
        // S of block j, and (already complete) the stage's load, for its bad-page mask
        bool w = pf_wait(sm, &sm.s_full[b], uint32_t(gb >> 1) & 1, a.status) &&
                 pf_wait(sm, &sm.kv_full[st], uint32_t(gb / kPfStages) & 1, a.status);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[64];
        {
          uint32_t x0[32], x1[32];
          tmem_ld32(lane_base + kColS + b * kPfKeys, x0);
          tmem_ld32(lane_base + kColS + b * kPfKeys + 32, x1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = __uint_as_float(x0[c]);
            sv[32 + c] = __uint_as_float(x1[c]);
          }
        }
        // keys after this row's position, and the keys of invalid pages (loaded as
        // zeros), are masked: left out of the max, weight 0
        const int key0 = j * kPfKeys;
        const int bad = sm.kv_bad[st];
        const bool masked = !(key0 + kPfKeys - 1 <= pos && bad == 0);
        uint64_t valid = ~0ull;
        if (masked) {
          // keys c <= pos - key0 are causal; each invalid page clears its 16 keys
          const int lim = pos - key0;
          valid = lim >= kPfKeys - 1 ? ~0ull : (lim < 0 ? 0ull : (2ull << lim) - 1ull);
#pragma unroll
          for (int pp = 0; pp < kPfPagesPerBlock; ++pp)
            if ((bad >> pp) & 1) valid &= ~(0xffffull << (pp * kPageTokens));
        }
        const float mx = signed_max(sv, masked, valid, a.neg != 0);  // in units of sigma * s
        // move the reference max only on a row's first block or when this block's max
        // passes it by more than 8 in the exponent (a factor 2^8)
        const bool move = j == 0 || mx > m_ref + a.move_thresh;
        float alpha = 1.f;
        if (move) {
          alpha = ex2_approx((m_ref - mx) * a.scale_log2);
          m_ref = mx;
        }
        // P = 2^((s - m) * scale log2 e) as bf16 hi + lo, keys 2c and 2c + 1 packed in
        // column c (the A operand of P V); the row sum comes from P V's ones column
        uint32_t hi[32], lo[32];
        if (!masked)
          block_probs<false>(sv, valid, sig * m_ref, c2, hi, lo);
        else
          block_probs<true>(sv, valid, sig * m_ref, c2, hi, lo);
        // P overwrites this block's S in tensor memory (its S is in registers; the P V
        // that last read this buffer finished before S was written)
        tmem_st32(lane_base + kColS + b * kPfKeys, hi);
        tmem_st32(lane_base + kColS + b * kPfKeys + 32, lo);
        if (j == 0 && fin && !finish()) {  // the previous tile's P V is done once this P is out
          ok = false;
          break;
        }
        if (j >= 1 && __any_sync(0xffffffffu, move)) {
          // a row's reference max moved: once the previous block's P V is done, rescale
          // its O and row sum (before a tile's first block there is nothing to rescale)
          w = pf_wait(sm, &sm.p_free[(gb - 1) & 1], uint32_t((gb - 1) >> 1) & 1, a.status);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + 32 * half, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(lane_base + kColO + 32 * half, o);
          }
          tmem_st1(lane_base + kColO + kHeadDim,
                   __float_as_uint(__uint_as_float(tmem_ld1(lane_base + kColO + kHeadDim)) * alpha));
        }
        tc_fence_before();  // the reads of O above precede this tile's first P V (ordered by p_full)
        mbar_arrive(&sm.p_full[b]);
      }
      if (!ok) break;
      fin = true;
      fin_q0 = t.q0;
      fin_t0 = t.t0;
      fin_n = t.n;
      fin_g = t.g;
    }
    if (ok && fin) finish();
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
                                           int num_q_rows, const int32_t *query_start, const int32_t *block_tables,
                                           int64_t block_table_stride, const int32_t *context_lens, int num_seqs,
                                           int max_query, int max_context, float scale, int32_t *device_status,
                                           void *stream) {
  return pkv_paged_prefill_attention_ex(pool, out, q, num_q_heads, num_q_rows, query_start, block_tables,
                                        block_table_stride, context_lens, num_seqs, max_query, max_context, scale,
                                        device_status, 0u, stream);
}

extern "C" int pkv_paged_prefill_attention_ex(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                              int num_q_rows, const int32_t *query_start, const int32_t *block_tables,
                                              int64_t block_table_stride, const int32_t *context_lens, int num_seqs,
                                              int max_query, int max_context, float scale, int32_t *device_status,
                                              unsigned flags, void *stream) {
  if (flags & ~unsigned(PKV_OVERLAP_PREVIOUS)) return PKV_ERR_SHAPE;
  int rc = pkv::check_pool(pool);
  if (rc != PKV_OK) return rc;
  if (num_q_heads != pkv::kQHeads) return PKV_ERR_UNSUPPORTED;
  if (num_seqs < 0 || max_query < 0 || max_context < 0 || block_table_stride < 0 || num_q_rows < 0)
    return PKV_ERR_SHAPE;
  if (num_seqs == 0 || max_query == 0 || num_q_rows == 0) return PKV_OK;
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
  rc = pkv::query_tensor_map(q, num_q_rows, pkv::kQHeads, pkv::kHeadDim, pkv::kGroup, pkv::kPfTok, &a.tmap_q);
  if (rc != PKV_OK) return rc;
  a.num_pages = pool->num_pages;
  a.num_q_rows = num_q_rows;
  a.out = out;
  a.query_start = query_start;
  a.block_tables = block_tables;
  a.bt_stride = block_table_stride;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.max_context = max_context;
  a.tiles_per_seq = int(tiles);
  a.scale_log2 = fabsf(scale) * pkv::kLog2e;
  a.move_thresh = a.scale_log2 > 0.f ? pkv::kRescaleLog2 / a.scale_log2 : INFINITY;
  a.neg = scale < 0.f ? 1 : 0;
  a.status = device_status;
  a.num_tiles = int((long long)num_seqs * tiles * pkv::kKvHeads);
  const int sms = pkv::device_sm_count();
  const int resident = (sms > 0 ? sms : 148) * pkv::kPfCtasPerSm;
  const int by_table = (a.num_tiles + pkv::kPfMaxTiles - 1) / pkv::kPfMaxTiles;  // tiles per CTA <= kPfMaxTiles
  const int g = resident > by_table ? resident : by_table;
  const unsigned grid = unsigned(a.num_tiles < g ? a.num_tiles : g);
  if (flags & PKV_OVERLAP_PREVIOUS) {
    // programmatic stream serialization: the set-up (tile table, block-table entries, the first
    // tile's Q) overlaps the end of the kernel before this one
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(pkv::kPfThreads);
    cfg.dynamicSmemBytes = pkv::kPfSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, pkv::paged_prefill_kernel, a) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_LAUNCH;
    }
    return PKV_OK;
  }
  pkv::paged_prefill_kernel<<<grid, pkv::kPfThreads, pkv::kPfSmemBytes, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}
