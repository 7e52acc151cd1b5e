/*
 * pkv.h - C ABI of the paged KV-cache decode library for GB300 (sm_103a).
 *
 * Single-token decode attention over a paged BF16 KV cache.  Each sequence's K
 * and V live in physical pages of a shared pool, reached through a block table
 * per (sequence, layer); decode appends one token's K/V into its slot, then
 * every query head attends over the sequence's cached tokens with an FP32
 * online softmax, without gathering a contiguous prefix or storing scores.
 *
 * Sources (web pages on the method):
 *  - "6 Hours of YouTube ... LLM Inference" (samir-vllm README), section "What
 *    works so far": one shared BF16 page pool, a block table per sequence and
 *    layer, 16 tokens of K and V per page, decode appends one token at its
 *    absolute position, paged decode attention with an FP32 online softmax
 *    that streams each sequence's pages; section "Current scope": 2048-token
 *    context, 128 MiB default pool.
 *  - "tiny-vllm part 3: the prefill path", section "Distributing K/V into paged
 *    blocks" (block = token / 16, block table lookup, -1 = unassigned, K at the
 *    block start and V at a fixed offset); section "Per-head attention scores
 *    and GQA" (32 query heads share 8 K/V heads, query head h reads K/V head
 *    h / 4, scale 1/sqrt(64)); section "causalMask and online softmax" (the
 *    merge rule of two partial softmax states: m = max(ma, mb),
 *    d = da*exp(ma - m) + db*exp(mb - m)).
 *
 * Conventions for every entry point:
 *  - Buffers are owned by the caller.  The library never allocates, frees or
 *    synchronises; device work is enqueued on the caller's stream.
 *  - "device" pointers must be CUDA device (or managed) memory of the current
 *    device; "host" pointers are ordinary host memory.  An argument marked
 *    "device or mapped host" may also be pinned host memory mapped into the device
 *    address space (cudaHostAlloc, cudaHostRegister): the kernel then reads or writes
 *    it over the host link (NVLink-C2C on Grace-Blackwell), with no separate copy.
 *  - bf16 values are passed as raw 16-bit patterns (bfloat16, i.e. the upper
 *    half of an IEEE binary32).
 *  - Host-checkable faults return a negative PKV_ERR_* code and enqueue
 *    nothing.  Faults only the device can see (bad slots, context lengths or
 *    block-table entries) are OR-ed as PKV_DEV_* bits into *device_status when
 *    that pointer is non-null; the host never reads device memory.
 *  - `stream` is a cudaStream_t (0 = legacy default stream).
 *
 * Supported geometry in this build: page_tokens 16, head_dim 64, 8 K/V heads,
 * 32 query heads (group 4).  Other values are rejected with
 * PKV_ERR_UNSUPPORTED.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (host side) ------------------------------------------ */
#define PKV_OK 0
#define PKV_ERR_NULL (-1)          /* a required pointer is null */
#define PKV_ERR_SHAPE (-2)         /* a size or count is out of range */
#define PKV_ERR_UNSUPPORTED (-3)   /* geometry this build does not compile */
#define PKV_ERR_ALIGN (-4)         /* pointer or stride not 16-byte aligned */
#define PKV_ERR_SCALE (-5)         /* scale is not finite */
#define PKV_ERR_WORKSPACE (-6)     /* workspace smaller than pkv_decode_workspace_bytes() */
#define PKV_ERR_LAUNCH (-7)        /* the CUDA runtime refused a kernel launch */
#define PKV_ERR_CUDA (-8)          /* another CUDA runtime call failed */
#define PKV_ERR_EXCEEDS_POOL (-9)  /* scheduler: a request's page budget exceeds the whole pool */
#define PKV_ERR_NO_PAGE (-10)      /* allocator: no free page */
#define PKV_ERR_STATE (-11)        /* scheduler/allocator used out of order */
#define PKV_ERR_NOALLOC_LIMIT (-12) /* num_seqs above the fixed scratch of the allocation-free entry point */
#define PKV_ERR_NO_CREDIT (-13)    /* allocator: a request's credits do not fit beside the admitted ones now */

/* ---- device status bits (OR-ed into *device_status) --------------------- */
#define PKV_DEV_BAD_SLOT 1u        /* kv_append: slot >= num_pages * page_tokens; decode_step: slot is not
                                      position ctx - 1 of the sequence; the token is not written */
#define PKV_DEV_BAD_CONTEXT 2u     /* context_lens[s] < 0 or > max_context; row s of out is zeros */
#define PKV_DEV_BAD_PAGE 4u        /* block-table entry outside [0, num_pages) inside the context;
                                      that page's tokens are left out of the softmax */
#define PKV_DEV_TIMEOUT 8u         /* an internal pipeline wait gave up (about 2 s); the CTA stopped */

/*
 * Pool descriptor (plain data; copying it is free).
 *
 * K element (page p, kv_head g, row r, dim d) is the bf16 at
 *     k_base + p * page_stride_bytes + ((g * page_tokens + r) * head_dim + d) * 2
 * and V likewise from v_base.  In the default interleaved buffer
 * (pkv_kv_pool_bytes) a page is [K | V][kv_head][row][dim]: K in the first
 * half and V at +num_kv_heads*page_tokens*head_dim*2 bytes (16 KiB for the
 * supported geometry), page stride 32 KiB.  Slot s names page
 * s / page_tokens, row s % page_tokens.
 */
typedef struct pkv_pool {
    void *k_base;               /* device */
    void *v_base;               /* device */
    int64_t page_stride_bytes;  /* bytes between consecutive pages (same for K and V) */
    int32_t num_pages;
    int32_t page_tokens;
    int32_t num_kv_heads;
    int32_t head_dim;
} pkv_pool;

/* Bytes of one interleaved pool buffer of num_pages pages ([page][K|V][kv_head][row][dim] bf16). */
size_t pkv_kv_pool_bytes(int num_pages, int page_tokens, int num_kv_heads, int head_dim);

/*
 * pkv_kv_pool_create - describe caller-owned pool memory (no allocation, no device work).
 *   k_pool, v_pool     device; for the interleaved buffer pass v_pool = k_pool + half a page
 *                      and page_stride_bytes = 0 (meaning: 2 * half page).
 *   page_stride_bytes  bytes between pages, >= half a page, multiple of 16 (0 = interleaved default)
 *   out                host; receives the descriptor.
 * Returns PKV_OK, PKV_ERR_NULL, PKV_ERR_SHAPE, PKV_ERR_ALIGN (pointers or stride not
 * 16-byte aligned) or PKV_ERR_UNSUPPORTED.
 * Cited: samir-vllm README "What works so far" (shared BF16 page pool, 16-token pages).
 */
int pkv_kv_pool_create(void *k_pool, void *v_pool, int64_t page_stride_bytes, int num_pages,
                       int page_tokens, int num_kv_heads, int head_dim, pkv_pool *out);

/*
 * pkv_kv_append - scatter the K/V of num_tokens new tokens into their slots (bit copy).
 *   pool          host; descriptor from pkv_kv_pool_create.
 *   k_new, v_new  device or mapped host; bf16 [num_tokens][num_kv_heads][head_dim], 16-byte aligned.
 *   slot_mapping  device or mapped host; int32 [num_tokens]; slot = page * page_tokens + row; a negative slot
 *                 is padding and is skipped; a slot >= num_pages * page_tokens is skipped and
 *                 sets PKV_DEV_BAD_SLOT.
 *   device_status device int32, nullable.
 * Two tokens naming the same slot race (either may win).  num_tokens = 0 enqueues nothing.
 * A kernel launched right after it with PKV_OVERLAP_PREVIOUS (pkv_decode_step_ex,
 * pkv_paged_prefill_attention_ex) may begin its set-up while it runs.
 * Cited: samir-vllm README "What works so far" (decode appends one new token at its absolute
 * position); tiny-vllm part 3, "Distributing K/V into paged blocks" (page/row of a token,
 * K and V copied into the block).
 */
int pkv_kv_append(const pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                  int num_tokens, int32_t *device_status, void *stream);

/*
 * Workspace bytes pkv_paged_decode_attention needs for num_seqs sequences: one slot
 * per (CTA, sequence) pair of the split, holding a partial softmax state and a
 * ticket counter.  Zero-fill the workspace once before its first use (e.g.
 * cudaMemsetAsync); every completed call leaves the counters at zero again, so the
 * same workspace serves later calls of any batch size up to the one it was sized
 * for.  After a call that reported PKV_DEV_TIMEOUT, zero it again.  0 on bad arguments.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim);

/*
 * pkv_paged_decode_attention - one decode step of attention for num_seqs sequences.
 *
 *   out[s][h][:] = sum_{t < ctx_s} w_t V_t[h / group][:],
 *   w = softmax_t( scale * q[s][h] . K_t[h / group] ),   group = num_q_heads / num_kv_heads,
 *   K_t, V_t read from page block_tables[s * block_table_stride + t / page_tokens],
 *   row t % page_tokens.
 *
 *   pool               host; descriptor.
 *   out                device or mapped host; float32 [num_seqs][num_q_heads][head_dim], 8-byte aligned.
 *   q                  device or mapped host; bf16 [num_seqs][num_q_heads][head_dim], 16-byte aligned.
 *   block_tables       device; int32; row s starts at s * block_table_stride and holds at least
 *                      ceil(max_context / page_tokens) entries (a multi-layer table
 *                      [seq][layer][blocks] is passed as base + layer * blocks with
 *                      stride layers * blocks).
 *   context_lens       device; int32 [num_seqs]; tokens to attend (the new token included).
 *                      0 gives a zero output row.
 *   max_context        host bound on every context_lens[s] (chooses the work split; a larger
 *                      length sets PKV_DEV_BAD_CONTEXT and zeroes that row).
 *   scale              softmax scale (1/sqrt(head_dim) for the pages' model).
 *   workspace          device, >= pkv_decode_workspace_bytes(num_seqs, ...), 16-byte aligned,
 *                      zero-filled before its first use (see pkv_decode_workspace_bytes).
 *   device_status      device int32, nullable.
 * Enqueues one kernel: the pages of all sequences are split evenly over its CTAs,
 * and the last CTA to finish a sequence that was cut merges its partial states.
 * Calls sharing a workspace must not overlap on the GPU.
 * Returns PKV_OK or a negative PKV_ERR_* code (then nothing was enqueued).
 * Cited: samir-vllm README "What works so far" (direct paged decode attention, FP32
 * online softmax, no contiguous gather, no stored scores; separate page maps and
 * lengths per sequence); tiny-vllm part 3, "Per-head attention scores and GQA" and
 * "causalMask and online softmax" (GQA mapping, scale, softmax merge rule).
 */
int pkv_paged_decode_attention(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                               const int32_t *block_tables, int64_t block_table_stride,
                               const int32_t *context_lens, int num_seqs, int max_context, float scale,
                               void *workspace, size_t workspace_bytes, int32_t *device_status,
                               void *stream);

/*
 * pkv_decode_step - one decode step for num_seqs sequences in one launch: append each
 * sequence's new token, then attend (pkv_kv_append followed by pkv_paged_decode_attention,
 * fused).  k_new, v_new (device or mapped host, bf16 [num_seqs][num_kv_heads][head_dim], 16-byte aligned)
 * hold sequence s's new token, which is position context_lens[s] - 1 (the last token
 * attended); slot_mapping[s] (device or mapped host, int32) is that position's slot in the
 * pool: block_tables[s][(ctx - 1) / page_tokens] * page_tokens + (ctx - 1) % page_tokens.
 * A negative slot means sequence s has no new token this step (its cached tokens are
 * attended as they are).  The CTA that holds a sequence's last page takes the new token's
 * rows straight from k_new/v_new and writes them to the pool.  Any other non-negative slot
 * (not that position, or past the pool) sets PKV_DEV_BAD_SLOT: the token is neither stored
 * nor attended, and the sequence is attended over its cached rows as they are.  A sequence
 * with context 0 appends nothing.  Other arguments, errors and results are those of
 * pkv_paged_decode_attention.
 * Cited: samir-vllm README "What works so far" (decode appends one new token at its
 * absolute position, then paged attention over the sequence's pages).
 */
int pkv_decode_step(const pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                    float *out, const void *q, int num_q_heads, const int32_t *block_tables,
                    int64_t block_table_stride, const int32_t *context_lens, int num_seqs, int max_context,
                    float scale, void *workspace, size_t workspace_bytes, int32_t *device_status, void *stream);

/*
 * pkv_decode_step_ex - pkv_decode_step with launch flags.
 *   flags   0, or PKV_OVERLAP_PREVIOUS: the kernel is launched with programmatic stream
 *           serialization, so it may start while the kernel before it on the stream is still
 *           running.  It then reads context_lens, block_tables and the pool pages it attends
 *           (and issues their copies) at once, and reads q, k_new, v_new, slot_mapping and
 *           writes out, the pool, the workspace and device_status only after that kernel has
 *           completed.  Use it only when the kernel before it on the stream writes none of
 *           context_lens, block_tables or those pool pages (for example the previous layer's
 *           step of a multi-layer decode, whose pages differ); inside a CUDA graph capture the
 *           relation becomes a programmatic edge between the two kernel nodes.
 *           Other bits return PKV_ERR_SHAPE.
 * Everything else as pkv_decode_step.
 */
#define PKV_OVERLAP_PREVIOUS 1u
int pkv_decode_step_ex(const pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *slot_mapping,
                       float *out, const void *q, int num_q_heads, const int32_t *block_tables,
                       int64_t block_table_stride, const int32_t *context_lens, int num_seqs, int max_context,
                       float scale, void *workspace, size_t workspace_bytes, int32_t *device_status,
                       unsigned flags, void *stream);

/*
 * pkv_paged_prefill_attention - causal attention of a chunk of query tokens per sequence
 * over its paged K/V (prefill, chunked prefill; one query per sequence is decode).
 *
 *   out[i][h][:] = sum_{t <= p_i} w_t V_t[h / group][:],
 *   w = softmax_{t <= p_i}( scale * q[i][h] . K_t[h / group] ),
 *   p_i = context_lens[s] - n_s + (i - query_start[s])   for query row i of sequence s,
 *   n_s = query_start[s+1] - query_start[s]: the queries are the last n_s cached tokens
 *   (append them with pkv_kv_append first).
 *
 *   out            device; float32 [total][num_q_heads][head_dim], total = query_start[num_seqs],
 *                  16-byte aligned.
 *   q              device; bf16 [total][num_q_heads][head_dim], 16-byte aligned.
 *   num_q_rows     rows of q and out (>= total); the kernel reads and writes no row at or
 *                  past it (a sequence whose query rows would reach past it counts as invalid).
 *   query_start    device; int32 [num_seqs + 1], non-decreasing, query_start[0] = 0.
 *   block_tables, block_table_stride, context_lens, max_context: as for decode.
 *   max_query      host bound on every n_s (sizes the grid; longer runs are not computed).
 * A sequence with n_s > context_lens[s] or an invalid context gets zero rows and
 * PKV_DEV_BAD_CONTEXT; an invalid page id inside a query's span sets PKV_DEV_BAD_PAGE
 * (that page is left out).  No workspace.  One kernel launch.
 * Cited: tiny-vllm part 3, "Per-head attention scores and GQA" and "causalMask and online
 * softmax" (per-head scores, causal mask keeping the diagonal, softmax, scores x V), with
 * K/V read through the block table as in "Distributing K/V into paged blocks".
 */
int pkv_paged_prefill_attention(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                int num_q_rows, const int32_t *query_start, const int32_t *block_tables,
                                int64_t block_table_stride, const int32_t *context_lens, int num_seqs,
                                int max_query, int max_context, float scale, int32_t *device_status,
                                void *stream);

/*
 * pkv_paged_prefill_attention_ex - pkv_paged_prefill_attention with launch flags.
 *   flags   0, or PKV_OVERLAP_PREVIOUS: launched with programmatic stream serialization, the
 *           kernel may start while the kernel before it on the stream is still running; it
 *           reads query_start, context_lens, block_tables and q at once, and the pool pages
 *           (and writes out and device_status) only after that kernel has completed.  Use it
 *           only when the kernel before it writes none of q, query_start, context_lens or
 *           block_tables - for example pkv_kv_append of the prompt's K/V, which writes only the
 *           pool.  Other bits return PKV_ERR_SHAPE.
 * Everything else as pkv_paged_prefill_attention.
 */
int pkv_paged_prefill_attention_ex(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                   int num_q_rows, const int32_t *query_start, const int32_t *block_tables,
                                   int64_t block_table_stride, const int32_t *context_lens, int num_seqs,
                                   int max_query, int max_context, float scale, int32_t *device_status,
                                   unsigned flags, void *stream);

/*
 * Same as pkv_paged_decode_attention with the number of CTAs of the split-context pass
 * fixed by the caller (1 .. pkv_decode_max_ctas(); 0 = automatic).  The result must not
 * depend on it beyond FP32 rounding; tests sweep it.
 */
int pkv_paged_decode_attention_ctas(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                    const int32_t *block_tables, int64_t block_table_stride,
                                    const int32_t *context_lens, int num_seqs, int max_context,
                                    float scale, void *workspace, size_t workspace_bytes,
                                    int32_t *device_status, int num_ctas, void *stream);

/* Largest CTA count the split-context pass may use (sizes the workspace). */
int pkv_decode_max_ctas(void);

/*
 * Launch plan of pkv_paged_decode_attention on the current device: CTAs of the
 * split-context pass and kernel launches per call.  Returns PKV_OK or an error.
 */
int pkv_decode_plan(int num_seqs, int max_context, int *num_ctas, int *launches);

/*
 * pkv_paged_decode_attention_noalloc - pkv_paged_decode_attention for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry point.
 *
 * Some callers have no way to obtain a workspace: a plugin loaded into a host runtime
 * that owns every device buffer and hands out only inputs and outputs, or a C/FFI
 * caller with no device allocator of its own that must not call cudaMalloc (which can
 * synchronise the device and fail under memory pressure mid-run).  This entry point
 * takes the same inputs and output but no workspace: the split-context partial states
 * live in one fixed array of device memory inside this library, sized for
 * PKV_NOALLOC_MAX_SEQS sequences (about 12.5 MiB), which every GPU that loads the
 * library holds until the process exits.  It calls no allocator.
 *
 *  - num_seqs > PKV_NOALLOC_MAX_SEQS returns PKV_ERR_NOALLOC_LIMIT and enqueues nothing.
 *  - The first call on a device (with that device current) looks up the array's device
 *    address once; make that first call before any stream capture on that device.
 *  - The first call on a device also clears the array once, enqueued on that call's
 *    stream ahead of its kernel (the merge counters must start at zero; every completed
 *    call leaves them at zero again).  A later call on another stream must be ordered
 *    after that first call, like any two calls (see below).
 *  - The looked-up address is kept for the life of the process: after cudaDeviceReset
 *    (or any re-creation of the device's primary context) this entry point is not
 *    supported on that device.
 *  - All calls on a device share the one array and it keeps the last call's contents;
 *    calls that overlap on the GPU - on different streams, or from different host
 *    threads without ordering - race on it: serialise them.
 * Other arguments, errors and results are those of pkv_paged_decode_attention.
 */
#define PKV_NOALLOC_MAX_SEQS 512
int pkv_paged_decode_attention_noalloc(const pkv_pool *pool, float *out, const void *q, int num_q_heads,
                                       const int32_t *block_tables, int64_t block_table_stride,
                                       const int32_t *context_lens, int num_seqs, int max_context,
                                       float scale, int32_t *device_status, void *stream);

/* ---- host page allocator (no GPU) ------------------------------------------------------
 *
 * The admission credits, lazy page assignment and page release that the scheduler below
 * is built from, for a caller that runs its own scheduler.  The allocator owns the pool's
 * free list and a host block table [max_seqs][num_layers][max_blocks] (max_blocks =
 * ceil(max_context / page_tokens), -1 = unassigned) that a caller copies to the device for
 * the attention calls.  Host memory only; not thread-safe (one caller thread at a time).
 *
 * Cited: samir-vllm README, "Current scope" (admission credits = pages for prompt + new - 1
 * tokens, rounded up to 16-token pages, in every layer; the new-token budget is clamped to
 * the context limit; credits are separate from physical pages, which are assigned lazily;
 * a request larger than the whole pool is rejected; completion returns pages and credits);
 * tiny-vllm part 3, "Distributing K/V into paged blocks" (a page is popped from the back of
 * the free list when a block is first written; -1 marks an unassigned block).
 */
typedef struct pkv_alloc pkv_alloc;

/* free_order: host, nullable - the initial free list (num_pages distinct ids, popped from the
 * back; pass a seeded permutation for a shuffled pool); NULL means 0 .. num_pages-1.
 * Returns PKV_OK, PKV_ERR_NULL (out) or PKV_ERR_SHAPE. */
int pkv_alloc_create(int num_pages, int num_layers, int page_tokens, int max_context, int max_seqs,
                     const int32_t *free_order, pkv_alloc **out);
void pkv_alloc_destroy(pkv_alloc *alloc);
/* Admit a request into sequence seq (0 .. max_seqs-1, not admitted now): reserve its credits,
 * ceil((prompt + new - 1) / page_tokens) * num_layers with new = min(max_new_tokens,
 * max_context + 1 - prompt_tokens).  *credits (nullable) receives that count whatever the
 * outcome.  Returns PKV_OK; PKV_ERR_EXCEEDS_POOL if the credits exceed the whole pool (the
 * request can never be admitted); PKV_ERR_NO_CREDIT if they do not fit beside the credits
 * already held (nothing reserved: retry after a sequence is freed); PKV_ERR_STATE if seq is
 * admitted already; PKV_ERR_SHAPE for prompt < 1, prompt > max_context, max_new_tokens < 1 or
 * seq out of range. */
int pkv_alloc_admit(pkv_alloc *alloc, int seq, int prompt_tokens, int max_new_tokens, int32_t *credits);
/* Physical page of logical block `block` of (seq, layer): the table entry when assigned,
 * else the page popped from the back of the free list (the first write of that block).
 * The slot of token t is then page * page_tokens + t % page_tokens with block = t / page_tokens.
 * Returns PKV_OK, PKV_ERR_NO_PAGE (free list empty; cannot happen while every sequence
 * stays within its credits), PKV_ERR_STATE (seq not admitted) or PKV_ERR_SHAPE. */
int pkv_alloc_page(pkv_alloc *alloc, int seq, int layer, int block, int32_t *page);
/* Return every page of seq to the free list (layers in order, blocks ascending, each pushed on
 * the back) and release its credits; its table rows become -1.  PKV_OK, PKV_ERR_STATE (seq not
 * admitted) or PKV_ERR_SHAPE. */
int pkv_alloc_free_seq(pkv_alloc *alloc, int seq);
/* The allocator's block table [max_seqs][num_layers][max_blocks] (valid until destroy). */
const int32_t *pkv_alloc_block_tables(const pkv_alloc *alloc);
/* Pages on the free list and credits held now (either pointer nullable). */
int pkv_alloc_state(const pkv_alloc *alloc, int32_t *free_pages, int32_t *credits_in_use);

/* ---- continuous-batching scheduler (no GPU) ----------------------------------------------
 *
 * Cited: samir-vllm README, "What works so far" (requests share the pool; static and
 * continuous batching admit queued prompts by page budget and return pages and budgets on
 * completion) and "Current scope" (admission credits = pages for prompt + new - 1 tokens,
 * rounded up to 16-token pages, in every layer; the new-token budget is clamped to the
 * context limit; credits are separate from pages, which are assigned lazily; FIFO waits;
 * a request larger than the whole pool is rejected; --stats counters); tiny-vllm part 3,
 * "Distributing K/V into paged blocks" (pages popped from the back of a free list when a
 * block is first written; -1 marks an unassigned block).
 *
 * A step: (1) retire the requests that finished last step (their pages go back on the free
 * list, block order per layer, and their credits are released); (2) admit queued requests
 * in FIFO order into the lowest free slots while their credits fit (head-of-line blocking;
 * a blocked head with a free slot counts one admission wait per step) and plan the append
 * of their prompt tokens; (3) every active request with tokens left to decode appends one
 * token (a just-admitted one included) and attends.  A request with prompt P and budget N
 * decodes N - 1 tokens, so its context ends at P + N - 1.  Pages are taken from the back of
 * the free list when a token is the first of its block, in every layer.
 */
typedef struct pkv_sched pkv_sched;

typedef struct pkv_step_plan {
    int32_t num_finished;              /* requests retired at the start of this step */
    const int64_t *finished_request;   /* [num_finished] */
    int32_t num_admitted;
    const int64_t *admitted_request;   /* [num_admitted] */
    const int32_t *admitted_slot;      /* [num_admitted] */
    int32_t num_appends;               /* tokens to append: admitted prompts, then one per decoding slot */
    const int64_t *append_request;     /* [num_appends] request of each token */
    const int32_t *append_position;    /* [num_appends] absolute position of the token in its request */
    const int32_t *append_slot_mapping;/* [num_layers][num_appends]: page * page_tokens + row */
    int32_t num_decode;                /* slots that decode this step */
    const int32_t *decode_slot;        /* [num_decode] ascending */
    const int32_t *context_lens;       /* [num_slots]: context after this step's append, 0 if idle */
    const int32_t *block_tables;       /* [num_slots][num_layers][max_blocks], -1 = unassigned */
    int32_t max_blocks;                /* ceil(max_context / page_tokens) */
} pkv_step_plan;

typedef struct pkv_sched_stats {
    int32_t pool_pages;
    int32_t peak_active;       /* most requests holding a slot at once */
    int32_t largest_batch;     /* most sequences decoding in one step */
    int32_t peak_pages;        /* most pages assigned at once */
    int32_t admission_waits;   /* steps in which the queue head waited for credits with a slot free */
    int32_t free_pages;        /* pages on the free list now */
    int32_t credits_in_use;
    int32_t active;
    int32_t queued;
    int64_t steps;
} pkv_sched_stats;

/* free_order: host, nullable - initial free list (num_pages distinct ids, popped from the
 * back); NULL means 0 .. num_pages-1.  Returns PKV_OK, PKV_ERR_NULL or PKV_ERR_SHAPE. */
int pkv_sched_create(int num_pages, int num_layers, int page_tokens, int max_context, int num_slots,
                     const int32_t *free_order, pkv_sched **out);
void pkv_sched_destroy(pkv_sched *sched);
/* Queue a request.  max_new_tokens is clamped so prompt + new - 1 <= max_context.
 * PKV_ERR_EXCEEDS_POOL if its credits exceed the whole pool (it is not queued),
 * PKV_ERR_SHAPE for prompt < 1, prompt > max_context or max_new_tokens < 1. */
int pkv_sched_submit(pkv_sched *sched, int64_t request_id, int prompt_tokens, int max_new_tokens);
/* Run one step and describe it in *plan (pointers stay valid until the next call).
 * PKV_ERR_NO_PAGE if the free list ran dry (cannot happen while credits are honoured). */
int pkv_sched_step(pkv_sched *sched, pkv_step_plan *plan);
int pkv_sched_stats_get(const pkv_sched *sched, pkv_sched_stats *out);

/* Short English text for a PKV_ERR_* code or PKV_OK. */
const char *pkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
