/*
 * CPU oracle for single-token decode attention over a paged BF16 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA path: no headers, no helpers, no constants.
 *
 * Plain, slow and written for reading.  Every floating-point step is FP64.
 *
 * Sources (web pages on paged KV caches for a Llama 3.2 1B engine):
 *  - "6 Hours of YouTube ... LLM Inference" (samir-vllm README), "What works so
 *    far": one shared BF16 pool of physical pages of 16 tokens holding K and V,
 *    a block table per (sequence, layer); decode appends one token at its
 *    absolute position; decode attention is an exact softmax over the cached
 *    tokens, computed without gathering a contiguous prefix.
 *  - "tiny-vllm part 3: the prefill path", section "Distributing K/V into paged
 *    blocks": logical block = token / 16, physical block from the block table,
 *    -1 = unassigned, K at the start of the block and V at a fixed offset.
 *  - same page, section "Per-head attention scores and GQA": 32 query heads,
 *    8 K/V heads, query head h reads K/V head h / 4; scale 1/sqrt(64).
 *  - same page, section "causalMask and online softmax": softmax(x) =
 *    exp(x - max) / sum exp(x - max).  The oracle takes the two-pass form of
 *    that definition (max first, then weights), not the online merge.
 *
 * Pool layout (the library's layout; written out here independently): K
 * element (page, kv_head g, row r, dim d) sits at
 *     k_pool[page * page_stride + (g * page_tokens + r) * head_dim + d]
 * and V likewise in v_pool.  Slot s names page s / page_tokens, row
 * s % page_tokens.
 *
 * Every entry point returns 0, or an OR of ORACLE_ERR_* bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ERR_SLOT 1      /* slot >= num_pages * page_tokens */
#define ORACLE_ERR_CONTEXT 2   /* context length < 0 or > max_context */
#define ORACLE_ERR_PAGE 4      /* block-table entry outside [0, num_pages) inside the context */
#define ORACLE_ERR_ARGS 8      /* shapes that make no sense */

/* bfloat16 holds the upper 16 bits of an IEEE binary32 value. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int64_t element_index(int64_t page_stride, int64_t page, int kv_head, int row,
                             int page_tokens, int head_dim)
{
    return page * page_stride + ((int64_t)kv_head * page_tokens + row) * head_dim;
}

/*
 * Append: for token i with slot_mapping[i] >= 0, copy its K and V rows
 * (num_kv_heads x head_dim values, token-major input [num_tokens][num_kv_heads][head_dim])
 * into the page and row the slot names.  Negative slots are padding and are
 * skipped; out-of-range slots are skipped and reported.
 */
int oracle_kv_append(uint16_t *k_pool, uint16_t *v_pool, int64_t page_stride, int num_pages,
                     int page_tokens, int num_kv_heads, int head_dim,
                     const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *slot_mapping, int num_tokens)
{
    int err = 0;
    if (num_pages < 0 || page_tokens <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_tokens < 0)
        return ORACLE_ERR_ARGS;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_pages * page_tokens) {
            err |= ORACLE_ERR_SLOT;
            continue;
        }
        int64_t page = slot / page_tokens;
        int row = (int)(slot % page_tokens);
        for (int g = 0; g < num_kv_heads; ++g) {
            int64_t dst = element_index(page_stride, page, g, row, page_tokens, head_dim);
            int64_t src = ((int64_t)i * num_kv_heads + g) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                k_pool[dst + d] = k_new[src + d];
                v_pool[dst + d] = v_new[src + d];
            }
        }
    }
    return err;
}

/* Physical page and row of logical token t of a sequence, or -1 when the table entry is invalid. */
static int64_t token_page(const int32_t *table_row, int t, int page_tokens, int num_pages)
{
    int32_t p = table_row[t / page_tokens];
    if (p < 0 || p >= num_pages)
        return -1;
    return p;
}

/*
 * Scores x_t = scale * sum_d q[d] * K_t[d] of one query head against the
 * logical tokens 0..ctx-1 of one sequence, read through its block table.
 * Returns nonzero if a table entry inside the context is invalid.
 */
static int head_scores(const uint16_t *k_pool, int64_t page_stride, int num_pages, int page_tokens,
                       int head_dim, const uint16_t *q_head, int kv_head, const int32_t *table_row,
                       int ctx, double scale, double *x)
{
    for (int t = 0; t < ctx; ++t) {
        int64_t page = token_page(table_row, t, page_tokens, num_pages);
        if (page < 0)
            return 1;
        int64_t k0 = element_index(page_stride, page, kv_head, t % page_tokens, page_tokens, head_dim);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_value(q_head[d]) * bf16_value(k_pool[k0 + d]);
        x[t] = scale * dot;
    }
    return 0;
}

/* Two-pass softmax weights w_t = exp(x_t - max x) / sum_u exp(x_u - max x). */
static void softmax_weights(const double *x, int n, double *w)
{
    double m = x[0];
    for (int t = 1; t < n; ++t)
        if (x[t] > m)
            m = x[t];
    double z = 0.0;
    for (int t = 0; t < n; ++t) {
        w[t] = exp(x[t] - m);
        z += w[t];
    }
    for (int t = 0; t < n; ++t)
        w[t] /= z;
}

/*
 * Decode attention:
 *   out[s][h][:] = sum_t w_t * V_t[h / group][:],  w = softmax(scale * q[s][h] . K_t[h / group])
 * over t < context_lens[s], group = num_q_heads / num_kv_heads.  q is
 * [num_seqs][num_q_heads][head_dim] bf16; sequence s reads its block-table row
 * at block_tables + s * bt_stride.  out is FP64 [num_seqs][num_q_heads][head_dim].
 * A sequence with context 0, an invalid context length or an invalid page gets
 * an all-zero output row (the last two are also reported).
 */
int oracle_paged_decode_attention(const uint16_t *k_pool, const uint16_t *v_pool, int64_t page_stride,
                                  int num_pages, int page_tokens, int num_kv_heads, int head_dim,
                                  const uint16_t *q, int num_q_heads,
                                  const int32_t *block_tables, int64_t bt_stride,
                                  const int32_t *context_lens, int num_seqs, int max_context,
                                  double scale, double *out)
{
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        page_tokens <= 0 || num_seqs < 0 || max_context < 0)
        return ORACLE_ERR_ARGS;
    int group = num_q_heads / num_kv_heads;
    int err = 0;
    double *x = (double *)malloc(sizeof(double) * (size_t)(max_context > 0 ? max_context : 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)(max_context > 0 ? max_context : 1));
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        double *o_seq = out + (int64_t)s * num_q_heads * head_dim;
        for (int i = 0; i < num_q_heads * head_dim; ++i)
            o_seq[i] = 0.0;
        if (ctx < 0 || ctx > max_context) {
            err |= ORACLE_ERR_CONTEXT;
            continue;
        }
        if (ctx == 0)
            continue;
        const int32_t *row = block_tables + (int64_t)s * bt_stride;
        for (int h = 0; h < num_q_heads; ++h) {
            int g = h / group;
            const uint16_t *qh = q + ((int64_t)s * num_q_heads + h) * head_dim;
            if (head_scores(k_pool, page_stride, num_pages, page_tokens, head_dim, qh, g, row, ctx,
                            scale, x)) {
                err |= ORACLE_ERR_PAGE;
                for (int i = 0; i < num_q_heads * head_dim; ++i)
                    o_seq[i] = 0.0;
                break;
            }
            softmax_weights(x, ctx, w);
            double *o = o_seq + (int64_t)h * head_dim;
            for (int t = 0; t < ctx; ++t) {
                int64_t page = token_page(row, t, page_tokens, num_pages);
                int64_t v0 = element_index(page_stride, page, g, t % page_tokens, page_tokens, head_dim);
                for (int d = 0; d < head_dim; ++d)
                    o[d] += w[t] * bf16_value(v_pool[v0 + d]);
            }
        }
    }
    free(x);
    free(w);
    return err;
}

/*
 * The softmax weights of one (sequence, query head), for invariant checks
 * (they must sum to one).  w has room for context_lens[seq] values.
 */
int oracle_attention_weights(const uint16_t *k_pool, int64_t page_stride, int num_pages,
                             int page_tokens, int num_kv_heads, int head_dim,
                             const uint16_t *q, int num_q_heads,
                             const int32_t *block_tables, int64_t bt_stride,
                             const int32_t *context_lens, int seq, int head, double scale, double *w)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return ORACLE_ERR_ARGS;
    int ctx = context_lens[seq];
    if (ctx <= 0)
        return ORACLE_ERR_CONTEXT;
    int group = num_q_heads / num_kv_heads;
    double *x = (double *)malloc(sizeof(double) * (size_t)ctx);
    const uint16_t *qh = q + ((int64_t)seq * num_q_heads + head) * head_dim;
    int bad = head_scores(k_pool, page_stride, num_pages, page_tokens, head_dim, qh, head / group,
                          block_tables + (int64_t)seq * bt_stride, ctx, scale, x);
    if (!bad)
        softmax_weights(x, ctx, w);
    free(x);
    return bad ? ORACLE_ERR_PAGE : 0;
}

/*
 * Paged prefill (and chunked prefill) attention: the query tokens of each sequence are
 * the last n_s of its context_lens[s] tokens; query j of sequence s sits at position
 * p = context_lens[s] - n_s + j and attends causally over tokens 0 .. p:
 *   out[i][h][:] = sum_{t <= p} w_t V_t[h / group][:],  w = softmax_t(scale * q[i][h] . K_t[h / group])
 * (the prefill path of "tiny-vllm part 3": per-head scores, causal mask keeping the
 * diagonal, softmax, scores x V - here reading K/V through the block table).
 * Query rows of sequence s are query_start[s] .. query_start[s+1]-1 of q
 * ([total][num_q_heads][head_dim] bf16); out is FP64 [total][num_q_heads][head_dim].
 * A sequence with n_s > context_lens[s], a context outside [0, max_context] or an
 * invalid page gets zero rows and an error bit.
 */
int oracle_paged_prefill_attention(const uint16_t *k_pool, const uint16_t *v_pool, int64_t page_stride,
                                   int num_pages, int page_tokens, int num_kv_heads, int head_dim,
                                   const uint16_t *q, int num_q_heads, const int32_t *query_start,
                                   const int32_t *block_tables, int64_t bt_stride, const int32_t *context_lens,
                                   int num_seqs, int max_context, double scale, double *out)
{
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        page_tokens <= 0 || num_seqs < 0 || max_context < 0)
        return ORACLE_ERR_ARGS;
    int group = num_q_heads / num_kv_heads;
    int err = 0;
    double *x = (double *)malloc(sizeof(double) * (size_t)(max_context > 0 ? max_context : 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)(max_context > 0 ? max_context : 1));
    for (int s = 0; s < num_seqs; ++s) {
        int q0 = query_start[s], n = query_start[s + 1] - query_start[s];
        int ctx = context_lens[s];
        double *o_seq = out + (int64_t)q0 * num_q_heads * head_dim;
        for (int64_t i = 0; i < (int64_t)n * num_q_heads * head_dim; ++i)
            o_seq[i] = 0.0;
        if (n <= 0)
            continue;
        if (ctx < 0 || ctx > max_context || n > ctx) {
            err |= ORACLE_ERR_CONTEXT;
            continue;
        }
        const int32_t *row = block_tables + (int64_t)s * bt_stride;
        int bad = 0;
        for (int j = 0; j < n && !bad; ++j) {
            int pos = ctx - n + j;
            for (int h = 0; h < num_q_heads; ++h) {
                int g = h / group;
                const uint16_t *qh = q + ((int64_t)(q0 + j) * num_q_heads + h) * head_dim;
                if (head_scores(k_pool, page_stride, num_pages, page_tokens, head_dim, qh, g, row, pos + 1, scale,
                                x)) {
                    bad = 1;
                    break;
                }
                softmax_weights(x, pos + 1, w);
                double *o = o_seq + ((int64_t)j * num_q_heads + h) * head_dim;
                for (int t = 0; t <= pos; ++t) {
                    int64_t page = token_page(row, t, page_tokens, num_pages);
                    int64_t v0 = element_index(page_stride, page, g, t % page_tokens, page_tokens, head_dim);
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += w[t] * bf16_value(v_pool[v0 + d]);
                }
            }
        }
        if (bad) {
            err |= ORACLE_ERR_PAGE;
            for (int64_t i = 0; i < (int64_t)n * num_q_heads * head_dim; ++i)
                o_seq[i] = 0.0;
        }
    }
    free(x);
    free(w);
    return err;
}
