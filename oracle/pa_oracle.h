/*
 * pa_oracle.h -- CPU oracle for exact paged attention (TEST INFRASTRUCTURE).
 *
 * This header belongs to the oracle only.  It is not included by, and shares
 * no code, constants or helpers with, the CUDA library under
 * paged_kv_cache_03_gb300/.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load the oracle.
 *
 * What it computes (plain definition, fp64):
 *   - GQA head map: kv_head = q_head / (H_q / H_kv)
 *       ("Week 2 Day 5: Fused Decode Attention", Task 1)
 *   - Page translation of every logical key position s < context_len:
 *       logical_page = s / page_size, slot = s % page_size,
 *       physical_page = block_table[b, logical_page],
 *       row = pages[physical_page, kv_head, slot, :]
 *       ("Week 3 Day 5: Paged FlashAttention", Task 1)
 *   - Causal visibility: key s is visible to query row l iff
 *       s <= l + context_len - L   ("Week 3 Day 5", Task 2)
 *   - One softmax over the gathered, visible scores, then the weighted sum
 *       of value rows ("Day 22: the fused paged-attention kernel", the
 *       gather-then-softmax reference it is pinned against).
 *
 * Layouts (all row-major, contiguous):
 *   query        [B, H_q, L, D]
 *   key_pages    [num_pages, H_kv, page_size, D]
 *   value_pages  [num_pages, H_kv, page_size, D]
 *   block_table  [B, max_pages_per_seq]   int32
 *   context_lens [B]                      int32
 *   out          [B, H_q, L, D]           double
 * Element type of query/key_pages/value_pages: dtype 0 = bf16 bit patterns
 * (uint16), dtype 1 = IEEE fp32.  Both widen exactly to double.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int B, H_q, H_kv, L, D, num_pages, page_size, max_pages_per_seq;
    int dtype; /* 0 = bf16 bits, 1 = fp32 */
} oracle_shape;

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_INVALID_ARG = 1,    /* bad shape, H_q % H_kv != 0, bad context length */
    ORACLE_ERR_BAD_BLOCK_TABLE = 3, /* a page id that would be read is out of range */
    ORACLE_ERR_NOMEM = 7
};

/* Dense gather through the block table: k_dense/v_dense [B, H_kv, max_S, D]
 * (double).  Positions s >= context_lens[b] are written as 0. */
int oracle_gather(const oracle_shape* sh, const void* key_pages, const void* value_pages,
                  const int32_t* block_table, const int32_t* context_lens, int max_S,
                  double* k_dense, double* v_dense);

/* Full attention for every (b, q_head, l) row; out is [B, H_q, L, D] double. */
int oracle_paged_attention(const oracle_shape* sh, const void* query, const void* key_pages,
                           const void* value_pages, const int32_t* block_table,
                           const int32_t* context_lens, double scale, int causal,
                           double* out, int num_threads);

/* Full attention with an explicit additive mask (fp32) over logical key
 * positions, laid out [B * H_q, L, mask_S] with mask_S >= every context
 * length: mask[(b * H_q + h) * L + l][s] is added to the scaled score of key
 * s for row (b, h, l) before the softmax ("Week 2 Day 5: Fused Decode
 * Attention", Task 1 normalises explicit masks to [B * H_q, L, S]); the causal
 * rule still applies when causal != 0.  A row whose every visible score is
 * -inf outputs 0.  mask == NULL is oracle_paged_attention. */
int oracle_paged_attention_masked(const oracle_shape* sh, const void* query,
                                  const void* key_pages, const void* value_pages,
                                  const int32_t* block_table, const int32_t* context_lens,
                                  double scale, int causal, const float* mask, int mask_S,
                                  double* out, int num_threads);

/* The same, for a chosen list of rows only: rows is [n_rows][3] = (b, q_head, l);
 * out is [n_rows, D] double. */
int oracle_paged_attention_rows(const oracle_shape* sh, const void* query,
                                const void* key_pages, const void* value_pages,
                                const int32_t* block_table, const int32_t* context_lens,
                                double scale, int causal, const int32_t* rows, int n_rows,
                                double* out, int num_threads);

/* Ragged batch: sequence b has L_b = cu_q[b+1] - cu_q[b] query positions
 * (0 <= L_b <= sh->L; cu_q[0] = 0, cu_q[B] = total_q), the last L_b of its
 * context; query and out are packed [total_q, H_q, D] (row (b, h, l) is token
 * cu_q[b] + l).  Sequences with L_b = 0 are skipped unread. */
int oracle_paged_attention_varlen(const oracle_shape* sh, const void* query,
                                  const void* key_pages, const void* value_pages,
                                  const int32_t* block_table, const int32_t* context_lens,
                                  const int32_t* cu_q, int total_q, double scale, int causal,
                                  double* out, int num_threads);

/* Append of new keys and values (the step before the path: the new tokens'
 * K/V stored in their pages).  Shape fields used: B, H_kv, L (new tokens per
 * sequence), D, num_pages, page_size, max_pages_per_seq, dtype.  The new
 * tokens of sequence b are its last L logical positions
 * s = context_lens[b] - L + t; their rows are copied, as stored, from
 * k_new/v_new [B, H_kv, L, D] to
 *   key_pages/value_pages[block_table[b, s / page_size], kv_head, s % page_size, :].
 * Sequences with context_lens[b] < L or beyond the table's capacity are
 * skipped (ORACLE_ERR_INVALID_ARG); tokens whose page id is out of range are
 * skipped (ORACLE_ERR_BAD_BLOCK_TABLE). */
int oracle_append_kv(const oracle_shape* sh, const void* k_new, const void* v_new,
                     void* key_pages, void* value_pages, const int32_t* block_table,
                     const int32_t* context_lens);

#ifdef __cplusplus
}
#endif
#endif
