/*
 * pa_oracle.c -- plain, slow, obviously correct CPU oracle for exact paged
 * attention, in fp64.  TEST INFRASTRUCTURE ONLY: nothing on the product path
 * links, loads or calls this file.  It shares no code with the CUDA library.
 *
 * The method, as the pages define it, and the function below that follows it:
 *
 *   gather_one()  -- "Week 3 Day 5: Paged FlashAttention", Task 1: every
 *                    logical key position s is translated through the block
 *                    table (logical_page = s / page_size, slot = s % page_size,
 *                    physical_page = block_table[batch, logical_page]) and the
 *                    row pages[physical_page, kv_head, slot, :] is read.  The
 *                    whole history is first gathered into a contiguous buffer,
 *                    as the reference of "Day 22: the fused paged-attention
 *                    kernel" (What I added today) does.
 *   kv_head_of()  -- "Week 2 Day 5: Fused Decode Attention", Task 1:
 *                    kv_head = query_head / (H_q / H_kv).
 *   attend_row()  -- scaled scores, softmax, weighted sum of values, written
 *                    out explicitly ("Week 2 Day 5", Task 1: the readable
 *                    equation kept as the oracle), restricted to the visible
 *                    keys s <= l + context_len - L under the causal rule of
 *                    "Week 3 Day 5", Task 2.  Natural exp in double; the max
 *                    is subtracted before exponentiating (stable softmax).
 *
 *   oracle_paged_attention_varlen() -- a ragged batch (per-sequence query
 *                    counts, tokens packed): each sequence's rows are those of
 *                    a batch of that sequence alone ("Day 22: the fused
 *                    paged-attention kernel": decode steps, causal prefills
 *                    and partial continuations are all the same fold; "Week 3
 *                    Day 5", Task 2: the causal offset is that sequence's
 *                    context length minus its own query count).
 *   oracle_append_kv() -- the step before the path: the new tokens' K/V rows
 *                    are stored in their pages.  The pages introduce physical
 *                    pages and block tables as the prerequisite of "Week 3 Day
 *                    5: Paged FlashAttention" (Prerequisites) and give the
 *                    read-side translation in Task 1; the write uses the same
 *                    translation for the last L positions of each context.
 *
 * No tiling, no online rescaling, no reordering beyond the definition.
 * Parallelism: independent (batch, kv_head) items run on OpenMP threads; each
 * row is computed by one thread in the definition's order.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake.  It
 * exists only so that the CPU test suite can show that its pins catch such
 * mistakes; the normal build never defines it.
 */
#include "pa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* Exact widening of one stored element to double. */
static double widen(const void* base, int dtype, int64_t idx) {
    if (dtype == 0) {
        uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

static int check_shape(const oracle_shape* sh) {
    if (!sh) return ORACLE_ERR_INVALID_ARG;
    if (sh->B < 1 || sh->H_q < 1 || sh->H_kv < 1 || sh->L < 1 || sh->D < 1 ||
        sh->num_pages < 1 || sh->page_size < 1 || sh->max_pages_per_seq < 1)
        return ORACLE_ERR_INVALID_ARG;
    if (sh->H_q % sh->H_kv != 0) return ORACLE_ERR_INVALID_ARG;
    if (sh->dtype != 0 && sh->dtype != 1) return ORACLE_ERR_INVALID_ARG;
    return ORACLE_OK;
}

/* Validates what the method will read for sequence b: its context length and
 * the block-table entries of its ceil(S / page_size) logical pages. */
static int check_sequence_lq(const oracle_shape* sh, const int32_t* block_table,
                             const int32_t* context_lens, int b, int causal, int L) {
    const int S = context_lens[b];
    if (S < 1 || (int64_t)S > (int64_t)sh->max_pages_per_seq * sh->page_size)
        return ORACLE_ERR_INVALID_ARG;
    if (causal && L > S) return ORACLE_ERR_INVALID_ARG;
    const int npg = (S + sh->page_size - 1) / sh->page_size;
    for (int lp = 0; lp < npg; ++lp) {
        const int32_t pp = block_table[(int64_t)b * sh->max_pages_per_seq + lp];
        if (pp < 0 || pp >= sh->num_pages) return ORACLE_ERR_BAD_BLOCK_TABLE;
    }
    return ORACLE_OK;
}

/* The same for sequences with sh->L query positions each. */
static int check_sequence(const oracle_shape* sh, const int32_t* block_table,
                          const int32_t* context_lens, int b, int causal) {
    return check_sequence_lq(sh, block_table, context_lens, b, causal, sh->L);
}

static int kv_head_of(const oracle_shape* sh, int h) {
#if ORACLE_MUTANT == 2
    return h % sh->H_kv; /* planted: wrong GQA head map */
#else
    return h / (sh->H_q / sh->H_kv);
#endif
}

/* Gathers the S logical rows of (b, kvh) into K[S][D], V[S][D]. */
static void gather_one(const oracle_shape* sh, const void* key_pages, const void* value_pages,
                       const int32_t* block_table, int b, int kvh, int S, double* K,
                       double* V) {
    const int ps = sh->page_size, D = sh->D;
    for (int s = 0; s < S; ++s) {
        const int logical_page = s / ps;
#if ORACLE_MUTANT == 12
        const int slot = (s + 1) % ps; /* planted: slot off by one within its page */
#else
        const int slot = s % ps;
#endif
#if ORACLE_MUTANT == 3
        const int64_t physical_page = logical_page; /* planted: block table ignored */
#else
        const int64_t physical_page =
            block_table[(int64_t)b * sh->max_pages_per_seq + logical_page];
#endif
        const int64_t row = ((physical_page * sh->H_kv + kvh) * ps + slot) * (int64_t)D;
        for (int d = 0; d < D; ++d) {
#if ORACLE_MUTANT == 5
            K[(int64_t)s * D + d] = widen(value_pages, sh->dtype, row + d); /* planted: K/V swapped */
            V[(int64_t)s * D + d] = widen(key_pages, sh->dtype, row + d);
#else
            K[(int64_t)s * D + d] = widen(key_pages, sh->dtype, row + d);
            V[(int64_t)s * D + d] = widen(value_pages, sh->dtype, row + d);
#endif
        }
    }
}

/* One output row (b, h, l) from the gathered K/V of its kv head.
 * x is scratch for S scores, o receives D outputs.  mask_row, when not NULL,
 * is the row's additive mask over logical key positions: it is added to the
 * scaled score before the softmax ("Week 2 Day 5: Fused Decode Attention",
 * Task 1, step 3: the score is scaled, then masked, then the causal rule
 * applies).  A row whose every visible score is -inf has no softmax; its
 * output is 0. */
static void attend_row(const oracle_shape* sh, const void* query, int64_t qbase, int l, int L,
                       int S, const double* K, const double* V, double scale, int causal,
                       const float* mask_row, double* x, double* o) {
    /* qbase: index of the row's first query element; l: its position among
     * the sequence's L query positions (the last L of its S keys) */
    const int D = sh->D;
    /* last visible key: s <= l + S - L under causal, s <= S - 1 otherwise */
#if ORACLE_MUTANT == 1
    int last = causal ? l + S - L - 1 : S - 1; /* planted: causal off by one */
#elif ORACLE_MUTANT == 7
    int last = causal ? l - S + L : S - 1; /* planted: causal offset sign flipped */
#else
    int last = causal ? l + S - L : S - 1;
#endif
    if (last > S - 1) last = S - 1;

    double M = -INFINITY;
    for (int s = 0; s <= last; ++s) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += widen(query, sh->dtype, qbase + d) * K[(int64_t)s * D + d];
#if ORACLE_MUTANT == 4
        x[s] = acc; /* planted: scale dropped */
#else
        x[s] = scale * acc;
#endif
#if ORACLE_MUTANT == 9
        if (mask_row) x[s] -= (double)mask_row[s]; /* planted: mask subtracted */
#else
        if (mask_row) x[s] += (double)mask_row[s];
#endif
        if (x[s] > M) M = x[s];
    }
    double den = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (M == -INFINITY) return; /* every visible key masked out */
    for (int s = 0; s <= last; ++s) {
#if ORACLE_MUTANT == 11
        const double w = exp(x[s]); /* planted: the max not subtracted */
#else
        const double w = exp(x[s] - M);
#endif
#if ORACLE_MUTANT == 6
        if (s > 0) den += w; /* planted: a dropped term in the normaliser */
#else
        den += w;
#endif
        for (int d = 0; d < D; ++d) o[d] += w * V[(int64_t)s * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= den;
}

static int validate_all(const oracle_shape* sh, const int32_t* block_table,
                        const int32_t* context_lens, int causal) {
    int st = check_shape(sh);
    if (st) return st;
    for (int b = 0; b < sh->B; ++b) {
        st = check_sequence(sh, block_table, context_lens, b, causal);
        if (st) return st;
    }
    return ORACLE_OK;
}

int oracle_gather(const oracle_shape* sh, const void* key_pages, const void* value_pages,
                  const int32_t* block_table, const int32_t* context_lens, int max_S,
                  double* k_dense, double* v_dense) {
    if (!key_pages || !value_pages || !block_table || !context_lens || !k_dense || !v_dense)
        return ORACLE_ERR_INVALID_ARG;
    int st = validate_all(sh, block_table, context_lens, 0);
    if (st) return st;
    const int D = sh->D;
    for (int b = 0; b < sh->B; ++b)
        if (context_lens[b] > max_S) return ORACLE_ERR_INVALID_ARG;
    for (int b = 0; b < sh->B; ++b) {
        for (int kvh = 0; kvh < sh->H_kv; ++kvh) {
            const int64_t base = ((int64_t)b * sh->H_kv + kvh) * max_S * D;
            memset(k_dense + base, 0, sizeof(double) * (size_t)max_S * D);
            memset(v_dense + base, 0, sizeof(double) * (size_t)max_S * D);
            gather_one(sh, key_pages, value_pages, block_table, b, kvh, context_lens[b],
                       k_dense + base, v_dense + base);
        }
    }
    return ORACLE_OK;
}

int oracle_paged_attention(const oracle_shape* sh, const void* query, const void* key_pages,
                           const void* value_pages, const int32_t* block_table,
                           const int32_t* context_lens, double scale, int causal,
                           double* out, int num_threads) {
    return oracle_paged_attention_masked(sh, query, key_pages, value_pages, block_table,
                                         context_lens, scale, causal, NULL, 0, out, num_threads);
}

int oracle_paged_attention_masked(const oracle_shape* sh, const void* query,
                                  const void* key_pages, const void* value_pages,
                                  const int32_t* block_table, const int32_t* context_lens,
                                  double scale, int causal, const float* mask, int mask_S,
                                  double* out, int num_threads) {
    if (!query || !key_pages || !value_pages || !block_table || !context_lens || !out)
        return ORACLE_ERR_INVALID_ARG;
    int st = validate_all(sh, block_table, context_lens, causal);
    if (st) return st;
    if (mask)
        for (int b = 0; b < sh->B; ++b)
            if (context_lens[b] > mask_S) return ORACLE_ERR_INVALID_ARG;
    const int G = sh->H_q / sh->H_kv, D = sh->D;
    const int n_items = sh->B * sh->H_kv;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int item = 0; item < n_items; ++item) {
        const int b = item / sh->H_kv, kvh = item % sh->H_kv;
#if ORACLE_MUTANT == 13
        const int S = context_lens[b] - 1; /* planted: the context's last key dropped */
#else
        const int S = context_lens[b];
#endif
        double* K = (double*)malloc(sizeof(double) * (size_t)S * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)S * D);
        double* x = (double*)malloc(sizeof(double) * (size_t)S);
        if (!K || !V || !x) {
            failed = 1;
        } else {
            gather_one(sh, key_pages, value_pages, block_table, b, kvh, S, K, V);
            for (int h = 0; h < sh->H_q; ++h) {
                if (kv_head_of(sh, h) != kvh) continue;
                for (int l = 0; l < sh->L; ++l)
                    attend_row(sh, query, (((int64_t)b * sh->H_q + h) * sh->L + l) * D, l,
                               sh->L, S, K, V, scale, causal,
                               mask ? mask + (((int64_t)b * sh->H_q + h) * sh->L + l) * mask_S
                                    : NULL,
                               x, out + (((int64_t)b * sh->H_q + h) * sh->L + l) * D);
            }
        }
        free(K);
        free(V);
        free(x);
    }
    (void)G;
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int oracle_paged_attention_rows(const oracle_shape* sh, const void* query,
                                const void* key_pages, const void* value_pages,
                                const int32_t* block_table, const int32_t* context_lens,
                                double scale, int causal, const int32_t* rows, int n_rows,
                                double* out, int num_threads) {
    if (!query || !key_pages || !value_pages || !block_table || !context_lens || !out ||
        (!rows && n_rows > 0) || n_rows < 0)
        return ORACLE_ERR_INVALID_ARG;
    int st = validate_all(sh, block_table, context_lens, causal);
    if (st) return st;
    for (int i = 0; i < n_rows; ++i) {
        const int b = rows[3 * i], h = rows[3 * i + 1], l = rows[3 * i + 2];
        if (b < 0 || b >= sh->B || h < 0 || h >= sh->H_q || l < 0 || l >= sh->L)
            return ORACLE_ERR_INVALID_ARG;
    }
    const int D = sh->D;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int i = 0; i < n_rows; ++i) {
        const int b = rows[3 * i], h = rows[3 * i + 1], l = rows[3 * i + 2];
        const int S = context_lens[b];
        const int kvh = kv_head_of(sh, h);
        double* K = (double*)malloc(sizeof(double) * (size_t)S * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)S * D);
        double* x = (double*)malloc(sizeof(double) * (size_t)S);
        if (!K || !V || !x) {
            failed = 1;
        } else {
            gather_one(sh, key_pages, value_pages, block_table, b, kvh, S, K, V);
            attend_row(sh, query, (((int64_t)b * sh->H_q + h) * sh->L + l) * D, l, sh->L, S, K,
                       V, scale, causal, NULL, x, out + (int64_t)i * D);
        }
        free(K);
        free(V);
        free(x);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Ragged batch: sequence b has L_b = cu_q[b + 1] - cu_q[b] query positions,
 * its last L_b of context_lens[b] keys (a decode step has L_b = 1, a prefill
 * chunk L_b > 1, a sequence without new queries L_b = 0).  Queries and
 * outputs are packed by token: row (b, h, l) is token cu_q[b] + l of
 * [total_q, H_q, D].  Each row is the row of a batch of one sequence with L_b
 * positions; rows of sequences with L_b = 0 do not exist and nothing of
 * those sequences is read. */
int oracle_paged_attention_varlen(const oracle_shape* sh, const void* query,
                                  const void* key_pages, const void* value_pages,
                                  const int32_t* block_table, const int32_t* context_lens,
                                  const int32_t* cu_q, int total_q, double scale, int causal,
                                  double* out, int num_threads) {
    if (!query || !key_pages || !value_pages || !block_table || !context_lens || !cu_q || !out)
        return ORACLE_ERR_INVALID_ARG;
    int st = check_shape(sh);
    if (st) return st;
    if (cu_q[0] != 0 || cu_q[sh->B] != total_q) return ORACLE_ERR_INVALID_ARG;
    for (int b = 0; b < sh->B; ++b) {
        const int Lb = cu_q[b + 1] - cu_q[b];
        if (Lb < 0 || Lb > sh->L) return ORACLE_ERR_INVALID_ARG;
        if (Lb == 0) continue;
        st = check_sequence_lq(sh, block_table, context_lens, b, causal, Lb);
        if (st) return st;
    }
    const int D = sh->D;
    const int n_items = sh->B * sh->H_kv;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int item = 0; item < n_items; ++item) {
        const int b = item / sh->H_kv, kvh = item % sh->H_kv;
        const int Lb = cu_q[b + 1] - cu_q[b];
        if (Lb == 0) continue;
        const int S = context_lens[b];
        double* K = (double*)malloc(sizeof(double) * (size_t)S * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)S * D);
        double* x = (double*)malloc(sizeof(double) * (size_t)S);
        if (!K || !V || !x) {
            failed = 1;
        } else {
            gather_one(sh, key_pages, value_pages, block_table, b, kvh, S, K, V);
            for (int h = 0; h < sh->H_q; ++h) {
                if (kv_head_of(sh, h) != kvh) continue;
                for (int l = 0; l < Lb; ++l) {
                    const int64_t row = ((int64_t)(cu_q[b] + l) * sh->H_q + h) * D;
#if ORACLE_MUTANT == 10
                    const int Lq = sh->L; /* planted: the batch's longest query as offset */
#else
                    const int Lq = Lb;
#endif
                    attend_row(sh, query, row, l, Lq, S, K, V, scale, causal, NULL, x, out + row);
                }
            }
        }
        free(K);
        free(V);
        free(x);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Append of new keys and values.  The L new tokens of sequence b are the last
 * L logical positions of its context, s = context_lens[b] - L + t, and are
 * written through the block table into
 *   pages[block_table[b, s / page_size], kv_head, s % page_size, :].
 * Elements are copied as stored (bf16 bit patterns or fp32), so the append is
 * exact.  Sequences whose context length is < L or > the table's capacity are
 * skipped (ORACLE_ERR_INVALID_ARG); a token whose page id is out of range is
 * skipped (ORACLE_ERR_BAD_BLOCK_TABLE); everything else is written. */
int oracle_append_kv(const oracle_shape* sh, const void* k_new, const void* v_new,
                     void* key_pages, void* value_pages, const int32_t* block_table,
                     const int32_t* context_lens) {
    int st = check_shape(sh);
    if (st != ORACLE_OK) return st;
    const int64_t es = sh->dtype == 0 ? 2 : 4;
    const int64_t row_bytes = (int64_t)sh->D * es;
    const int ps = sh->page_size, L = sh->L;
    int bad_ctx = 0, bad_page = 0;
    for (int b = 0; b < sh->B; ++b) {
        const int S = context_lens[b];
        if (S < L || (int64_t)S > (int64_t)sh->max_pages_per_seq * ps) {
            bad_ctx = 1;
            continue;
        }
        for (int kvh = 0; kvh < sh->H_kv; ++kvh) {
            for (int t = 0; t < L; ++t) {
                const int s = S - L + t;
#if ORACLE_MUTANT == 8
                const int slot = (s + 1) % ps; /* planted: slot off by one */
#else
                const int slot = s % ps;
#endif
                const int32_t pp = block_table[(int64_t)b * sh->max_pages_per_seq + s / ps];
                if (pp < 0 || pp >= sh->num_pages) {
                    bad_page = 1;
                    continue;
                }
                const int64_t src = (((int64_t)b * sh->H_kv + kvh) * L + t) * row_bytes;
                const int64_t dst = (((int64_t)pp * sh->H_kv + kvh) * ps + slot) * row_bytes;
                memcpy((char*)key_pages + dst, (const char*)k_new + src, (size_t)row_bytes);
                memcpy((char*)value_pages + dst, (const char*)v_new + src, (size_t)row_bytes);
            }
        }
    }
    if (bad_ctx) return ORACLE_ERR_INVALID_ARG;
    return bad_page ? ORACLE_ERR_BAD_BLOCK_TABLE : ORACLE_OK;
}
