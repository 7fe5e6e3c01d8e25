/*
 * dsa_oracle.c -- plain, slow CPU oracle for the DSA indexer.  TEST
 * INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
 * baseline call it; the library under sparse_attention_token_gb300/ never does.
 * It shares no code, header or table with the CUDA path.
 *
 * What it computes (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子"
 * and "性能模型设计" buckets 6-8: q-k index score, head weight multiply + head
 * reduce + FP8 q/k scale shaping, top-k selection):
 *
 *   x[t,h,s]  = sq[t,h] * sk[s] * sum_d q[t,h,d] * k[s,d]     (fp64; sq = sk = 1 for bf16)
 *   score[t,s] = sum_h w[t,h] * max(x[t,h,s], 0)               (fp64)
 *
 * for every key s visible to query t (causal: s <= pos(t)), then the
 * min(topk_limit, n_visible) keys with the highest score, ties broken toward
 * the lower key index, written as int32 and padded with -1 up to k_out
 * (the op returns top-k of width min(topk_limit, active_seq_len), same page,
 * "DSA Indexer 融合语义算子").  Scores compare as values, so -0.0 == +0.0.
 *
 * Inputs are decoded to fp64 exactly from their bit patterns:
 *   bf16: the upper 16 bits of an IEEE binary32;
 *   e4m3 (OCP FP8): sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0
 *   is subnormal (m/8 * 2^-6); S.1111.111 is NaN (rejected); max 448.
 *
 * Everything is straight loops: one fp64 dot product per (t,h,s), a full
 * qsort of every row by (score desc, index asc), no blocking, no fusion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_E4M3 = 1 };
enum { OR_ORDER_SCORE = 0, OR_ORDER_INDEX = 1 };

/* ---- exact decoding of the storage formats ---------------------------- */

double oracle_bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_double(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

static double load_elem(const void* base, int dtype, int64_t i) {
    if (dtype == OR_BF16) return oracle_bf16_to_double(((const uint16_t*)base)[i]);
    return oracle_e4m3_to_double(((const uint8_t*)base)[i]);
}

/* ---- one row: scores of every visible key ------------------------------ */

typedef struct {
    int q_dtype, k_dtype, H, D;
    const void* q;            /* [total_q, H, D] */
    const float* q_scale;     /* [total_q, H] or NULL */
    const float* w;           /* [total_q, H] */
    const void* k;            /* dense [S, D] or paged [num_pages, page_size, D] */
    const float* k_scale;     /* dense [S] or paged [num_pages, page_size], or NULL */
    int page_size;            /* 0 = dense */
    int num_pages;
    const int32_t* block_row; /* this sequence's block table row (paged) */
    int n_block_row;
} row_ctx;

/* Physical row of logical key s; -1 when the page table does not cover it. */
static int64_t key_row(const row_ctx* c, int64_t s) {
    if (c->page_size == 0) return s;
    int64_t j = s / c->page_size;
    if (j >= c->n_block_row) return -1;
    int32_t page = c->block_row[j];
    if (page < 0 || page >= c->num_pages) return -1;
    return (int64_t)page * c->page_size + s % c->page_size;
}

/* score[t, s] for s in [0, n_vis); bound[s] = sk * sum_h |w'| * sum_d |q k|
 * (the condition number of the sum, for tolerances).  Returns 0 or -1. */
static int score_row(const row_ctx* c, int64_t t, int64_t n_vis, double* score, double* bound) {
    const int H = c->H, D = c->D;
    for (int64_t s = 0; s < n_vis; ++s) {
        int64_t kr = key_row(c, s);
        if (kr < 0) return -1;
        double sk = c->k_scale ? (double)c->k_scale[kr] : 1.0;
        double acc = 0.0, acc_abs = 0.0;
        for (int h = 0; h < H; ++h) {
            double dot = 0.0, dot_abs = 0.0;
            for (int d = 0; d < D; ++d) {
                double qv = load_elem(c->q, c->q_dtype, ((int64_t)t * H + h) * D + d);
                double kv = load_elem(c->k, c->k_dtype, kr * D + d);
                if (isnan(qv) || isnan(kv)) return -1;
                dot += qv * kv;
                dot_abs += fabs(qv * kv);
            }
            double sq = c->q_scale ? (double)c->q_scale[t * H + h] : 1.0;
            double x = sq * sk * dot;
            double wv = (double)c->w[t * H + h];
            acc += wv * (x > 0.0 ? x : 0.0);
            acc_abs += fabs(wv) * sq * sk * dot_abs;
        }
        score[s] = acc;
        if (bound) bound[s] = acc_abs;
    }
    return 0;
}

/* ---- top-k by full sort ----------------------------------------------- */

typedef struct { double score; int64_t idx; } pair_t;

static int cmp_score_desc_idx_asc(const void* a, const void* b) {
    const pair_t* x = (const pair_t*)a;
    const pair_t* y = (const pair_t*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

static int cmp_i32_asc(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* out[0..k_out): the min(topk_limit, n) best of score[0..n), then -1. */
static void topk_row(const double* score, int64_t n, int topk_limit, int k_out, int order,
                     int32_t* out) {
    int64_t keep = n < topk_limit ? n : topk_limit;
    if (keep > k_out) keep = k_out;
    pair_t* p = (pair_t*)malloc(sizeof(pair_t) * (size_t)(n > 0 ? n : 1));
    for (int64_t s = 0; s < n; ++s) { p[s].score = score[s]; p[s].idx = s; }
    qsort(p, (size_t)n, sizeof(pair_t), cmp_score_desc_idx_asc);
    for (int64_t i = 0; i < keep; ++i) out[i] = (int32_t)p[i].idx;
    if (order == OR_ORDER_INDEX) qsort(out, (size_t)keep, sizeof(int32_t), cmp_i32_asc);
    for (int64_t i = keep; i < k_out; ++i) out[i] = -1;
    free(p);
}

/* ---- entry points ------------------------------------------------------ */

/* Top-k of caller-given scores (row r has n[r] visible entries at row*ld). */
int oracle_topk(const double* scores, int64_t ld, int n_rows, const int64_t* n_visible,
                int topk_limit, int k_out, int order, int32_t* topk, int n_threads) {
    if (n_threads > 0) {
#ifdef _OPENMP
        omp_set_num_threads(n_threads);
#endif
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r)
        topk_row(scores + (int64_t)r * ld, n_visible[r], topk_limit, k_out, order,
                 topk + (int64_t)r * k_out);
    return 0;
}

/*
 * Dense single sequence: query t sits at position q_pos0 + t and sees keys
 * s <= min(q_pos0 + t, S - 1).  rows[] selects which query rows to compute
 * (NULL = all T); outputs are indexed by the position in rows[].
 * scores/bound (optional) are [n_rows, ld] fp64, -inf / 0 where invisible.
 */
int oracle_dense(int q_dtype, int k_dtype, const void* q, const float* q_scale, const float* w,
                 const void* k, const float* k_scale, int T, int S, int H, int D, int q_pos0,
                 int topk_limit, int k_out, int order, const int64_t* rows, int n_rows,
                 int32_t* topk, double* scores, double* bound, int64_t ld, int n_threads) {
    if (n_threads > 0) {
#ifdef _OPENMP
        omp_set_num_threads(n_threads);
#endif
    }
    int failed = 0;
    int nr = rows ? n_rows : T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nr; ++i) {
        int64_t t = rows ? rows[i] : i;
        row_ctx c = {q_dtype, k_dtype, H, D, q, q_scale, w, k, k_scale, 0, 0, NULL, 0};
        int64_t pos = (int64_t)q_pos0 + t;
        int64_t n_vis = pos + 1 < S ? pos + 1 : S;
        if (n_vis < 0) n_vis = 0;
        double* sc = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        double* bd = bound ? (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1)) : NULL;
        if (score_row(&c, t, n_vis, sc, bd) != 0) {
#pragma omp atomic write
            failed = 1;
        }
        if (topk) topk_row(sc, n_vis, topk_limit, k_out, order, topk + (int64_t)i * k_out);
        if (scores) {
            for (int64_t s = 0; s < S; ++s)
                scores[(int64_t)i * ld + s] = s < n_vis ? sc[s] : -INFINITY;
        }
        if (bound) {
            for (int64_t s = 0; s < S; ++s) bound[(int64_t)i * ld + s] = s < n_vis ? bd[s] : 0.0;
            free(bd);
        }
        free(sc);
    }
    return failed ? -1 : 0;
}

/*
 * Paged varlen batch: sequence b owns query rows cu_q_lens[b]..cu_q_lens[b+1]-1;
 * its i-th query sits at pos = seq_lens[b] - q_len_b + i and sees keys 0..pos,
 * key s stored at k_cache[block_tables[b][s / page_size]][s % page_size].
 * rows[] (global query row ids, NULL = all) selects the rows to compute.
 * scores/bound (optional) are [n_rows, ld] fp64.
 */
int oracle_paged(int q_dtype, int k_dtype, const void* q, const float* q_scale, const float* w,
                 const void* k_cache, const float* k_scale_cache, int num_pages, int page_size,
                 const int32_t* block_tables, int max_pages_per_seq, const int32_t* cu_q_lens,
                 const int32_t* seq_lens, int B, int H, int D, int topk_limit, int k_out, int order,
                 const int64_t* rows, int n_rows, int32_t* topk, double* scores, double* bound,
                 int64_t ld, int n_threads) {
    if (n_threads > 0) {
#ifdef _OPENMP
        omp_set_num_threads(n_threads);
#endif
    }
    int total_q = cu_q_lens[B];
    int nr = rows ? n_rows : total_q;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nr; ++i) {
        int64_t r = rows ? rows[i] : i;
        int b = 0;
        while (b < B && cu_q_lens[b + 1] <= r) ++b;
        int64_t q_len = cu_q_lens[b + 1] - cu_q_lens[b];
        int64_t local = r - cu_q_lens[b];
        int64_t pos = (int64_t)seq_lens[b] - q_len + local;
        int64_t n_vis = pos + 1;
        if (n_vis < 0) n_vis = 0;
        row_ctx c = {q_dtype, k_dtype, H, D, q, q_scale, w, k_cache, k_scale_cache, page_size,
                     num_pages, block_tables + (int64_t)b * max_pages_per_seq, max_pages_per_seq};
        double* sc = (double*)malloc(sizeof(double) * (size_t)(n_vis > 0 ? n_vis : 1));
        double* bd = bound ? (double*)malloc(sizeof(double) * (size_t)(n_vis > 0 ? n_vis : 1)) : NULL;
        if (score_row(&c, r, n_vis, sc, bd) != 0) {
#pragma omp atomic write
            failed = 1;
        }
        if (topk) topk_row(sc, n_vis, topk_limit, k_out, order, topk + (int64_t)i * k_out);
        if (scores) {
            for (int64_t s = 0; s < ld; ++s)
                scores[(int64_t)i * ld + s] = s < n_vis ? sc[s] : -INFINITY;
        }
        if (bound) {
            for (int64_t s = 0; s < ld; ++s) bound[(int64_t)i * ld + s] = s < n_vis ? bd[s] : 0.0;
            free(bd);
        }
        free(sc);
    }
    return failed ? -1 : 0;
}

/* ---- cache append -------------------------------------------------------
 * The fused op takes the indexer cache as a mutable argument together with
 * slot_mapping (GLM5 TensorCast adaptation design, "DSA Indexer 融合语义算子"), and
 * its FP8 path writes the key cache and the scale cache after an activation
 * quantisation ("FP8 key cache/scale cache 写入"; cost buckets 9 and 10).  The pages
 * do not print the quantiser; the reading taken is one fp32 scale per token,
 * scale = amax / 448 (amax = the largest |k| of the token's row; 1 for an all-zero
 * row), and code = the e4m3 value nearest to k / scale.
 *
 * Encoding to e4m3 by its definition: the finite non-negative codes 0x00..0x7E are
 * enumerated and the one whose value is nearest to |v| wins; of two equally near
 * neighbours the one with an even code (mantissa lsb 0) wins; beyond 448 the
 * nearest finite code is 448 itself (saturation).  The sign bit is copied, so -0.0
 * becomes 0x80.  NaN becomes 0x7F. */
uint8_t oracle_e4m3_encode(float v) {
    if (v != v) return 0x7F;
    const double a = fabs((double)v);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double d = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* k_new [n, D] bf16 rows go to cache slots slots[i] (slot = page * page_size + row;
 * negative: the token is skipped).  bf16 cache: the row is copied.  e4m3 cache: the
 * row is quantised as above, in fp32 arithmetic (amax of the decoded values, one
 * division for the scale, one division per element), and the scale goes to
 * scale_cache[slot].  Returns -1 (writing nothing further) at a slot >= n_slots. */
int oracle_cache_append(const uint16_t* k_new, int n, int D, const int64_t* slots, int cache_dtype, void* cache,
                        float* scale_cache, int64_t n_slots) {
    for (int i = 0; i < n; ++i) {
        const int64_t slot = slots[i];
        if (slot < 0) continue;
        if (slot >= n_slots) return -1;
        const uint16_t* row = k_new + (int64_t)i * D;
        if (cache_dtype == OR_BF16) {
            memcpy((uint16_t*)cache + slot * D, row, (size_t)D * sizeof(uint16_t));
            continue;
        }
        float amax = 0.0f;
        for (int d = 0; d < D; ++d) {
            const float x = (float)oracle_bf16_to_double(row[d]);
            if (fabsf(x) > amax) amax = fabsf(x);
        }
        const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        uint8_t* out = (uint8_t*)cache + slot * D;
        for (int d = 0; d < D; ++d) out[d] = oracle_e4m3_encode((float)oracle_bf16_to_double(row[d]) / scale);
        scale_cache[slot] = scale;
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
