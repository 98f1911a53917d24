/*
 * dattn oracle: TEST INFRASTRUCTURE ONLY.
 *
 * This is a plain, slow CPU implementation of what the split-KV decode path computes. It
 * works in double precision and is written to be checked by eye against the source pages.
 * It exists only to check the CUDA library: only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header, table or helper with
 * the CUDA path. It takes the same bf16 inputs (as raw 16-bit patterns) and widens them
 * exactly to double.
 *
 * Sources, cited by page title and section:
 *  [IL]  "Infinite-LLM: Efficient LLM Service for Long Context with DistAttention and
 *        Distributed KVCache" (paper notes).
 *        - 速读 / 怎么做的: the MicroAttention equations for m_j, e_j, MA_j and the
 *          aggregation equations for m_g, e_g and Attention.
 *        - 分布式注意力机制的通信挑战: full softmax attention written with the global max m_g.
 *        - DistAttention 的等价数学变换: MicroAttention over a local chunk of seq_p keys.
 *        - 结果聚合与通信开销降低: aggregation of the b partial results (Fig. 4b).
 *  [LS]  "LoongServe: Efficiently Serving Long-Context Large Language Models with Elastic
 *        Sequence Parallelism" (paper notes). §4.2 Elastic Scale-up: single-master and
 *        multi-master distributed decoding. The master saves the new token's KV locally,
 *        every instance computes local attention, and the results are merged.
 *  [LV]  "LLM长序列服务优化：LServe的块稀疏注意力技术" (blog article).
 *        - §2.2.2 解码阶段创新: hierarchical paging (64-token physical pages of 16-token
 *          logical pages with k_max/k_min) and the reusable page selector.
 *        - §3.1.1 流式头的转换与优化: streaming heads attend sink tokens plus a local window.
 *        - §3.1.2 动态稀疏的层次化选择: logical-page statistics, physical-page scoring as a
 *          max over logical pages, and top-K selection. Statistics are computed when the KV
 *          cache is written.
 *
 * Readings taken where the pages leave a step open (labels are local to this file):
 *  R1  A logit is s_i = scale * (q . k_i); the pages write QK without the 1/sqrt(d) factor.
 *  R2  GQA: query head h reads KV head h / g, where g = Hq / Hkv.
 *  R3  An empty key set gives m = -inf, e = 0 and MA = out = 0.
 *  R4  The logical-page score is sum_d max(q_d*kmax_d, q_d*kmin_d). The physical-page
 *      score is the max over its logical pages that hold at least one written token.
 *  R5  With g query heads sharing a KV head, the page score is the max over the g heads.
 *  R6  Top-K order: higher score first; ties go to the lower page index. The result is
 *      returned in ascending page order, padded with -1.
 *  R7  A streaming head at length L attends [0, min(S, L)) U [max(S, L - W), L).
 *  R8  k_max/k_min use strict comparison in token order, so the first-seen value wins a
 *      tie (this matters only for +0/-0).
 *  R9  The page selection is defined by the fp64 score (R4, R5) and the top-K rule (R6).
 *      A GPU computes the score in fp32, so where two pages' scores lie within the
 *      rounding error of an fp32 evaluation the selection is not unique. The oracle
 *      therefore returns, next to each fp64 score, a bound on the error of ANY fp32
 *      evaluation of it (any summation order): the classical bound for a floating-point
 *      sum of n terms, |fl(sum) - sum| <= (n-1) u / (1 - (n-1) u) * sum |t_i|
 *      (Higham, "Accuracy and Stability of Numerical Algorithms", 2nd ed., eq. 4.4),
 *      with u = 2^-24. It is taken as d * 2^-23 * sum |t_i|, which covers n = 2d terms
 *      (an evaluation may add the k_max and the k_min half as separate products), plus
 *      2d * 2^-150 for products that fall below the fp32 normal range. The tests accept a
 *      GPU selection bit for bit where the margin between the chosen and the rejected
 *      pages exceeds these bounds, and otherwise check that it is a valid top-K under them.
 *  R10 The 8-bit KV cache: the pages give retrieval heads 2-8 bit configurable quantization
 *      and no scheme. Here: FP8 E4M3 codes with one fp32 scale per (token, KV head) row of
 *      K and of V, scale = max|x| / 448, code = E4M3(x / scale) rounded to nearest even;
 *      attention runs over code * scale. Statistics for page selection are still taken
 *      from the bf16 keys as written.
 *  R12 The 4-bit KV cache: the pages keep streaming heads at 4 bits and give retrieval heads
 *      2-8 bit configurable quantization, again with no scheme. Here: symmetric integer
 *      codes with one fp32 scale per (token, KV head) row of K and of V, scale = max|x| / 7
 *      and code = x / scale rounded to the nearest integer, ties to even, in [-7, 7] (both
 *      divisions in IEEE fp32). Byte i of a row holds code + 8 of channel 2i in its low
 *      nibble and of channel 2i + 1 in its high nibble; a row whose scale is 0 has code 0
 *      (nibble 8) everywhere. Attention runs over code * scale; statistics for page
 *      selection are still taken from the bf16 keys as written.
 *  R11 Block-sparse prefill [LV §2.1.1, §2.1.2, §2.2.1]: key blocks of 64 tokens. Query token
 *      t of a chunk of Tq new tokens sits at position p = L - Tq + t (L counts the chunk) and
 *      attends the keys i <= p whose block kb = i / 64 its head keeps for the query's block
 *      qb = p / 64: every kb <= qb (dense head); kb < sink_blocks or qb - local_blocks <
 *      kb <= qb (streaming head, the Lambda shape); the listed blocks (retrieval head, the
 *      caller's runtime selection, taken literally as the decode takes its page selection).
 */
#include "dattn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double. A bf16 value is the high half of an IEEE binary32, so widening is exact. */
double orc_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static float bf16_to_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Logit of one key, per reading R1: s = scale * sum_d q_d k_d, summed in double. */
static double logit(const uint16_t *q, const uint16_t *k, int d, double scale)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
        acc += orc_bf16_to_double(q[c]) * orc_bf16_to_double(k[c]);
    return scale * acc;
}

static int64_t row_of(const int64_t *rows, int64_t i) { return rows ? rows[i] : i; }

/*
 * Full softmax attention of one query over a key set [IL, 分布式注意力机制的通信挑战]:
 *   m_g = max_i s_i,   Attention = sum_i exp(s_i - m_g) v_i / sum_j exp(s_j - m_g).
 * Row r of K and V starts at K + r * row_stride. The key set is rows[0..n), or 0..n-1 when
 * rows is NULL. out has d entries. e_out receives sum_j exp(s_j - m_g).
 */
void orc_attention(const uint16_t *q, const uint16_t *K, const uint16_t *V, int64_t row_stride,
                   int d, const int64_t *rows, int64_t n, double scale, double *out,
                   double *m_out, double *e_out)
{
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (n <= 0) { /* reading R3 */
        *m_out = -INFINITY;
        *e_out = 0.0;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        s[i] = logit(q, K + row_of(rows, i) * row_stride, d, scale);
        if (s[i] > m) m = s[i];
    }
    double e = 0.0;
    for (int64_t i = 0; i < n; ++i) e += exp(s[i] - m);
    for (int64_t i = 0; i < n; ++i) {
        const double w = exp(s[i] - m) / e;
        const uint16_t *v = V + row_of(rows, i) * row_stride;
        for (int c = 0; c < d; ++c) out[c] += w * orc_bf16_to_double(v[c]);
    }
    free(s);
    *m_out = m;
    *e_out = e;
}

/*
 * MicroAttention over one chunk of keys [IL, DistAttention 的等价数学变换]:
 *   m_j = max_i s_i,  e_j = sum_i exp(s_i - m_j),  MA_j = sum_i exp(s_i - m_j) v_i.
 * MA_j is left unnormalised, as on the page. An empty chunk gives (-inf, 0, 0) (R3).
 */
void orc_partial(const uint16_t *q, const uint16_t *K, const uint16_t *V, int64_t row_stride,
                 int d, const int64_t *rows, int64_t n, double scale, double *m_j, double *e_j,
                 double *MA_j)
{
    for (int c = 0; c < d; ++c) MA_j[c] = 0.0;
    if (n <= 0) {
        *m_j = -INFINITY;
        *e_j = 0.0;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        s[i] = logit(q, K + row_of(rows, i) * row_stride, d, scale);
        if (s[i] > m) m = s[i];
    }
    double e = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double w = exp(s[i] - m);
        const uint16_t *v = V + row_of(rows, i) * row_stride;
        e += w;
        for (int c = 0; c < d; ++c) MA_j[c] += w * orc_bf16_to_double(v[c]);
    }
    free(s);
    *m_j = m;
    *e_j = e;
}

/*
 * Aggregation of b partial results [IL, 结果聚合与通信开销降低]:
 *   m_g = max_j m_j,  e_g = sum_j e_j exp(m_j - m_g),
 *   Attention = sum_j MA_j exp(m_j - m_g) / e_g.
 * MA is [b][d]. out (nullable) gets the normalised result. MA_g (nullable) gets the
 * unnormalised merged partial sum_j MA_j exp(m_j - m_g), so a merge can feed another
 * merge. When every partial is empty: m_g = -inf, e_g = 0, out = MA_g = 0 (R3).
 */
void orc_merge(int b, const double *m, const double *e, const double *MA, int d, double *m_g,
               double *e_g, double *out, double *MA_g)
{
    double mg = -INFINITY;
    for (int j = 0; j < b; ++j)
        if (m[j] > mg) mg = m[j];
    double eg = 0.0;
    double *acc = (double *)calloc((size_t)d, sizeof(double));
    if (mg != -INFINITY) {
        for (int j = 0; j < b; ++j) {
            if (m[j] == -INFINITY) continue; /* exp(-inf) = 0: an empty chunk adds nothing */
            const double w = exp(m[j] - mg);
            eg += e[j] * w;
            for (int c = 0; c < d; ++c) acc[c] += MA[(int64_t)j * d + c] * w;
        }
    }
    for (int c = 0; c < d; ++c) {
        if (out) out[c] = eg > 0.0 ? acc[c] / eg : 0.0;
        if (MA_g) MA_g[c] = acc[c];
    }
    free(acc);
    *m_g = mg;
    *e_g = eg;
}

/*
 * Paged KV write of T new tokens of one request [LS §4.2: the master saves the new
 * token's KV in its local pool]. The pool layout is [num_pages][Hkv][P][d]. Token at
 * position pos goes to page block_table_row[pos / P], slot pos % P. k_new and v_new are
 * [T][Hkv][d]. Returns the number of tokens skipped because their page was unmapped (-1),
 * beyond the table or outside the pool. Nothing is written for a skipped token.
 */
int64_t orc_kv_write(uint16_t *k_pool, uint16_t *v_pool, int Hkv, int P, int d,
                     const int32_t *block_table_row, int max_pages, int num_pages,
                     const uint16_t *k_new, const uint16_t *v_new, int64_t pos0, int64_t T)
{
    int64_t skipped = 0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t pos = pos0 + t;
        const int64_t lp = pos / P;
        if (lp >= max_pages) { ++skipped; continue; }
        const int32_t page = block_table_row[lp];
        if (page < 0 || page >= num_pages) { ++skipped; continue; }
        const int64_t slot = pos % P;
        for (int h = 0; h < Hkv; ++h) {
            const int64_t dst = (((int64_t)page * Hkv + h) * P + slot) * d;
            const int64_t src = (t * Hkv + h) * (int64_t)d;
            memcpy(k_pool + dst, k_new + src, (size_t)d * sizeof(uint16_t));
            memcpy(v_pool + dst, v_new + src, (size_t)d * sizeof(uint16_t));
        }
    }
    return skipped;
}

/*
 * k_max / k_min of the keys in a logical page [LV §3.1.2, compute_page_stats: max and min
 * over the page's tokens, per channel]. The keys are rows [t0, t1) of K (row stride
 * row_stride). Per reading R8, a strict comparison in token order keeps the first-seen
 * value on ties.
 */
void orc_logical_page_stats(const uint16_t *K, int64_t row_stride, int d, int64_t t0,
                            int64_t t1, uint16_t *kmax, uint16_t *kmin)
{
    for (int c = 0; c < d; ++c) {
        uint16_t hi = K[t0 * row_stride + c], lo = hi;
        for (int64_t t = t0 + 1; t < t1; ++t) {
            const uint16_t k = K[t * row_stride + c];
            if (bf16_to_float(k) > bf16_to_float(hi)) hi = k;
            if (bf16_to_float(k) < bf16_to_float(lo)) lo = k;
        }
        kmax[c] = hi;
        kmin[c] = lo;
    }
}

/*
 * Logical-page score, the definition (reading R4) in double:
 *   sigma = sum_d max(q_d * kmax_d, q_d * kmin_d).
 * It bounds q . k from above for every key k in the page, because kmin_d <= k_d <= kmax_d.
 */
double orc_logical_score_f64(const uint16_t *q, const uint16_t *kmax, const uint16_t *kmin, int d)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c) {
        const double qc = orc_bf16_to_double(q[c]);
        const double a = qc * orc_bf16_to_double(kmax[c]);
        const double b = qc * orc_bf16_to_double(kmin[c]);
        acc += a > b ? a : b;
    }
    return acc;
}

/*
 * Bound on the error of an fp32 evaluation of a logical-page score whose exact terms are
 * t_c = max(q_c * kmax_c, q_c * kmin_c), c < d (reading R9): d * 2^-23 * sum |t_c| plus
 * 2d * 2^-150. Each t_c is a product of two bf16 values and so exact in fp32 unless it falls
 * below the normal range; every addition of a sum of n <= 2d terms rounds by at most u = 2^-24
 * relative, in whatever order the terms are added.
 */
double orc_logical_score_bound(const uint16_t *q, const uint16_t *kmax, const uint16_t *kmin,
                               int d)
{
    double abs_sum = 0.0;
    for (int c = 0; c < d; ++c) {
        const double qc = orc_bf16_to_double(q[c]);
        const double a = qc * orc_bf16_to_double(kmax[c]);
        const double b = qc * orc_bf16_to_double(kmin[c]);
        abs_sum += fabs(a > b ? a : b);
    }
    return (double)d * ldexp(1.0, -23) * abs_sum + 2.0 * d * ldexp(1.0, -150);
}

/*
 * Physical-page scores of one request and one KV head [LV §3.1.2 score_pages: max over the
 * logical pages of a physical page], with the GQA reading R5 (max over the g query heads),
 * in fp64. Logical-page statistics are recomputed here from the token-ordered keys (rows
 * 0..L-1 of K, stride row_stride). Q holds g query vectors of d entries. score has
 * ceil(L / P) entries. If bound is not NULL, bound[p] gets the largest fp32 error bound
 * (orc_logical_score_bound) over the (logical page, head) pairs of page p: a max of values
 * each off by at most its own bound is off by at most the largest of them.
 */
void orc_page_scores(const uint16_t *Q, int g, const uint16_t *K, int64_t row_stride, int d,
                     int64_t L, int P, double *score, double *bound)
{
    const int LPG = 16; /* logical page size [LV §2.2.2: 16-token logical pages] */
    uint16_t *kmax = (uint16_t *)malloc((size_t)d * sizeof(uint16_t));
    uint16_t *kmin = (uint16_t *)malloc((size_t)d * sizeof(uint16_t));
    const int64_t npages = (L + P - 1) / P;
    for (int64_t p = 0; p < npages; ++p) {
        double best = -INFINITY, err = 0.0;
        for (int64_t t0 = p * P; t0 < (p + 1) * P && t0 < L; t0 += LPG) {
            const int64_t t1 = (t0 + LPG < L) ? t0 + LPG : L;
            orc_logical_page_stats(K, row_stride, d, t0, t1, kmax, kmin);
            for (int j = 0; j < g; ++j) {
                const double s = orc_logical_score_f64(Q + (int64_t)j * d, kmax, kmin, d);
                if (s > best) best = s;
                const double e = orc_logical_score_bound(Q + (int64_t)j * d, kmax, kmin, d);
                if (e > err) err = e;
            }
        }
        score[p] = best;
        if (bound) bound[p] = err;
    }
    free(kmax);
    free(kmin);
}

/*
 * Top-K physical pages [LV §3.1.2: keep the K highest-scoring pages] with reading R6.
 * Plain repeated selection: each round takes the highest remaining score, and the lower
 * index on ties. sel gets the chosen indices in ascending order, padded with -1 up to
 * top_k.
 */
void orc_topk(const double *score, int64_t n, int top_k, int32_t *sel)
{
    char *taken = (char *)calloc((size_t)(n > 0 ? n : 1), 1);
    int count = 0;
    for (int r = 0; r < top_k && r < n; ++r) {
        int64_t best = -1;
        for (int64_t i = 0; i < n; ++i) {
            if (taken[i]) continue;
            if (best < 0 || score[i] > score[best]) best = i; /* strict: lower index wins ties */
        }
        taken[best] = 1;
        sel[count++] = (int32_t)best;
    }
    /* ascending page order (insertion sort) */
    for (int i = 1; i < count; ++i) {
        int32_t v = sel[i];
        int j = i - 1;
        while (j >= 0 && sel[j] > v) { sel[j + 1] = sel[j]; --j; }
        sel[j + 1] = v;
    }
    for (int i = count; i < top_k; ++i) sel[i] = -1;
    free(taken);
}

/*
 * Token set one head attends in the block-sparse decode.
 *  kind 0 (dense):     every token 0..L-1.
 *  kind 1 (retrieval): the tokens < L of the selected physical pages [LV §2.2.2, §3.1.2:
 *                      only the selected pages' KV is loaded].
 *  kind 2 (streaming): [0, min(S, L)) U [max(S, L - W), L) [LV §3.1.1; reading R7].
 * rows must have room for L entries. Returns the number of rows, in ascending order.
 */
int64_t orc_sparse_rows(int kind, int64_t L, int P, const int32_t *sel, int top_k, int sinks,
                        int local, int64_t *rows)
{
    int64_t n = 0;
    if (kind == 0) {
        for (int64_t t = 0; t < L; ++t) rows[n++] = t;
    } else if (kind == 1) {
        /* visit the selected pages in ascending order; an index appears at most once */
        for (int64_t p = 0; p * P < L; ++p) {
            int chosen = 0;
            for (int i = 0; i < top_k; ++i)
                if (sel[i] == p) chosen = 1;
            if (!chosen) continue;
            for (int64_t t = p * P; t < (p + 1) * P && t < L; ++t) rows[n++] = t;
        }
    } else {
        const int64_t s_end = sinks < L ? sinks : L;
        for (int64_t t = 0; t < s_end; ++t) rows[n++] = t;
        int64_t l0 = L - local;
        if (l0 < sinks) l0 = sinks;
        for (int64_t t = l0; t < L; ++t) rows[n++] = t;
    }
    return n;
}

/*
 * Key rows that query token t of a Tq-token chunk attends in the block-sparse prefill
 * (reading R11). kind 0 dense, 1 retrieval (blocks = the key-block list of the query's
 * block, nblk entries, -1 ignored), 2 streaming (sink_blocks, local_blocks). rows must have
 * room for L entries. Returns the number of rows, in ascending order.
 */
int64_t orc_prefill_rows(int kind, int64_t L, int64_t Tq, int64_t t, int sink_blocks,
                         int local_blocks, const int32_t *blocks, int nblk, int64_t *rows)
{
    const int64_t p = L - Tq + t;
    const int64_t qb = p / 64;
    int64_t n = 0;
    for (int64_t i = 0; i <= p; ++i) {
        const int64_t kb = i / 64;
        int keep = 0;
        if (kind == 0) {
            keep = 1;
        } else if (kind == 2) {
            keep = kb < sink_blocks || kb > qb - local_blocks;
        } else {
            for (int j = 0; j < nblk; ++j)
                if (blocks[j] == kb) keep = 1;
        }
        if (keep) rows[n++] = i;
    }
    return n;
}

/* ---- 8-bit KV cache (reading R10): FP8 E4M3 codes with one fp32 scale per row ---------- */

/*
 * Value of an E4M3 code (the OCP 8-bit floating-point format: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals mantissa/8 * 2^-6;
 * there are no infinities, and S.1111.111 is NaN).
 */
double orc_e4m3_value(uint8_t code)
{
    const int sgn = code >> 7, ef = (code >> 3) & 15, mf = code & 7;
    if (ef == 15 && mf == 7) return NAN;
    const double v = ef == 0 ? ldexp((double)mf, -9) : ldexp(8.0 + mf, ef - 10);
    return sgn ? -v : v;
}

/*
 * E4M3 code of a finite float: round to the nearest representable value, ties to the even
 * mantissa, and saturate at the largest finite magnitude 448 (code 0x7E). The sign of a
 * result that rounds to zero is kept.
 */
uint8_t orc_e4m3_code(float f)
{
    const uint8_t sgn = signbit(f) ? 0x80 : 0x00;
    const double a = fabs((double)f);
    if (a == 0.0) return sgn;
    int e;
    frexp(a, &e);
    int E = e - 1; /* a = (1.mmm...) * 2^E */
    if (E < -6) {  /* subnormal range: multiples of 2^-9 */
        const int n = (int)rint(a / ldexp(1.0, -9)); /* 0 .. 8, ties to even */
        return sgn | (uint8_t)(n == 8 ? 0x08 : n);  /* 8 * 2^-9 is the smallest normal */
    }
    int n = (int)rint(a / ldexp(1.0, E - 3)); /* 8 .. 16: 1 + mantissa/8 in units of 1/8 */
    if (n == 16) {
        n = 8;
        E += 1;
    }
    if (E > 8 || (E == 8 && n > 14)) return sgn | 0x7E; /* saturate at 448 */
    return sgn | (uint8_t)(((E + 7) << 3) | (n - 8));
}

/*
 * One row of d bf16 values in the 8-bit format: scale = max_c |x_c| / 448 and
 * code_c = E4M3(x_c / scale), both divisions in IEEE fp32. A row whose scale is 0 has +0
 * codes. The row's values are code * scale.
 */
void orc_quantize_row_fp8(const uint16_t *x, int d, uint8_t *codes, float *scale)
{
    float mx = 0.0f;
    for (int c = 0; c < d; ++c) {
        const float v = fabsf(bf16_to_float(x[c]));
        if (v > mx) mx = v;
    }
    const float s = mx / 448.0f;
    *scale = s;
    for (int c = 0; c < d; ++c) codes[c] = s > 0.0f ? orc_e4m3_code(bf16_to_float(x[c]) / s) : 0;
}

/* code * scale of one row, exactly (an E4M3 value times an fp32 value fits in a double). */
void orc_dequantize_row_fp8(const uint8_t *codes, float scale, int d, double *out)
{
    for (int c = 0; c < d; ++c) out[c] = orc_e4m3_value(codes[c]) * (double)scale;
}

/* The two row functions above over n consecutive rows of d values. */
void orc_quantize_rows_fp8(const uint16_t *x, int64_t n, int d, uint8_t *codes, float *scales)
{
    for (int64_t r = 0; r < n; ++r) orc_quantize_row_fp8(x + r * d, d, codes + r * d, scales + r);
}

void orc_dequantize_rows_fp8(const uint8_t *codes, const float *scales, int64_t n, int d,
                             double *out)
{
    for (int64_t r = 0; r < n; ++r)
        orc_dequantize_row_fp8(codes + r * d, scales[r], d, out + r * d);
}

/*
 * Paged write of T new tokens in the 8-bit format [LS §4.2, with reading R10]: the codes of
 * each (token, KV head) row go to k_pool / v_pool [num_pages][Hkv][P][d] and its scale to
 * k_scale / v_scale [num_pages][Hkv][P], at the place orc_kv_write uses. Returns the number
 * of skipped tokens, as orc_kv_write does.
 */
int64_t orc_kv_write_fp8(uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                         int Hkv, int P, int d, const int32_t *block_table_row, int max_pages,
                         int num_pages, const uint16_t *k_new, const uint16_t *v_new,
                         int64_t pos0, int64_t T)
{
    int64_t skipped = 0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t pos = pos0 + t;
        const int64_t lp = pos / P;
        if (lp >= max_pages) { ++skipped; continue; }
        const int32_t page = block_table_row[lp];
        if (page < 0 || page >= num_pages) { ++skipped; continue; }
        for (int h = 0; h < Hkv; ++h) {
            const int64_t row = ((int64_t)page * Hkv + h) * P + pos % P;
            const int64_t src = (t * Hkv + h) * (int64_t)d;
            orc_quantize_row_fp8(k_new + src, d, k_pool + row * d, k_scale + row);
            orc_quantize_row_fp8(v_new + src, d, v_pool + row * d, v_scale + row);
        }
    }
    return skipped;
}

/* ---- 4-bit KV cache (reading R12): symmetric codes with one fp32 scale per row --------- */

/*
 * One row of d bf16 values (d even) in the 4-bit format: scale = max_c |x_c| / 7 and
 * code_c = x_c / scale rounded to the nearest integer (ties to even), kept in [-7, 7]; both
 * divisions in IEEE fp32. Channel c goes to byte c / 2 as the nibble code_c + 8, channel 2i
 * in the low nibble. A row whose scale is 0 has code 0 everywhere.
 */
void orc_quantize_row_int4(const uint16_t *x, int d, uint8_t *packed, float *scale)
{
    float mx = 0.0f;
    for (int c = 0; c < d; ++c) {
        const float v = fabsf(bf16_to_float(x[c]));
        if (v > mx) mx = v;
    }
    const float s = mx / 7.0f;
    *scale = s;
    for (int i = 0; i < d / 2; ++i) {
        int nib[2];
        for (int j = 0; j < 2; ++j) {
            int code = 0;
            if (s > 0.0f) {
                const float r = rintf(bf16_to_float(x[2 * i + j]) / s);
                code = r > 7.0f ? 7 : (r < -7.0f ? -7 : (int)r);
            }
            nib[j] = code + 8;
        }
        packed[i] = (uint8_t)(nib[0] | (nib[1] << 4));
    }
}

/* Value of code c of a packed 4-bit row (the nibble minus 8). */
int orc_int4_code(const uint8_t *packed, int c)
{
    const int byte = packed[c / 2];
    return ((c & 1) ? (byte >> 4) : (byte & 15)) - 8;
}

/* code * scale of one packed row, exactly (a small integer times an fp32 value). */
void orc_dequantize_row_int4(const uint8_t *packed, float scale, int d, double *out)
{
    for (int c = 0; c < d; ++c) out[c] = (double)orc_int4_code(packed, c) * (double)scale;
}

/* The two row functions above over n consecutive rows (d values, d / 2 bytes each). */
void orc_quantize_rows_int4(const uint16_t *x, int64_t n, int d, uint8_t *packed, float *scales)
{
    for (int64_t r = 0; r < n; ++r)
        orc_quantize_row_int4(x + r * d, d, packed + r * (d / 2), scales + r);
}

void orc_dequantize_rows_int4(const uint8_t *packed, const float *scales, int64_t n, int d,
                              double *out)
{
    for (int64_t r = 0; r < n; ++r)
        orc_dequantize_row_int4(packed + r * (d / 2), scales[r], d, out + r * d);
}

/*
 * Paged write of T new tokens in the 4-bit format [LS §4.2, with reading R12]: the packed
 * codes of each (token, KV head) row go to k_pool / v_pool [num_pages][Hkv][P][d / 2] and its
 * scale to k_scale / v_scale [num_pages][Hkv][P], at the place orc_kv_write uses. Returns
 * the number of skipped tokens, as orc_kv_write does.
 */
int64_t orc_kv_write_int4(uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                          int Hkv, int P, int d, const int32_t *block_table_row, int max_pages,
                          int num_pages, const uint16_t *k_new, const uint16_t *v_new,
                          int64_t pos0, int64_t T)
{
    int64_t skipped = 0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t pos = pos0 + t;
        const int64_t lp = pos / P;
        if (lp >= max_pages) { ++skipped; continue; }
        const int32_t page = block_table_row[lp];
        if (page < 0 || page >= num_pages) { ++skipped; continue; }
        for (int h = 0; h < Hkv; ++h) {
            const int64_t row = ((int64_t)page * Hkv + h) * P + pos % P;
            const int64_t src = (t * Hkv + h) * (int64_t)d;
            orc_quantize_row_int4(k_new + src, d, k_pool + row * (d / 2), k_scale + row);
            orc_quantize_row_int4(v_new + src, d, v_pool + row * (d / 2), v_scale + row);
        }
    }
    return skipped;
}

/*
 * orc_attention and orc_partial over keys and values given as doubles (row r of K and V
 * starts at K + r * row_stride): the same equations, for the dequantized 8-bit format.
 */
static double logit_f64(const uint16_t *q, const double *k, int d, double scale)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += orc_bf16_to_double(q[c]) * k[c];
    return scale * acc;
}

void orc_attention_f64(const uint16_t *q, const double *K, const double *V, int64_t row_stride,
                       int d, const int64_t *rows, int64_t n, double scale, double *out,
                       double *m_out, double *e_out)
{
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (n <= 0) {
        *m_out = -INFINITY;
        *e_out = 0.0;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        s[i] = logit_f64(q, K + row_of(rows, i) * row_stride, d, scale);
        if (s[i] > m) m = s[i];
    }
    double e = 0.0;
    for (int64_t i = 0; i < n; ++i) e += exp(s[i] - m);
    for (int64_t i = 0; i < n; ++i) {
        const double w = exp(s[i] - m) / e;
        const double *v = V + row_of(rows, i) * row_stride;
        for (int c = 0; c < d; ++c) out[c] += w * v[c];
    }
    free(s);
    *m_out = m;
    *e_out = e;
}

void orc_partial_f64(const uint16_t *q, const double *K, const double *V, int64_t row_stride,
                     int d, const int64_t *rows, int64_t n, double scale, double *m_j,
                     double *e_j, double *MA_j)
{
    for (int c = 0; c < d; ++c) MA_j[c] = 0.0;
    if (n <= 0) {
        *m_j = -INFINITY;
        *e_j = 0.0;
        return;
    }
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        s[i] = logit_f64(q, K + row_of(rows, i) * row_stride, d, scale);
        if (s[i] > m) m = s[i];
    }
    double e = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double w = exp(s[i] - m);
        const double *v = V + row_of(rows, i) * row_stride;
        e += w;
        for (int c = 0; c < d; ++c) MA_j[c] += w * v[c];
    }
    free(s);
    *m_j = m;
    *e_j = e;
}

/* ---- batch driver: plain attention over many (request, head) pairs on host threads ---- */

typedef struct {
    const uint16_t *q;      /* [B][Hq][d] */
    const uint16_t *K, *V;  /* token-ordered, [sum L][Hkv][d] */
    const int64_t *offs;    /* [B+1] token offsets of each request */
    const int32_t *pairs;   /* [npairs][2] = (b, h) */
    int64_t npairs;
    int Hq, Hkv, d;
    double scale;
    double *out, *m, *e;    /* [npairs][d], [npairs], [npairs] */
    int64_t next;
    pthread_mutex_t lock;
} batch_job;

static void *batch_worker(void *arg)
{
    batch_job *job = (batch_job *)arg;
    const int g = job->Hq / job->Hkv;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        const int64_t i = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (i >= job->npairs) break;
        const int b = job->pairs[2 * i], h = job->pairs[2 * i + 1];
        const int kvh = h / g; /* reading R2 */
        const int64_t stride = (int64_t)job->Hkv * job->d;
        const uint16_t *Kb = job->K + job->offs[b] * stride + (int64_t)kvh * job->d;
        const uint16_t *Vb = job->V + job->offs[b] * stride + (int64_t)kvh * job->d;
        const uint16_t *qh = job->q + ((int64_t)b * job->Hq + h) * job->d;
        orc_attention(qh, Kb, Vb, stride, job->d, NULL, job->offs[b + 1] - job->offs[b],
                      job->scale, job->out + i * job->d, job->m + i, job->e + i);
    }
    return NULL;
}

/*
 * Dense decode attention for a list of (request, query head) pairs, spread over nthreads
 * host threads. Each pair is an independent orc_attention call over all of that
 * request's tokens. Returns the number of threads used.
 */
int orc_attention_pairs_mt(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                           const int64_t *offs, int Hq, int Hkv, int d, double scale,
                           const int32_t *pairs, int64_t npairs, int nthreads, double *out,
                           double *m, double *e)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    batch_job job = {q, K, V, offs, pairs, npairs, Hq, Hkv, d, scale, out, m, e, 0,
                     PTHREAD_MUTEX_INITIALIZER};
    pthread_t *th = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, batch_worker, &job);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    return nthreads;
}
