/*
 * dattn oracle: TEST INFRASTRUCTURE ONLY. This header belongs to the oracle alone; the CUDA
 * library neither includes it nor shares anything with it. Each function is documented at
 * its definition in dattn_oracle.c, with the passage it follows.
 */
#ifndef DATTN_ORACLE_H
#define DATTN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double orc_bf16_to_double(uint16_t h);

void orc_attention(const uint16_t *q, const uint16_t *K, const uint16_t *V, int64_t row_stride,
                   int d, const int64_t *rows, int64_t n, double scale, double *out,
                   double *m_out, double *e_out);

void orc_partial(const uint16_t *q, const uint16_t *K, const uint16_t *V, int64_t row_stride,
                 int d, const int64_t *rows, int64_t n, double scale, double *m_j, double *e_j,
                 double *MA_j);

void orc_merge(int b, const double *m, const double *e, const double *MA, int d, double *m_g,
               double *e_g, double *out, double *MA_g);

int64_t orc_kv_write(uint16_t *k_pool, uint16_t *v_pool, int Hkv, int P, int d,
                     const int32_t *block_table_row, int max_pages, int num_pages,
                     const uint16_t *k_new, const uint16_t *v_new, int64_t pos0, int64_t T);

void orc_logical_page_stats(const uint16_t *K, int64_t row_stride, int d, int64_t t0,
                            int64_t t1, uint16_t *kmax, uint16_t *kmin);

double orc_logical_score_f64(const uint16_t *q, const uint16_t *kmax, const uint16_t *kmin, int d);

double orc_logical_score_bound(const uint16_t *q, const uint16_t *kmax, const uint16_t *kmin,
                               int d);

void orc_page_scores(const uint16_t *Q, int g, const uint16_t *K, int64_t row_stride, int d,
                     int64_t L, int P, double *score, double *bound);

void orc_topk(const double *score, int64_t n, int top_k, int32_t *sel);

int64_t orc_sparse_rows(int kind, int64_t L, int P, const int32_t *sel, int top_k, int sinks,
                        int local, int64_t *rows);
int64_t orc_prefill_rows(int kind, int64_t L, int64_t Tq, int64_t t, int sink_blocks,
                         int local_blocks, const int32_t *blocks, int nblk, int64_t *rows);

double orc_e4m3_value(uint8_t code);

uint8_t orc_e4m3_code(float f);

void orc_quantize_row_fp8(const uint16_t *x, int d, uint8_t *codes, float *scale);

void orc_dequantize_row_fp8(const uint8_t *codes, float scale, int d, double *out);
void orc_quantize_rows_fp8(const uint16_t *x, int64_t n, int d, uint8_t *codes, float *scales);
void orc_dequantize_rows_fp8(const uint8_t *codes, const float *scales, int64_t n, int d,
                             double *out);

int64_t orc_kv_write_fp8(uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                         int Hkv, int P, int d, const int32_t *block_table_row, int max_pages,
                         int num_pages, const uint16_t *k_new, const uint16_t *v_new,
                         int64_t pos0, int64_t T);

/* 4-bit KV cache (reading R12) */
void orc_quantize_row_int4(const uint16_t *x, int d, uint8_t *packed, float *scale);
int orc_int4_code(const uint8_t *packed, int c);
void orc_dequantize_row_int4(const uint8_t *packed, float scale, int d, double *out);
void orc_quantize_rows_int4(const uint16_t *x, int64_t n, int d, uint8_t *packed, float *scales);
void orc_dequantize_rows_int4(const uint8_t *packed, const float *scales, int64_t n, int d,
                              double *out);
int64_t orc_kv_write_int4(uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                          int Hkv, int P, int d, const int32_t *block_table_row, int max_pages,
                          int num_pages, const uint16_t *k_new, const uint16_t *v_new,
                          int64_t pos0, int64_t T);

void orc_attention_f64(const uint16_t *q, const double *K, const double *V, int64_t row_stride,
                       int d, const int64_t *rows, int64_t n, double scale, double *out,
                       double *m_out, double *e_out);

void orc_partial_f64(const uint16_t *q, const double *K, const double *V, int64_t row_stride,
                     int d, const int64_t *rows, int64_t n, double scale, double *m_j,
                     double *e_j, double *MA_j);

int orc_attention_pairs_mt(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                           const int64_t *offs, int Hq, int Hkv, int d, double scale,
                           const int32_t *pairs, int64_t npairs, int nthreads, double *out,
                           double *m, double *e);

#ifdef __cplusplus
}
#endif

#endif /* DATTN_ORACLE_H */
