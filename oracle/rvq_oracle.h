/*
 * CPU oracle for the RVQ Mixture-of-Experts expert FFN (test infrastructure).
 * Declarations only; see rvq_oracle.c for the definitions and their sources.
 * Parity unpinned: none (every function is pinned by the CPU test suite).
 */
#ifndef RVQ_ORACLE_H
#define RVQ_ORACLE_H
#include <stddef.h>
#include <stdint.h>

void oracle_rvq_dequant_row(const uint8_t *codes, const float *cb, int32_t cols,
                            int32_t row, double *w_row);
void oracle_rvq_dequant(const uint8_t *codes, const float *cb, int32_t rows,
                        int32_t cols, double *w);
void oracle_rvq_gemv(const uint8_t *codes, const float *cb, int32_t rows, int32_t cols,
                     const double *x, int32_t n, double *y);
void oracle_rvq_lut_build(const float *cb, const double *x, int32_t cols, double *lut);
void oracle_rvq_lut_gemv(const uint8_t *codes, const double *lut, int32_t rows,
                         int32_t cols, double *y);
void oracle_router_logits(const float *wr, const float *bias, const double *x,
                          int32_t n, int32_t E, int32_t d, double *logits);
int32_t oracle_route(const float *logits, int32_t n, int32_t E, int32_t k,
                     int32_t *topk_idx, float *topk_w);
void oracle_group(const int32_t *topk_idx, int32_t n, int32_t E, int32_t k,
                  int32_t *offsets, int32_t *pairs);
double oracle_swiglu(double g, double u);
void oracle_expert_ffn(const uint8_t *gate_codes, const float *gate_cb,
                       const uint8_t *up_codes, const float *up_cb,
                       const uint8_t *down_codes, const float *down_cb,
                       int32_t d, int32_t f, const double *x, double *y, double *h_out);
void oracle_combine(const double *y_pair, const float *topk_w, int32_t n, int32_t k,
                    int32_t d, const double *residual, double *out);
void oracle_rms_norm(const double *x, int32_t n, int32_t d, double eps, double *out);
int32_t oracle_moe_layer(const uint8_t *const *codes, const float *const *cbs,
                         const float *wr, const float *bias,
                         int32_t n, int32_t E, int32_t k, int32_t d, int32_t f,
                         const double *x, const float *route_logits,
                         float *logits_used, int32_t *topk_idx, float *topk_w,
                         double *y_pair, double *out);
uint32_t oracle_crc32(const uint8_t *p, size_t n);
void oracle_rvq_encode(const float *w, int32_t rows, int32_t cols, int32_t iters,
                       uint8_t *codes, float *codebooks);
#endif
