/*
 * CPU oracle for the RVQ Mixture-of-Experts expert FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline / reference leg may load this library.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Plain C11, libc + libm, double precision throughout (one exception: the
 * offline encoder, oracle_rvq_encode, takes its distances in fp32 fused
 * multiply-adds and its means as int64 fixed-point sums, the reproducible
 * steps its codes are compared bit for bit against), no blocking, no
 * fusion: each function is the plain definition of one step, written so it
 * can be checked against the source pages by eye.  Sources (web pages on the
 * WASTE inference engine):
 *   [AL]  "WASTE Inference Engine: Running Kimi K3 2.78T on Consumer Hardware"
 *         (agentlenshq.com), section "Residual Vector Quantization (RVQ)".
 *   [SL]  "Running a 2.78-Trillion-Parameter Model on a Laptop: Inside WASTE's
 *         NVMe-Streaming Engine" (starlog.pages.dev), section "Technical Insight".
 *   [GN]  GeekNews topic 32035 (news.hada.io), sections "Quantization and
 *         accuracy" (양자화와 정확성) and "Read-ahead and router prediction"
 *         (읽기 선행과 라우터 예측); its German edition (de.news.hada.io),
 *         "Quantisierung und Genauigkeit".
 *
 * What the pages fix: expert weights are coded by 3-stage residual vector
 * quantisation of 8-dimensional sub-vectors with 256-entry codebooks (3.00
 * bits per weight) [GN, Quantization; AL, RVQ]; the residual decode of a
 * sub-vector is the sum of its three stage codewords [AL, RVQ]; an expert is
 * gate, up and down projection matrices [SL, Technical Insight]; the router
 * picks 16 experts per layer [GN, Read-ahead].  Readings where the pages are
 * silent (sub-vectors run along the input dimension; one codebook set per
 * matrix; softmax renormalised over the selected experts, ties to the lower
 * index; SwiGLU activation; weighted combine plus residual) are listed with
 * the design notes and stated again at each function.
 *
 * Layouts used here (the oracle's own, plain ones):
 *   codes      uint8  [rows][cols/8][3]   code of (row, chunk j, stage s)
 *   codebooks  float  [3][256][8]         stage s, entry k, dimension i
 *   weight row r, column 8j+i = C0[c(r,j,0)][i] + C1[c(r,j,1)][i] + C2[c(r,j,2)][i]
 */
#include "rvq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ RVQ */

/* Residual decode of one weight row (reading: sub-vectors lie along the
 * input dimension, so a row of cols weights is cols/8 sub-vectors).  Each
 * sub-vector is the sum of the three stage codewords [AL, RVQ; GN,
 * Quantization]. */
void oracle_rvq_dequant_row(const uint8_t *codes, const float *cb, int32_t cols,
                            int32_t row, double *w_row)
{
    const int32_t chunks = cols / 8;
    const uint8_t *c = codes + (size_t)row * chunks * 3;
    for (int32_t j = 0; j < chunks; ++j) {
        for (int32_t i = 0; i < 8; ++i) {
            double w = 0.0;
            for (int32_t s = 0; s < 3; ++s) {
                uint8_t k = c[j * 3 + s];
                w += (double)cb[((size_t)s * 256 + k) * 8 + i];
            }
            w_row[j * 8 + i] = w;
        }
    }
}

void oracle_rvq_dequant(const uint8_t *codes, const float *cb, int32_t rows,
                        int32_t cols, double *w)
{
    for (int32_t r = 0; r < rows; ++r)
        oracle_rvq_dequant_row(codes, cb, cols, r, w + (size_t)r * cols);
}

/* y[t][r] = sum_c W[r][c] * x[t][c], W the dequantised matrix: the explicit
 * dequantise-then-multiply definition that the lookup-table method reaches
 * without materialising W [SL, Technical Insight]. */
void oracle_rvq_gemv(const uint8_t *codes, const float *cb, int32_t rows, int32_t cols,
                     const double *x, int32_t n, double *y)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)cols);
    for (int32_t r = 0; r < rows; ++r) {
        oracle_rvq_dequant_row(codes, cb, cols, r, w);
        for (int32_t t = 0; t < n; ++t) {
            const double *xt = x + (size_t)t * cols;
            double acc = 0.0;
            for (int32_t c = 0; c < cols; ++c) acc += w[c] * xt[c];
            y[(size_t)t * rows + r] = acc;
        }
    }
    free(w);
}

/* Partial-dot lookup table "per codebook and position" [SL, Technical
 * Insight; GN, Quantization]: lut[j][s][k] = <x[8j .. 8j+7], C_s[k]>. */
void oracle_rvq_lut_build(const float *cb, const double *x, int32_t cols, double *lut)
{
    const int32_t chunks = cols / 8;
    for (int32_t j = 0; j < chunks; ++j)
        for (int32_t s = 0; s < 3; ++s)
            for (int32_t k = 0; k < 256; ++k) {
                double acc = 0.0;
                for (int32_t i = 0; i < 8; ++i)
                    acc += x[j * 8 + i] * (double)cb[((size_t)s * 256 + k) * 8 + i];
                lut[((size_t)j * 3 + s) * 256 + k] = acc;
            }
}

/* The lookup-table evaluation of one matrix: for each row, per chunk three
 * table reads and two additions, summed over chunks [AL, RVQ; GN,
 * Quantization].  Used to cross-check the explicit definition above. */
void oracle_rvq_lut_gemv(const uint8_t *codes, const double *lut, int32_t rows,
                         int32_t cols, double *y)
{
    const int32_t chunks = cols / 8;
    for (int32_t r = 0; r < rows; ++r) {
        const uint8_t *c = codes + (size_t)r * chunks * 3;
        double acc = 0.0;
        for (int32_t j = 0; j < chunks; ++j) {
            const double *t = lut + (size_t)j * 3 * 256;
            double row_chunk = t[c[j * 3 + 0]] + t[256 + c[j * 3 + 1]];
            row_chunk += t[512 + c[j * 3 + 2]];
            acc += row_chunk;
        }
        y[r] = acc;
    }
}

/* ---------------------------------------------------------------- router */

/* logits[t][e] = sum_c Wr[e][c] x[t][c] (+ bias[e]).  The pages only say a
 * resident router picks the experts [GN, Read-ahead]; a linear router over
 * the hidden state is the reading taken here. */
void oracle_router_logits(const float *wr, const float *bias, const double *x,
                          int32_t n, int32_t E, int32_t d, double *logits)
{
    for (int32_t t = 0; t < n; ++t)
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t c = 0; c < d; ++c)
                acc += (double)wr[(size_t)e * d + c] * x[(size_t)t * d + c];
            if (bias) acc += (double)bias[e];
            logits[(size_t)t * E + e] = acc;
        }
}

/* Strict order used for selection: larger logit first, equal logits by the
 * lower expert index (reading: the pages give no tie rule).  The row being
 * sorted is per thread, so concurrent calls (a thread pool in the tests and
 * the benchmark's baseline) do not share it. */
static _Thread_local const float *g_sort_row;
static int cmp_expert(const void *a, const void *b)
{
    int32_t ia = *(const int32_t *)a, ib = *(const int32_t *)b;
    float la = g_sort_row[ia], lb = g_sort_row[ib];
    if (la > lb) return -1;
    if (la < lb) return 1;
    return (ia < ib) ? -1 : (ia > ib);
}

/* Top-k selection and weights.  The router picks k expert IDs per token
 * (k = 16 for K3) [GN, Read-ahead]; no low-probability expert is dropped
 * [SL, Technical Insight].  Reading: the k largest fp32 logits in the order
 * above, weights softmax(logits) renormalised over the selected k, i.e.
 * w_i = exp(l_i - l_max) / sum_sel exp(l_j - l_max), computed in double and
 * stored as fp32.  Output slots are in selection order.  Returns 0, or -1 if
 * a logit is not finite. */
int32_t oracle_route(const float *logits, int32_t n, int32_t E, int32_t k,
                     int32_t *topk_idx, float *topk_w)
{
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t bad = 0;
    for (int32_t t = 0; t < n; ++t) {
        const float *row = logits + (size_t)t * E;
        for (int32_t e = 0; e < E; ++e) {
            order[e] = e;
            if (!isfinite(row[e])) bad = 1;
        }
        g_sort_row = row;
        qsort(order, (size_t)E, sizeof(int32_t), cmp_expert);
        double lmax = (double)row[order[0]];
        double denom = 0.0;
        for (int32_t i = 0; i < k; ++i) denom += exp((double)row[order[i]] - lmax);
        for (int32_t i = 0; i < k; ++i) {
            topk_idx[(size_t)t * k + i] = order[i];
            topk_w[(size_t)t * k + i] = (float)(exp((double)row[order[i]] - lmax) / denom);
        }
    }
    free(order);
    return bad ? -1 : 0;
}

/* Token-to-expert grouping (reading: a counting sort by expert, stable in
 * token order, which is what a chunked prefill that visits each selected
 * expert once needs).  offsets[e] .. offsets[e+1] is expert e's segment of
 * pairs; each entry is t * k + slot. */
void oracle_group(const int32_t *topk_idx, int32_t n, int32_t E, int32_t k,
                  int32_t *offsets, int32_t *pairs)
{
    int32_t *fill = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    for (int32_t e = 0; e <= E; ++e) offsets[e] = 0;
    for (int32_t p = 0; p < n * k; ++p) offsets[topk_idx[p] + 1] += 1;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    for (int32_t t = 0; t < n; ++t)
        for (int32_t s = 0; s < k; ++s) {
            int32_t e = topk_idx[(size_t)t * k + s];
            pairs[offsets[e] + fill[e]] = t * k + s;
            fill[e] += 1;
        }
    free(fill);
}

/* ----------------------------------------------------------- expert FFN */

/* SwiGLU gate: silu(g) * u with silu(g) = g / (1 + exp(-g)) (reading: the
 * pages name gate and up projections but not the activation). */
double oracle_swiglu(double g, double u) { return g / (1.0 + exp(-g)) * u; }

/* One expert on one token: g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h
 * [SL, Technical Insight: an expert is gate, up and down projection
 * matrices].  Shapes: Wg, Wu are [f][d]; Wd is [d][f]. */
void oracle_expert_ffn(const uint8_t *gate_codes, const float *gate_cb,
                       const uint8_t *up_codes, const float *up_cb,
                       const uint8_t *down_codes, const float *down_cb,
                       int32_t d, int32_t f, const double *x, double *y, double *h_out)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)f);
    double *u = (double *)malloc(sizeof(double) * (size_t)f);
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    oracle_rvq_gemv(gate_codes, gate_cb, f, d, x, 1, g);
    oracle_rvq_gemv(up_codes, up_cb, f, d, x, 1, u);
    for (int32_t r = 0; r < f; ++r) h[r] = oracle_swiglu(g[r], u[r]);
    oracle_rvq_gemv(down_codes, down_cb, d, f, h, 1, y);
    if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)f);
    free(g);
    free(u);
    free(h);
}

/* Weighted combine plus residual (reading: the standard MoE output,
 * out[t] = residual[t] + sum_slot w[t][slot] * y[t*k + slot]). */
void oracle_combine(const double *y_pair, const float *topk_w, int32_t n, int32_t k,
                    int32_t d, const double *residual, double *out)
{
    for (int32_t t = 0; t < n; ++t)
        for (int32_t c = 0; c < d; ++c) {
            double acc = residual[(size_t)t * d + c];
            for (int32_t s = 0; s < k; ++s)
                acc += (double)topk_w[(size_t)t * k + s] * y_pair[((size_t)t * k + s) * d + c];
            out[(size_t)t * d + c] = acc;
        }
}

/* Parameter-free RMS normalisation of each row (reading: the pages describe
 * no normalisation; a stack of their layers applies this before each layer,
 * as pre-norm transformer blocks do, and keeps the un-normalised stream as
 * the residual):  out[t][c] = x[t][c] / sqrt(mean_c x[t][c]^2 + eps). */
void oracle_rms_norm(const double *x, int32_t n, int32_t d, double eps, double *out)
{
    for (int32_t t = 0; t < n; ++t) {
        const double *r = x + (size_t)t * d;
        double ss = 0.0;
        for (int32_t c = 0; c < d; ++c) ss += r[c] * r[c];
        const double inv = 1.0 / sqrt(ss / (double)d + eps);
        for (int32_t c = 0; c < d; ++c) out[(size_t)t * d + c] = r[c] * inv;
    }
}

/* One MoE layer on n tokens, given each expert's three matrices through
 * pointer tables (entries of unselected experts may be NULL).  Routing uses
 * the fp32 logits passed in (route_logits); when that is NULL the oracle's own
 * logits, rounded to fp32, are used.  Outputs the fp32-rounded logits the
 * routing saw, the selection, and out = x + sum_slot w * expert(x). */
int32_t oracle_moe_layer(const uint8_t *const *codes, const float *const *cbs,
                         const float *wr, const float *bias,
                         int32_t n, int32_t E, int32_t k, int32_t d, int32_t f,
                         const double *x, const float *route_logits,
                         float *logits_used, int32_t *topk_idx, float *topk_w,
                         double *y_pair, double *out)
{
    double *lg = (double *)malloc(sizeof(double) * (size_t)n * E);
    oracle_router_logits(wr, bias, x, n, E, d, lg);
    for (size_t i = 0; i < (size_t)n * E; ++i)
        logits_used[i] = route_logits ? route_logits[i] : (float)lg[i];
    free(lg);
    int32_t rc = oracle_route(logits_used, n, E, k, topk_idx, topk_w);
    for (int32_t t = 0; t < n; ++t)
        for (int32_t s = 0; s < k; ++s) {
            int32_t e = topk_idx[(size_t)t * k + s];
            const uint8_t *const *ce = codes + (size_t)e * 3;
            const float *const *be = cbs + (size_t)e * 3;
            oracle_expert_ffn(ce[0], be[0], ce[1], be[1], ce[2], be[2], d, f,
                              x + (size_t)t * d, y_pair + ((size_t)t * k + s) * d, NULL);
        }
    oracle_combine(y_pair, topk_w, n, k, d, x, out);
    return rc;
}

/* CRC-32 of n bytes: the checksum the pages offer as an opt-in check of each
 * expert record's payload [GN, "Disk streaming structure"].  The pages do not
 * name the variant; this is the common CRC-32 (ISO-HDLC / IEEE 802.3):
 * reflected polynomial 0xEDB88320, register preset to all ones, bytes taken
 * least significant bit first, result complemented.  One bit per step. */
uint32_t oracle_crc32(const uint8_t *p, size_t n)
{
    uint32_t crc = 0xFFFFFFFFu;
    for (size_t i = 0; i < n; ++i) {
        crc ^= p[i];
        for (int b = 0; b < 8; ++b)
            crc = (crc & 1u) ? (crc >> 1) ^ 0xEDB88320u : crc >> 1;
    }
    return ~crc;
}

/* Offline RVQ encoder: residual k-means, one stage at a time, the pages'
 * conversion step (their converter encodes every expert matrix once, offline
 * [GN, "Conversion"]) for matrices given as fp32 weights.  The pages give no
 * algorithm; this is the plainest residual quantiser:
 *  - sub-vector i = W[r][8j .. 8j+7], i = r * (cols / 8) + j; R = W;
 *  - per stage s: codebook C[k] = R[floor(k * N / 256)] for k < 256, then
 *    `iters` rounds of (assign every sub-vector to its nearest codeword,
 *    ties to the lower index; replace each codeword that has members by
 *    their mean); a last assignment gives the stage's codes; R -= C[code].
 * Distances are taken in fp32 as d = fma(t, t, d) over the 8 dimensions in
 * order, t = r - c (the decision that sets an integer code is made in the
 * precision the device uses).  A mean is the members' sum in int64 fixed
 * point (each value times 2^32, rounded to nearest even), times 2^-32,
 * divided by the member count in double and rounded to fp32: the sum does
 * not depend on the order of the additions.  |W| < 1024 keeps every sum in
 * range.  codes: [rows][cols/8][3]; codebooks: [3][256][8]. */
static int32_t oracle_nearest(const float *r, const float *cb)
{
    int32_t best = 0;
    float bd = 0.f;
    for (int32_t k = 0; k < 256; ++k) {
        float d = 0.f;
        for (int i = 0; i < 8; ++i) {
            float t = r[i] - cb[k * 8 + i];
            d = fmaf(t, t, d);
        }
        if (k == 0 || d < bd) {
            bd = d;
            best = k;
        }
    }
    return best;
}

void oracle_rvq_encode(const float *w, int32_t rows, int32_t cols, int32_t iters,
                       uint8_t *codes, float *codebooks)
{
    const size_t N = (size_t)rows * (cols / 8);
    float *R = (float *)malloc(sizeof(float) * N * 8);
    int32_t *a = (int32_t *)malloc(sizeof(int32_t) * N);
    memcpy(R, w, sizeof(float) * N * 8);
    for (int s = 0; s < 3; ++s) {
        float *C = codebooks + (size_t)s * 256 * 8;
        for (int32_t k = 0; k < 256; ++k)
            memcpy(C + k * 8, R + ((size_t)k * N / 256) * 8, sizeof(float) * 8);
        for (int32_t it = 0; it <= iters; ++it) {
            for (size_t i = 0; i < N; ++i) a[i] = oracle_nearest(R + i * 8, C);
            if (it == iters) break;
            long long sum[256][8];
            long long cnt[256];
            memset(sum, 0, sizeof(sum));
            memset(cnt, 0, sizeof(cnt));
            for (size_t i = 0; i < N; ++i) {
                ++cnt[a[i]];
                for (int d = 0; d < 8; ++d)
                    sum[a[i]][d] += llrint((double)R[i * 8 + d] * 4294967296.0);
            }
            for (int32_t k = 0; k < 256; ++k)
                if (cnt[k] > 0)
                    for (int d = 0; d < 8; ++d)
                        C[k * 8 + d] = (float)(((double)sum[k][d] * (1.0 / 4294967296.0)) /
                                               (double)cnt[k]);
        }
        for (size_t i = 0; i < N; ++i) {
            codes[i * 3 + s] = (uint8_t)a[i];
            for (int d = 0; d < 8; ++d) R[i * 8 + d] -= C[a[i] * 8 + d];
        }
    }
    free(R);
    free(a);
}
