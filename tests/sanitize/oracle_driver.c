/*
 * Runs every oracle function on small seeded inputs under AddressSanitizer
 * and UndefinedBehaviorSanitizer (built and run by tests/test_sanitizers.py).
 * Besides the sanitizers' own checks, two consistency checks keep the run
 * meaningful: the table formulation of the GEMV equals the explicit decode
 * within 1e-12 (relative), and the grouping lists every (token, slot) once.
 * Exit status 0: clean.
 */
#include <math.h>
#include <stdio.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "rvq_oracle.h"

static uint64_t state = 0x5EEDu;
static uint64_t next_u64(void)
{
    /* xorshift64*: test-input randomness only */
    state ^= state >> 12;
    state ^= state << 25;
    state ^= state >> 27;
    return state * 0x2545F4914F6CDD1DULL;
}
static double uniform(void) { return (double)(next_u64() >> 11) / 9007199254740992.0 * 2.0 - 1.0; }

static void *xmalloc(size_t n)
{
    void *p = malloc(n ? n : 1);
    if (!p) { fprintf(stderr, "out of memory\n"); exit(2); }
    return p;
}

int main(void)
{
    const int32_t rows = 16, cols = 64, d = 64, f = 32, E = 6, k = 2, n = 3;
    int bad = 0;
    /* matrices: codes [rows][cols/8][3], codebooks [3][256][8] */
    uint8_t *codes = xmalloc((size_t)rows * cols / 8 * 3);
    float *cb = xmalloc(sizeof(float) * 3 * 256 * 8);
    for (size_t i = 0; i < (size_t)rows * cols / 8 * 3; ++i) codes[i] = (uint8_t)(next_u64() >> 56);
    for (int i = 0; i < 3 * 256 * 8; ++i) cb[i] = (float)(0.02 * uniform());
    double *x = xmalloc(sizeof(double) * n * cols), *y = xmalloc(sizeof(double) * n * rows);
    for (int i = 0; i < n * cols; ++i) x[i] = uniform();
    double *w = xmalloc(sizeof(double) * rows * cols);
    oracle_rvq_dequant(codes, cb, rows, cols, w);
    oracle_rvq_gemv(codes, cb, rows, cols, x, n, y);
    double *lut = xmalloc(sizeof(double) * (cols / 8) * 3 * 256), y2[16];
    oracle_rvq_lut_build(cb, x, cols, lut);
    oracle_rvq_lut_gemv(codes, lut, rows, cols, y2);
    for (int r = 0; r < rows; ++r)
        if (fabs(y2[r] - y[r]) > 1e-12 * (fabs(y[r]) + 1e-30) + 1e-15) bad |= 1;
    double wr0[64];
    oracle_rvq_dequant_row(codes, cb, cols, 3, wr0);
    /* router, routing, grouping */
    float *wr = xmalloc(sizeof(float) * E * d), bias[6];
    for (int i = 0; i < E * d; ++i) wr[i] = (float)(0.02 * uniform());
    for (int e = 0; e < E; ++e) bias[e] = (float)(-0.1 * e);
    double *xd = xmalloc(sizeof(double) * n * d), *lg = xmalloc(sizeof(double) * n * E);
    for (int i = 0; i < n * d; ++i) xd[i] = uniform();
    oracle_router_logits(wr, bias, xd, n, E, d, lg);
    float *lgf = xmalloc(sizeof(float) * n * E), *tw = xmalloc(sizeof(float) * n * k);
    for (int i = 0; i < n * E; ++i) lgf[i] = (float)lg[i];
    int32_t *ti = xmalloc(sizeof(int32_t) * n * k), *off = xmalloc(sizeof(int32_t) * (E + 1));
    int32_t *pairs = xmalloc(sizeof(int32_t) * n * k);
    if (oracle_route(lgf, n, E, k, ti, tw) != 0) bad |= 2;
    oracle_group(ti, n, E, k, off, pairs);
    int seen[6] = {0};
    for (int p = 0; p < n * k; ++p) seen[pairs[p]] += 1;
    for (int p = 0; p < n * k; ++p) if (seen[p] != 1) bad |= 4;
    (void)oracle_swiglu(0.5, -1.25);
    /* experts: gate/up [f][d], down [d][f] */
    uint8_t *ec[18];
    float *eb[18];
    for (int m = 0; m < 3 * E; ++m) {
        const size_t nb = (size_t)d * f / 8 * 3;
        ec[m] = xmalloc(nb);
        for (size_t i = 0; i < nb; ++i) ec[m][i] = (uint8_t)(next_u64() >> 56);
        eb[m] = xmalloc(sizeof(float) * 3 * 256 * 8);
        for (int i = 0; i < 3 * 256 * 8; ++i) eb[m][i] = (float)(0.02 * uniform());
    }
    double *yp = xmalloc(sizeof(double) * n * k * d), *h = xmalloc(sizeof(double) * f);
    oracle_expert_ffn(ec[0], eb[0], ec[1], eb[1], ec[2], eb[2], d, f, xd, yp, h);
    double *out = xmalloc(sizeof(double) * n * d);
    float *lused = xmalloc(sizeof(float) * n * E);
    if (oracle_moe_layer((const uint8_t *const *)ec, (const float *const *)eb, wr, bias, n, E, k,
                         d, f, xd, NULL, lused, ti, tw, yp, out) != 0)
        bad |= 8;
    oracle_combine(yp, tw, n, k, d, xd, out);
    double *nx = xmalloc(sizeof(double) * n * d);
    oracle_rms_norm(xd, n, d, 1e-6, nx);
    uint8_t msg[9] = {'1', '2', '3', '4', '5', '6', '7', '8', '9'};
    if (oracle_crc32(msg, 9) != 0xCBF43926u) bad |= 16;
    (void)oracle_crc32(NULL, 0);
    /* encoder on a small matrix (N = rows * cols / 8 = 256 sub-vectors) */
    const int32_t er = 32, ecl = 64;
    float *ew = xmalloc(sizeof(float) * er * ecl), *ecb = xmalloc(sizeof(float) * 3 * 256 * 8);
    uint8_t *eco = xmalloc((size_t)er * ecl / 8 * 3);
    for (int i = 0; i < er * ecl; ++i) ew[i] = (float)(0.02 * uniform());
    oracle_rvq_encode(ew, er, ecl, 2, eco, ecb);
    /* every allocation is released so the leak checker has nothing to report */
    free(codes); free(cb); free(x); free(y); free(w); free(lut); free(wr); free(xd); free(lg);
    free(lgf); free(tw); free(ti); free(off); free(pairs);
    for (int m = 0; m < 3 * E; ++m) { free(ec[m]); free(eb[m]); }
    free(yp); free(h); free(out); free(lused); free(nx); free(ew); free(ecb); free(eco);
    if (bad) fprintf(stderr, "oracle driver: consistency failures 0x%x\n", bad);
    printf("oracle driver done\n");
    return bad ? 1 : 0;
}
