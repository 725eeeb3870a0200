/*
 * dsa_oracle.c -- fp64 CPU oracle for top-k sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU baseline).  It
 * shares no code with the CUDA library and is deliberately plain: two passes
 * over the selected keys of one (row, head), no blocking, no fusion.
 *
 * Source of the definition: akol1 TensorFold PR #4, first commit message
 * (score the selected keys, running maximum, tile sum, value sum, sixteen
 * 32-wide output columns of one latent row) and TensorFold PR #1206, "What
 * changes" (per-head sinks that enter the softmax).  The tiled, online form
 * of those pages reaches this same value up to rounding: the rescaling by
 * exp(m_old - m_new) cancels between numerator and denominator.
 */
#include "dsa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define DSA_D 512

/* bf16 bit pattern -> double, exactly (a bf16 is the top half of a float). */
static double widen_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load(const void* base, int dtype, size_t i) {
    if (dtype == DSA_ORACLE_BF16) return widen_bf16(((const uint16_t*)base)[i]);
    return (double)((const float*)base)[i];
}

static int check_args(const void* q, const void* kv, const int32_t* idx,
                      const int32_t* n_sel, const float* sink, int dtype,
                      int R, int H, int N, int k_max) {
    if (!q || !kv || !idx || !n_sel || !sink) return 1;
    if (dtype != DSA_ORACLE_F32 && dtype != DSA_ORACLE_BF16) return 1;
    if (R < 0 || H <= 0 || N <= 0 || k_max <= 0) return 1;
    return 0;
}

/* One (row, head): the definition in dsa_oracle.h, written out. */
static void rowhead(const void* q, const void* kv, const int32_t* idx,
                    const int32_t* n_sel, const float* sink, float scale,
                    int dtype, int decode, int H, int N, int k_max,
                    int r, int h, double* out, double* s /* [k_max] scratch */) {
    const int K = n_sel[r];
    int c, j;
    /* contract: out-of-range selection -> NaN row */
    int bad = (K < 0 || K > k_max);
    for (j = 0; !bad && j < K; ++j) {
        int32_t p = idx[(size_t)r * k_max + j];
        if (p < 0 || p >= N) bad = 1;
    }
    if (bad) {
        for (c = 0; c < DSA_D; ++c) out[c] = NAN;
        return;
    }

    const size_t qoff = ((size_t)r * H + h) * DSA_D;
    /* decode: T = decode rows share a slot; row r reads slot r / T */
    const size_t slot = decode ? (size_t)(r / decode) * (size_t)N * DSA_D : 0;
    const double sc = (double)scale;
    const double sk = (double)sink[h];

    /* pass 1: scores and the finite stabiliser */
    int have = 0;
    double m = 0.0;
    if (isfinite(sk)) { m = sk; have = 1; }
    for (j = 0; j < K; ++j) {
        const size_t xoff = slot + (size_t)idx[(size_t)r * k_max + j] * DSA_D;
        double dot = 0.0;
        int d;
        for (d = 0; d < DSA_D; ++d) dot += load(q, dtype, qoff + d) * load(kv, dtype, xoff + d);
        s[j] = sc * dot;
        if (isfinite(s[j]) && (!have || s[j] > m)) { m = s[j]; have = 1; }
    }

    /* pass 2: weights, denominator (sink first, then keys in order), values */
    double L = exp(sk - m);
    for (c = 0; c < DSA_D; ++c) out[c] = 0.0;
    for (j = 0; j < K; ++j) {
        const size_t xoff = slot + (size_t)idx[(size_t)r * k_max + j] * DSA_D;
        const double w = exp(s[j] - m);
        L += w;
        for (c = 0; c < DSA_D; ++c) out[c] += w * load(kv, dtype, xoff + c);
    }
    for (c = 0; c < DSA_D; ++c) out[c] /= L;
}

int dsa_oracle_rowhead(const void* q, const void* kv, const int32_t* idx,
                       const int32_t* n_sel, const float* sink, float scale,
                       int dtype, int decode, int R, int H, int N, int k_max,
                       int r, int h, double* out512) {
    if (check_args(q, kv, idx, n_sel, sink, dtype, R, H, N, k_max) || !out512) return 1;
    if (r < 0 || r >= R || h < 0 || h >= H) return 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)k_max);
    if (!s) return 1;
    rowhead(q, kv, idx, n_sel, sink, scale, dtype, decode, H, N, k_max, r, h, out512, s);
    free(s);
    return 0;
}

int dsa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int dsa_oracle_pairs(const void* q, const void* kv, const int32_t* idx,
                     const int32_t* n_sel, const float* sink, float scale,
                     int dtype, int decode, int R, int H, int N, int k_max,
                     const int32_t* rows, const int32_t* heads, int n_pairs,
                     double* out, int threads, int* threads_used) {
    int i, err = 0;
    if (check_args(q, kv, idx, n_sel, sink, dtype, R, H, N, k_max) || !out) return 1;
    if (n_pairs < 0 || (n_pairs > 0 && (!rows || !heads))) return 1;
    for (i = 0; i < n_pairs; ++i)
        if (rows[i] < 0 || rows[i] >= R || heads[i] < 0 || heads[i] >= H) return 1;
    int nt = threads > 0 ? threads : dsa_oracle_max_threads();
#ifndef _OPENMP
    nt = 1;
#endif
    if (threads_used) *threads_used = nt;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)k_max);
        if (!s) {
            err = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (i = 0; i < n_pairs; ++i)
                rowhead(q, kv, idx, n_sel, sink, scale, dtype, decode, H, N, k_max,
                        rows[i], heads[i], out + (size_t)i * DSA_D, s);
            free(s);
        }
    }
    return err;
}

int dsa_oracle_attn(const void* q, const void* kv, const int32_t* idx,
                    const int32_t* n_sel, const float* sink, float scale,
                    int dtype, int decode, int R, int H, int N, int k_max,
                    double* out, int threads, int* threads_used) {
    if (check_args(q, kv, idx, n_sel, sink, dtype, R, H, N, k_max) || !out) return 1;
    const int n = R * H;
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t* heads = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    if (!rows || !heads) { free(rows); free(heads); return 1; }
    int i;
    for (i = 0; i < n; ++i) { rows[i] = i / H; heads[i] = i % H; }
    int rc = dsa_oracle_pairs(q, kv, idx, n_sel, sink, scale, dtype, decode, R, H, N,
                              k_max, rows, heads, n, out, threads, threads_used);
    free(rows);
    free(heads);
    return rc;
}

/* ------------------------------------------------------------- top-k */
typedef struct {
    float s;
    int32_t pos;
} sel_t;

/* The selection order of dsa_oracle_topk: non-NaN before NaN, then larger
 * score first (IEEE comparison, so -0 == +0), then smaller position. */
static int sel_cmp(const void* a, const void* b) {
    const sel_t* x = (const sel_t*)a;
    const sel_t* y = (const sel_t*)b;
    const int xn = isnan(x->s), yn = isnan(y->s);
    if (xn != yn) return xn - yn;
    if (!xn) {
        if (x->s > y->s) return -1;
        if (x->s < y->s) return 1;
    }
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int pos_cmp(const void* a, const void* b) {
    const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

int dsa_oracle_topk(const float* scores, int ld, const int32_t* n_valid, int R, int k,
                    int k_max, int32_t* idx, int32_t* n_sel, int32_t* bad) {
    if (R < 0 || ld < 0 || k < 1 || k > k_max) return 1;
    if (R == 0) return 0;
    if (!scores || !n_valid || !idx || !n_sel) return 1;
    sel_t* buf = (sel_t*)malloc(sizeof(sel_t) * (size_t)(ld > 0 ? ld : 1));
    if (!buf) return 1;
    int r, j;
    for (r = 0; r < R; ++r) {
        const int n = n_valid[r];
        const int ok = n >= 0 && n <= ld;
        if (bad) bad[r] = ok ? 0 : 1;
        const int m = ok ? (n < k ? n : k) : 0;
        for (j = 0; ok && j < n; ++j) {
            buf[j].s = scores[(size_t)r * (size_t)ld + (size_t)j];
            buf[j].pos = j;
        }
        if (ok && n > 1) qsort(buf, (size_t)n, sizeof(sel_t), sel_cmp);
        /* the picks, listed by ascending position */
        int32_t* out = idx + (size_t)r * (size_t)k_max;
        for (j = 0; j < m; ++j) out[j] = buf[j].pos;
        if (m > 1) qsort(out, (size_t)m, sizeof(int32_t), pos_cmp);
        for (j = m; j < k_max; ++j) out[j] = -1;
        n_sel[r] = m;
    }
    free(buf);
    return 0;
}

int dsa_oracle_oproj(const double* a_f64, const uint16_t* a_bf16, const uint16_t* w, int R, int K,
                     int d_out, double* out, double* abs_out, int threads) {
    if (R < 0 || K < 1 || d_out < 1 || !w || !out) return 1;
    if ((a_f64 == NULL) == (a_bf16 == NULL)) return 1;
    int nt = threads;
#ifdef _OPENMP
    if (nt <= 0) nt = omp_get_max_threads();
#else
    nt = 1;
#endif
    int r;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (r = 0; r < R; ++r) {
        double* o = out + (size_t)r * (size_t)d_out;
        double* ao = abs_out ? abs_out + (size_t)r * (size_t)d_out : NULL;
        int n, k;
        for (n = 0; n < d_out; ++n) {
            o[n] = 0.0;
            if (ao) ao[n] = 0.0;
        }
        for (k = 0; k < K; ++k) {
            const size_t ak = (size_t)r * (size_t)K + (size_t)k;
            const double a = a_f64 ? a_f64[ak] : widen_bf16(a_bf16[ak]);
            const uint16_t* wk = w + (size_t)k * (size_t)d_out;
            for (n = 0; n < d_out; ++n) {
                const double wv = widen_bf16(wk[n]);
                o[n] += a * wv;
                if (ao) ao[n] += fabs(a) * fabs(wv);
            }
        }
    }
    return 0;
}
