/*
 * dsa_oracle.h -- plain, slow, fp64 CPU definition of DeepSeek-V4.1 top-k
 * sparse attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the bench's CPU-baseline leg call it; the product never does.
 *
 * What is computed (akol1 TensorFold PR #4, first commit message: each
 * (row, head) scores its selected keys, keeps a running maximum, a tile sum
 * and a value sum, and writes sixteen 32-wide output columns; TensorFold
 * PR #1206, "What changes": one attention-sink logit per head):
 *
 *   x_j   = kv[slot(r)][idx[r][j]]                  j = 0 .. n_sel[r]-1
 *   s_j   = scale * sum_{d<512} q[r][h][d] * x_j[d]  (summed in order d)
 *   m     = largest FINITE value among {sink[h], s_0, ..., s_{K-1}} (0 if none)
 *   L     = exp(sink[h] - m) + sum_j exp(s_j - m)
 *   out[r][h][c] = (sum_j exp(s_j - m) * x_j[c]) / L
 *
 * The same 512-wide latent row is the key and the value.  All arithmetic is
 * IEEE double; inputs are widened exactly (float32, or bf16 bit patterns).
 * Taking the stabiliser m over finite logits only makes the result equal to
 * the unstabilised softmax in extended reals: a +inf sink gives 0, a +inf
 * score gives NaN, a -inf score gives weight 0.
 *
 * Library contract cases (not from the pages): a row whose n_sel is outside
 * [0, k_max], or whose first n_sel indices are not all in [0, N), yields NaN
 * in every output of that row.  Entries of idx at and beyond n_sel[r] are
 * never read.
 *
 * Layouts (row-major, contiguous):
 *   q    [R][H][512]        dtype elements
 *   kv   prefill (decode == 0): [N][512], one cache for every row;
 *        decode == T >= 1: [R/T][N][512], row r uses slot r / T (T query
 *        rows a slot, e.g. a decode step's draft tokens; T = 1 is the plain
 *        one-row-per-slot decode)
 *   idx  [R][k_max] int32,  n_sel [R] int32,  sink [H] float32
 *   out  double, [R][H][512] (dsa_oracle_attn) or [n_pairs][512]
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { DSA_ORACLE_F32 = 0, DSA_ORACLE_BF16 = 1 };

/* Returns 0 on success, 1 on an invalid argument (null pointer, bad size). */
int dsa_oracle_rowhead(const void* q, const void* kv, const int32_t* idx,
                       const int32_t* n_sel, const float* sink, float scale,
                       int dtype, int decode, int R, int H, int N, int k_max,
                       int r, int h, double* out512);

/* Every (row, head); threads <= 0 means all available threads.  The number
 * of threads actually used is stored in *threads_used when non-null. */
int dsa_oracle_attn(const void* q, const void* kv, const int32_t* idx,
                    const int32_t* n_sel, const float* sink, float scale,
                    int dtype, int decode, int R, int H, int N, int k_max,
                    double* out, int threads, int* threads_used);

/* A list of (row, head) pairs; out is [n_pairs][512]. */
int dsa_oracle_pairs(const void* q, const void* kv, const int32_t* idx,
                     const int32_t* n_sel, const float* sink, float scale,
                     int dtype, int decode, int R, int H, int N, int k_max,
                     const int32_t* rows, const int32_t* heads, int n_pairs,
                     double* out, int threads, int* threads_used);

/* Threads an all-thread call would use. */
int dsa_oracle_max_threads(void);

/*
 * Top-k selection of an indexer's scores (the "merge and finish" that turns
 * a row's index scores into the selection the attention reads: DeepSeek
 * V4.1 indexer PR #2, title: the indexer's merge and finish on a threadgroup
 * a row, the same picks).  The pages give the title only; the reading is:
 *
 *   candidates of row r: positions j in [0, n_valid[r]) with score s[r][j]
 *   order: larger score first; NaN after every number (also after -inf);
 *          -0 and +0 are equal; equal scores by smaller position first
 *   n_sel[r] = min(k, n_valid[r]); the picks are the first n_sel candidates
 *   in that order; idx[r][0 .. n_sel) = the picks in ascending position
 *   (the attention reads a set: its sum does not depend on the order, and
 *   ascending positions are its one canonical listing);
 *   idx[r][n_sel .. k_max) = -1.
 *
 * Library contract case (not from the pages): a row whose n_valid is outside
 * [0, ld] selects nothing (n_sel 0, idx all -1) and is reported in bad[r]
 * (1, else 0).
 *
 * Layouts: scores [R][ld] float32 (row r starts at r * ld), n_valid [R],
 * idx [R][k_max] int32, n_sel [R] int32, bad [R] int32 (may be null).
 * Returns 0, or 1 on an invalid argument (null pointer, k < 1, k > k_max,
 * ld < 0, R < 0).
 */
int dsa_oracle_topk(const float* scores, int ld, const int32_t* n_valid, int R, int k,
                    int k_max, int32_t* idx, int32_t* n_sel, int32_t* bad);

/*
 * Output projection, the step after the attention: a row's heads' outputs,
 * concatenated (k = h*512 + c), times the projection matrix (TensorFold PR
 * #1206, "What changes": the attention's output groups go to the output
 * projections; the pages give no shape for the matrix, so d_out is the
 * caller's):
 *   out[r][n] = sum_{k<K} a[r][k] * w[k][n]          (summed in order k)
 * a [R][K] is given either as doubles (a_f64, e.g. dsa_oracle_attn's output
 * with K = H*512) or as bf16 bit patterns (a_bf16); exactly one is non-null.
 * w [K][d_out] bf16 bit patterns.  out [R][d_out] double.  abs_out (may be
 * null) receives sum_k |a[r][k]| * |w[k][n]|, the scale of a rounding bound.
 * Returns 0, or 1 on an invalid argument.
 */
int dsa_oracle_oproj(const double* a_f64, const uint16_t* a_bf16, const uint16_t* w, int R, int K,
                     int d_out, double* out, double* abs_out, int threads);

#ifdef __cplusplus
}
#endif
#endif
