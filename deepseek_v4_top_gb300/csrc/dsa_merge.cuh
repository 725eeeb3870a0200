// Arithmetic of the merge of a decode row's key-chunk partials, shared by
// the combine kernel (dsa_simt.cu) and the merge inside the tensor-core
// kernel (dsa_tc.cu), so that both give the same bits.
//
// A chunk's partial for one head is (m, l, O): its reference maximum m (log2
// units; -inf when no key of the chunk had a finite score) and its sum l and
// value sum O, both relative to 2^m (2^0 when m is -inf).  Merged in chunk
// order (akol1 TensorFold PR #4, first commit message: a running maximum, a
// tile sum and a value sum; here the running state of each chunk is
// rescaled to the row's maximum and added), then the head's sink logit is
// folded into the denominator (TensorFold PR #1206, "What changes").
#pragma once

#include <math.h>

#include <cuda_bf16.h>

namespace dsa {

// Running maximum over the chunks' finite reference maxima.
__device__ __forceinline__ void merge_max(float& M, bool& have, float m) {
    if (m != -INFINITY) {
        M = have ? fmaxf(M, m) : m;
        have = true;
    }
}

// The merge's reference: the largest finite chunk maximum, or 0 if none.
__device__ __forceinline__ float merge_ref(float M, bool have) { return have ? M : 0.0f; }

// Weight of a chunk's (l, O) relative to the reference mu.
__device__ __forceinline__ float merge_weight(float m, float mu) {
    return m == -INFINITY ? 1.0f : exp2f(m - mu);
}

// Factor that turns the merged value sum (relative to 2^mu) into the
// output: 1 / (l + 2^(sink - mu)), computed against max(mu, sink) so that
// neither exponent overflows; a +inf sink gives 0, a -inf sink none.
__device__ __forceinline__ float merge_factor(float mu, float l, float sink) {
    const float s2 = sink * 1.4426950408889634f;
    const float mstar = isfinite(s2) ? fmaxf(mu, s2) : mu;
    const float e1 = exp2f(mu - mstar);
    const float e2 = exp2f(s2 - mstar);
    return e1 / (fmaf(l, e1, e2));
}

// Merges row r, head h: thread tid (0..127) owns output columns 4 tid ..
// 4 tid + 3.  part holds O [units][64][512] then (m, l) [units][2][64];
// row r's chunks are units r * chunks ...  Loads go through L2 (the
// partials may come from other CTAs of the same launch).  Up to kBatch
// chunks: every load is issued at once, then the maximum, then the sums in
// chunk order; more chunks: a first pass over m for the maximum, then the
// chunks kBatch at a time.  Both give the same arithmetic.  Writes the
// output row (fp32, or bf16 rounded to nearest even).
__device__ __forceinline__ void merge_row_head(const float* part, int units, int chunks, int H, int r, int h,
                                               int tid, float sink, void* out, int out_bf16) {
    constexpr int kBatch = 8;
    constexpr int kHP = 64, kDim = 512;
    const float* ml_base = part + static_cast<size_t>(units) * kHP * kDim;
    const size_t u0 = static_cast<size_t>(r) * chunks;
    float M = -INFINITY;
    bool have = false;
    float l = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float mu;
    if (chunks <= kBatch) {
        float mv[kBatch], lv[kBatch];
        float4 ov[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < chunks) {
                const size_t u = u0 + j;
                mv[j] = __ldcg(ml_base + u * 2 * kHP + h);
                lv[j] = __ldcg(ml_base + u * 2 * kHP + kHP + h);
                ov[j] = __ldcg(reinterpret_cast<const float4*>(part + (u * kHP + h) * kDim) + tid);
            } else {
                mv[j] = -INFINITY;
            }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) merge_max(M, have, mv[j]);
        mu = merge_ref(M, have);
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < chunks) {
                const float w = merge_weight(mv[j], mu);
                l = fmaf(w, lv[j], l);
                acc.x = fmaf(w, ov[j].x, acc.x);
                acc.y = fmaf(w, ov[j].y, acc.y);
                acc.z = fmaf(w, ov[j].z, acc.z);
                acc.w = fmaf(w, ov[j].w, acc.w);
            }
        }
    } else {
        for (int c0 = 0; c0 < chunks; c0 += kBatch) {
            float mv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                mv[j] = c0 + j < chunks ? __ldcg(ml_base + (u0 + c0 + j) * 2 * kHP + h) : -INFINITY;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) merge_max(M, have, mv[j]);
        }
        mu = merge_ref(M, have);
        for (int c0 = 0; c0 < chunks; c0 += kBatch) {
            float mv[kBatch], lv[kBatch];
            float4 ov[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (c0 + j < chunks) {
                    const size_t u = u0 + c0 + j;
                    mv[j] = __ldcg(ml_base + u * 2 * kHP + h);
                    lv[j] = __ldcg(ml_base + u * 2 * kHP + kHP + h);
                    ov[j] = __ldcg(reinterpret_cast<const float4*>(part + (u * kHP + h) * kDim) + tid);
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (c0 + j < chunks) {
                    const float w = merge_weight(mv[j], mu);
                    l = fmaf(w, lv[j], l);
                    acc.x = fmaf(w, ov[j].x, acc.x);
                    acc.y = fmaf(w, ov[j].y, acc.y);
                    acc.z = fmaf(w, ov[j].z, acc.z);
                    acc.w = fmaf(w, ov[j].w, acc.w);
                }
            }
        }
    }
    const float f = merge_factor(mu, l, sink);
    const float4 res = make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
    const size_t o0 = (static_cast<size_t>(r) * H + h) * kDim;
    if (out_bf16) {
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(out) + o0) + 2 * tid;
        o2[0] = __floats2bfloat162_rn(res.x, res.y);
        o2[1] = __floats2bfloat162_rn(res.z, res.w);
    } else {
        reinterpret_cast<float4*>(static_cast<float*>(out) + o0)[tid] = res;
    }
}

}  // namespace dsa
