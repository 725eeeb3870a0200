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

}  // namespace dsa
