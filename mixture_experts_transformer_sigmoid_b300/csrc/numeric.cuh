// Small floating-point helpers shared by the kernels.
#pragma once

namespace moe {

// Error-free addition (Knuth's two-sum): s + e == a + b exactly, s = fl(a + b).
// The _rn intrinsics keep the compiler from contracting or reordering it.
__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (hi + lo) / n rounded to fp32, in fp32 arithmetic only (the fp64 rate of
// this part is a small fraction of its fp32 rate).  The pair is first made
// non-overlapping (s + e == hi + lo exactly); q = fl(s / n) leaves the exact
// remainder s - q n (representable for a correctly rounded quotient, and
// produced by one FMA since n < 2^24 is exact in fp32); the remainder plus e,
// over n, is the correction, added with one rounding.  That correction is
// within about 2^-23 of itself, so the result is the correctly rounded
// quotient unless the exact one lies that close (in ulps) to a rounding
// boundary.
__device__ __forceinline__ float mean_of_pair(float hi, float lo, int n) {
    float s, e;
    two_sum_f(hi, lo, s, e);
    const float nf = static_cast<float>(n);
    const float q = __fdiv_rn(s, nf);
    const float r = fmaf(-q, nf, s);
    return __fadd_rn(q, __fdiv_rn(__fadd_rn(r, e), nf));
}

}  // namespace moe
