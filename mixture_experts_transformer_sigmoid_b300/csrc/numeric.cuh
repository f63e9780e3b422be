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

}  // namespace moe
