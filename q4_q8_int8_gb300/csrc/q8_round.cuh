// q8_1 rounding shared by the prepass and the fused-output epilogue:
// q = clamp(roundf(x / d), -127, 127) with the quotient of IEEE division,
// formed from the correctly rounded reciprocal with an exactness test.
#pragma once

namespace mmq {
namespace q8 {

// q = clamp(roundf(x / d), -127, 127) with IEEE division, computed without a
// division in almost every case.  r = 1/d correctly rounded; q0 = x * r then
// differs from the exact quotient y = x/d by at most 2^-23 |y| < 2^-16 (|y| is
// at most 127 * (1 + 2^-23)), and fl(y) differs from y by at most 2^-18.  If
// q0 is more than 2^-15 away from every half-integer, q0, y and fl(y) lie in
// the same open interval (k - 1/2, k + 1/2), so roundf(fl(y)) is q0 rounded to
// the nearest integer (no tie is possible there, so the rounding mode of the
// conversion does not matter).  Otherwise `redo` is set and the caller
// recomputes that element with IEEE division.
__device__ __forceinline__ int quant_fast(float x, float r, bool& redo) {
    const float q0 = x * r;
    const float fr = fabsf(q0 - truncf(q0));   // exact (Sterbenz)
    redo = redo || !(fabsf(fr - 0.5f) > 0x1p-15f);
    return __float2int_rn(q0);
}

__device__ __forceinline__ int quant_exact(float x, float d) {
    return static_cast<int>(roundf(__fdiv_rn(x, d)));
}

__device__ __forceinline__ int clamp127(int q) { return q > 127 ? 127 : (q < -127 ? -127 : q); }

}  // namespace q8
}  // namespace mmq
