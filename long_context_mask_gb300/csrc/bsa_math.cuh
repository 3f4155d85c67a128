// Exponentials for the softmax: the MUFU instruction, and a replacement on
// the FMA pipe that takes part of the load off the MUFU unit.
#pragma once

#include <stdint.h>

namespace bsa {

// 2^x with the hardware approximation (MUFU.EX2), flushing subnormals.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^x on the FMA pipe.  Method: Cody and Waite range reduction x = j + f with
// j = round(x), |f| <= 1/2, then 2^f from a degree-3 polynomial whose
// coefficients minimise the maximum relative error on [-1/2, 1/2] (fitted by
// fit_exp2_poly.py; max relative error 7.5e-5), then the exponent field is
// raised by j.  Valid for x <= 127.  Inputs below -125 are clamped to -125
// so that the result stays a normal number (a softmax term of 2^-125 is
// nothing next to a row sum of at least 1).
__device__ __forceinline__ float exp2_fma(float x) {
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23: x + kRound rounds x to an integer
    constexpr float c0 = 0x1.fff694p-1f, c1 = 0x1.62f31ap-1f, c2 = 0x1.f0ddccp-3f,
                    c3 = 0x1.c3f6a6p-5f;
    x = fmaxf(x, -125.0f);
    const float t = x + kRound;
    const float f = x - (t - kRound);
    float p = fmaf(f, c3, c2);
    p = fmaf(f, p, c1);
    p = fmaf(f, p, c0);
    // t's low mantissa bits hold j; shifting them into the exponent scales p by 2^j
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

}  // namespace bsa
