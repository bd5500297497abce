// exp2 on the FMA pipe, to share the softmax's exponentials between the
// special-function unit (ex2.approx) and the fused multiply-add units.
//
// Method: Cody-Waite style range reduction x = n + f with n = round(x) (by
// the add-and-subtract of 1.5 * 2^23) and f in [-1/2, 1/2], a degree-3
// polynomial for 2^f, and the scaling by 2^n done by adding n to the
// exponent field.  The coefficients were fitted for minimum maximum relative
// error on [-1/2, 1/2] (Lawson's iteratively reweighted least squares); the
// maximum relative error of the fp32 evaluation is 7.5e-5, far below the
// bf16 rounding (2^-9) that every probability goes through afterwards.  The
// same coefficients are checked on the host by tests/test_exp2_poly.py.
#pragma once

namespace nc {

constexpr float EXP2_C0 = 0.99992805719375610f;
constexpr float EXP2_C1 = 0.69326096773147583f;
constexpr float EXP2_C2 = 0.24261112511157990f;
constexpr float EXP2_C3 = 0.05517166480422020f;

// 2^x for x <= 0 (inputs below -125 return about 2^-125: harmless for
// probabilities, and the attention kernels never produce them).
__device__ __forceinline__ float exp2_poly(float x) {
    x = fmaxf(x, -125.f);
    const float t = x + 12582912.f;  // 1.5 * 2^23: round(x) lands in the low mantissa bits
    const float f = x - (t - 12582912.f);
    const float p = fmaf(fmaf(fmaf(EXP2_C3, f, EXP2_C2), f, EXP2_C1), f, EXP2_C0);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

}  // namespace nc
