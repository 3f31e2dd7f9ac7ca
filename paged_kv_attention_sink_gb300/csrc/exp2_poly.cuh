// 2^x on the FMA pipe, for the prefill softmax.
//
// The multi-function unit (MUFU, `ex2.approx`) gives 8 results per clock per
// SM sub-partition while the FMA pipe retires 32 fp32 lanes per clock, so part
// of a tile's exponentials can be evaluated as a polynomial on the FMA pipe
// instead (the prefill kernel's kPolyEvery selects the share).  On GB300 the
// kernel measured slower with every share tried, since the softmax warp's
// chain of dependent work, not the MUFU's rate, sets its pace; the share
// defaults to none and the function is kept, tested, for kernels where the
// MUFU is the limit.
//
// Method (written from the mathematics, not from any library's exp):
//
//  1. Clamp and scale.  y = sat(x / R + 1/2) with R = 252, folded into the
//     score's own fma: y = sat(s * (scale_log2 / R) + (1/2 - m / R)), so
//     x' = R * y - R / 2 is x clamped to [-126, 126] (NaN clamps to -126).
//     The clamp keeps the exponent arithmetic of step 4 inside the normal
//     range: a result below 2^-126 is at most 2^-126 instead of 0, and one
//     above 2^126 is 2^126, large enough to trip the prefill softmax's
//     row-sum check (2^64) that raises the running max and recomputes.
//  2. Range reduction (Cody-Waite for base 2: the split is exact).
//     t = fma_rm(y, R, C) with C = 1.5 * 2^23 - R / 2: the sum is exact in the
//     fma and rounding toward -inf at a magnitude where one ulp is 1 leaves
//     t = 1.5 * 2^23 + floor(x'), so the low mantissa bits of t hold the
//     integer part j = floor(x') in two's complement.  Then u = C - t is
//     exact (Sterbenz) and f = fma(y, R, u) = x' - j lies in [0, 1].
//  3. 2^f on [0, 1] by a cubic, Horner's rule, fp32 fma.  The coefficients
//     are the minimax fit of the RELATIVE error found by the Remez exchange
//     algorithm (float64, equioscillation on 5 points, then
//     rounded to fp32); the fit script sits beside this file
//     (fit_exp2_poly.py).  Fitted error 7.48e-5; with the fp32 argument
//     (the rounded scale s * a and sum y) and evaluation the whole sequence
//     stays within 9.0e-5 (2^-13.4) of 2^x for x in [-125.9, 8.5] and
//     logits up to ~70.  P is rounded to bf16 right after (relative error up
//     to 2^-9 = 1.95e-3), so this adds under 5% to P's rounding error, and
//     lse (from the unrounded sum) moves by at most 9.0e-5.
//  4. Scale by 2^j: add j << 23 to the bit pattern of p (p in [0.9999, 2]).
//     Since t's bit pattern is 0x4B400000 + j and 0x4B400000 << 23 wraps to
//     0, this is bits(p) + (bits(t) << 23) in 32-bit integer arithmetic.
//
// Steps 2-3 run as packed fp32x2 instructions on two scores at once.
#pragma once

#include <cstdint>

namespace attn {
namespace exp2poly {

constexpr float kRange = 252.0f;                    // R
constexpr float kInvRange = 1.0f / 252.0f;
constexpr float kShift = 12582912.0f - 126.0f;      // C = 1.5 * 2^23 - R / 2
// Minimax (relative error) cubic for 2^f on [0, 1]: c0 + c1 f + c2 f^2 + c3 f^3.
constexpr float kC0 = 0x1.fff632p-1f;   // 0.99992522
constexpr float kC1 = 0x1.64444cp-1f;   // 0.69583356
constexpr float kC2 = 0x1.cefc4cp-3f;   // 0.22606716
constexpr float kC3 = 0x1.3f96a4p-4f;   // 0.07802452

__device__ __forceinline__ uint64_t pair_bits(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

// Step 1 for one score: y = sat(s * a + b), a = scale_log2 / R,
// b = 1/2 - m / R (m = the running max in log2 units).
__device__ __forceinline__ float clamp_arg(float s, float a, float b) {
    float y;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(s), "f"(a), "f"(b));
    return y;
}

// Steps 2-4 for two clamped arguments (y0, y1); returns (2^x0', 2^x1').
__device__ __forceinline__ float2 from_clamped(float y0, float y1) {
    const uint64_t y = pair_bits(y0, y1);
    const uint64_t r2 = pair_bits(kRange, kRange), c2 = pair_bits(kShift, kShift);
    uint64_t t, u, f, p;
    asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(y), "l"(r2), "l"(c2));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(u) : "l"(c2), "l"(t));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(f) : "l"(y), "l"(r2), "l"(u));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(p) : "l"(pair_bits(kC3, kC3)), "l"(f), "l"(pair_bits(kC2, kC2)));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(p) : "l"(p), "l"(f), "l"(pair_bits(kC1, kC1)));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(p) : "l"(p), "l"(f), "l"(pair_bits(kC0, kC0)));
    const uint32_t lo = (uint32_t)p + ((uint32_t)t << 23);
    const uint32_t hi = (uint32_t)(p >> 32) + ((uint32_t)(t >> 32) << 23);
    return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// 2^(s * scale_log2 - m) for two scores, with a = scale_log2 / R and
// b = 1/2 - m / R precomputed by the caller.
__device__ __forceinline__ float2 exp2_pair(float s0, float s1, float a, float b) {
    return from_clamped(clamp_arg(s0, a, b), clamp_arg(s1, a, b));
}

}  // namespace exp2poly
}  // namespace attn
