// fa_exp2.cuh -- 2^x on the FMA pipe (Cody-Waite + degree-3 Horner).
//
// FlashAttention-4 blog, "Faster exponential: split 2^x between MUFU.EX2 and
// FMA": write 2^x = 2^n * 2^f with n = floor(x) and f = x - n in [0,1),
// approximate 2^f by p0 + f (p1 + f (p2 + f p3)) with p0 = 1, and apply 2^n by
// adding n to the float32 exponent field.  FlashAttention-4 paper summary
// §3.1.3 / Table 2: the degree-3 form stays within 8.77e-5 relative error in
// float32, far below the 2^-8 relative rounding of the bf16 P it feeds.
//
// Own derivation:
//  * Coefficients: minimax of the relative error on [0,1] with p0 = 1, fitted
//    by a linear program on a dense grid (max relative error 8.56e-5 before
//    float32 rounding of the evaluation), rounded to float32.
//  * floor(x) without a float->int conversion instruction (conversions issue
//    on the same narrow pipe as MUFU): adding 1.5 * 2^23 under round-toward-
//    minus-infinity leaves floor(x) in the low mantissa bits of the sum (the
//    classic "magic number" rounding trick, valid for |x| < 2^22); subtracting
//    the constant back gives floor(x) exactly as a float.  The exponent update
//    is then an integer shift-and-add of those low bits: (bits(j) << 23) ==
//    (n << 23) modulo 2^32 because the constant's own bits shift out.
//  * Inputs are clamped below at -127 (masked logits are -inf): the result is
//    then 0 (n = -127, f = 0) or below 2^-126.  Valid for x < 128.
#pragma once
#include <stdint.h>

#include "fa_prim.cuh"

namespace fa {

constexpr float kExp2P1 = 0x1.63e66ap-1f;  // 0.69511729
constexpr float kExp2P2 = 0x1.d236c6p-3f;  // 0.22764353
constexpr float kExp2P3 = 0x1.3babb0p-4f;  // 0.07706803

__device__ __forceinline__ float exp2_fma(float x) {
    x = fmaxf(x, -127.0f);
    const float j = __fadd_rd(x, 12582912.0f);  // 1.5 * 2^23, rounded down
    const float n = j - 12582912.0f;            // floor(x), exact
    const float f = x - n;                      // [0, 1), exact
    const float p = fmaf(f, fmaf(f, fmaf(f, kExp2P3, kExp2P2), kExp2P1), 1.0f);
    return __int_as_float(__float_as_int(p) + (__float_as_int(j) << 23));
}

// The same function on two lanes of a packed fp32 pair (sm_100 family f32x2
// arithmetic: one instruction per step for both elements); every step rounds
// exactly as in exp2_fma, so each element equals exp2_fma's result.
__device__ __forceinline__ void exp2_fma_x2(float x0, float x1, float& y0, float& y1) {
    uint64_t x, j, n, f, p;
    x = f2_pack(fmaxf(x0, -127.0f), fmaxf(x1, -127.0f));
    const uint64_t magic = f2_pack(12582912.0f, 12582912.0f);
    asm("add.rm.f32x2 %0, %1, %2;" : "=l"(j) : "l"(x), "l"(magic));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(n) : "l"(j), "l"(magic));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(f) : "l"(x), "l"(n));
    p = f2_fma(f, f2_pack(kExp2P3, kExp2P3), f2_pack(kExp2P2, kExp2P2));
    p = f2_fma(f, p, f2_pack(kExp2P1, kExp2P1));
    p = f2_fma(f, p, f2_pack(1.0f, 1.0f));
    float p0, p1, j0, j1;
    f2_unpack(p, p0, p1);
    f2_unpack(j, j0, j1);
    y0 = __int_as_float(__float_as_int(p0) + (__float_as_int(j0) << 23));
    y1 = __int_as_float(__float_as_int(p1) + (__float_as_int(j1) << 23));
}

}  // namespace fa
