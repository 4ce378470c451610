/*
 * exp2 by Cody-Waite range reduction and a degree-3 Horner polynomial, float32.
 *
 * TEST INFRASTRUCTURE ONLY: part of the CPU oracle, never linked into the
 * CUDA library.
 *
 * Follows the FlashAttention-4 blog, section "Faster exponential: split 2^x
 * between MUFU.EX2 and FMA", in its order:
 *   1. range reduction: 2^x = 2^n * 2^f with n = floor(x), f = x - n in [0,1);
 *   2. 2^f ~ p0 + f (p1 + f (p2 + f p3)) evaluated by Horner with fused
 *      multiply-adds (the FMA units the section names), p0 = 1;
 *   3. multiply by 2^n by adding n to the float32 exponent field (n << 23),
 *      because 2^f in [1,2) has biased exponent 127.
 * The coefficients are passed in (the oracle fits them itself, see
 * exp2_poly.py).  The FlashAttention-4 paper summary, §3.1.3 / Table 2,
 * states the maximum relative error of this degree-3 form on [0,1) as
 * 8.77e-5.
 *
 * Reading where the pages are silent: inputs below -127 (including -inf,
 * a masked logit) are clamped to -127, so the result is 0 or a value below
 * 2^-126; step 3 would otherwise wrap the exponent field.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

float exp2_poly(float x, float p1, float p2, float p3)
{
    if (!(x >= -127.0f)) x = -127.0f;           /* also catches -inf */
    float n = floorf(x);
    float f = x - n;                            /* exact: |x| < 2^23 */
    float p = fmaf(f, fmaf(f, fmaf(f, p3, p2), p1), 1.0f);
    uint32_t bits;
    memcpy(&bits, &p, sizeof bits);
    bits += (uint32_t)((int32_t)n) << 23;
    float r;
    memcpy(&r, &bits, sizeof r);
    return r;
}

void exp2_poly_many(const float *x, float *y, long n, float p1, float p2, float p3)
{
    for (long i = 0; i < n; ++i) y[i] = exp2_poly(x[i], p1, p2, p3);
}

/* Largest |exp2_poly(x) - 2^x| / 2^x over EVERY float32 x in [lo_bits, hi_bits]
 * (bit patterns of non-negative floats), 2^x taken in double.  With
 * lo_bits = 0 and hi_bits = 0x3f7fffff this is all of [0, 1). */
double exp2_poly_max_rel_err(uint32_t lo_bits, uint32_t hi_bits,
                             float p1, float p2, float p3, float *argmax)
{
    double worst = 0.0;
    float worst_x = 0.0f;
    #pragma omp parallel
    {
        double w = 0.0;
        float wx = 0.0f;
        #pragma omp for schedule(static)
        for (int64_t b = (int64_t)lo_bits; b <= (int64_t)hi_bits; ++b) {
            uint32_t u = (uint32_t)b;
            float x;
            memcpy(&x, &u, sizeof x);
            double exact = exp2((double)x);
            double e = fabs((double)exp2_poly(x, p1, p2, p3) - exact) / exact;
            if (e > w) { w = e; wx = x; }
        }
        #pragma omp critical
        {
            if (w > worst) { worst = w; worst_x = wx; }
        }
    }
    if (argmax) *argmax = worst_x;
    return worst;
}
