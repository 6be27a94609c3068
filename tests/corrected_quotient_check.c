/*
 * Host model of the quantisers' per-element arithmetic, for an exhaustive
 * check against the definition (test_corrected_quotient.py compiles and
 * drives it; no GPU, no CUDA code).
 *
 * The kernels code a value x of a group with scale s as
 *     q0 = RN(x r),  e = RN(x - q0 s) (fused),  q = RN(q0 + e r) (fused),
 *     code = E4M3(q)
 * with r one of RN(1/s) and its two fp32 neighbours (a correction step in the
 * manner of Markstein's division).  The definition is code = E4M3(RN(x / s)).
 * check_range() walks every bf16 amax in [amax_lo, amax_hi] (bit patterns of
 * positive finite values) whose scale s = RN(amax / 448) is at least 2^-100,
 * and every bf16 x with |x| <= amax except -0, and counts the pairs whose two
 * codes differ.  Codes come from the caller's encoder (the oracle's), which
 * is only called when the two fp32 quotients differ: equal quotients have
 * equal codes.
 *
 * Built with IEEE single precision semantics: no fast-math, no contraction
 * of a * b + c into a fused operation except where fmaf() says so.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef uint8_t (*encoder_fn)(float);

static float from_bits(uint32_t b)
{
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static uint32_t bits_of(float f)
{
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    return b;
}

/* variant: 0 -> r = RN(1/s); 1 -> its neighbour toward zero; 2 -> toward +inf;
 * 3 -> r = RN(1/s) without the correction (q = q0), a planted mistake.
 * Returns the number of mismatching pairs; *pairs receives the pairs checked,
 * *quotients_differ those whose fp32 quotients differ. */
long long check_range(uint32_t amax_lo, uint32_t amax_hi, int variant, encoder_fn enc, long long *pairs,
                      long long *quotients_differ)
{
    long long bad = 0, n = 0, qd = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(+ : bad, n, qd)
    for (int64_t ab = (int64_t)amax_lo; ab <= (int64_t)amax_hi; ++ab) {
        volatile float d448 = 448.0f, one = 1.0f;
        const float amax = from_bits((uint32_t)ab << 16);
        const float s = amax / d448;
        if (!(s >= 0x1p-100f) || !(s <= 3.40282347e38f))
            continue;
        float r = one / s;
        if (variant == 1)
            r = nextafterf(r, 0.0f);
        else if (variant == 2)
            r = nextafterf(r, INFINITY);
        const float ns = -s;
        for (uint32_t xs = 0; xs < 2u * ((uint32_t)ab + 1u); ++xs) {
            const uint32_t xb = (xs >> 1) | ((xs & 1u) << 15);   /* +m, -m for every magnitude m <= amax */
            if (xb == 0x8000u)
                continue;                                        /* -0 takes the division in the kernels */
            const float x = from_bits(xb << 16);
            const float ref = x / s;
            const float q0 = x * r;
            const float e = fmaf(q0, ns, x);
            const float q = variant == 3 ? q0 : fmaf(e, r, q0);
            ++n;
            if (bits_of(ref) != bits_of(q)) {
                ++qd;
                if (enc(ref) != enc(q))
                    ++bad;
            }
        }
    }
    *pairs = n;
    *quotients_differ = qd;
    return bad;
}
