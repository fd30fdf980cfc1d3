/*
 * mx.c -- MXFP8 activations (OCP Microscaling formats): E4M3 elements with
 * one E8M0 scale per 32.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * "Models and formats" page, "Tensor formats": MXFP4 weights (E2M1 codes with
 * an E8M0 scale per 32) are among the formats read.  A tensor-core product of
 * such weights that keeps them in their own block-scaled form needs the
 * activations in a block-scaled 8-bit form too; the pages do not print one.
 * The reading taken is the OCP Microscaling (MX) specification v1.0's MXFP8
 * (E4M3) and its conversion from a vector of scalars (section 6.3):
 *
 *   per block of 32 values x_i:
 *     amax = max |x_i|
 *     E    = floor(log2(amax)) - 8           (8: the largest E4M3 exponent,
 *                                             448 = 1.75 * 2^8), and -127 for
 *                                             a block of zeros; E >= -127
 *     X    = 2^E, stored as the E8M0 byte E + 127
 *     q_i  = E4M3(x_i / X), rounded to nearest (ties to even) and clamped
 *            to the largest finite magnitude 448 (the specification leaves
 *            overflow to the implementation; clamping is its saturating form)
 *   block layout: E8M0 byte | 32 E4M3 bytes                  -> 33 bytes
 *
 * E4M3 (the "fn" variant of the specification): sign | 4-bit exponent, bias 7
 * | 3-bit mantissa; exponent 0 holds the subnormals m * 2^-9; S.1111.111 is NaN
 * and there are no infinities.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

double orc_e4m3_to_f64(uint8_t b)
{
    const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

uint8_t orc_f64_to_e4m3_rn_sat(double v)
{
    if (isnan(v)) return 0x7f;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7e;            /* 1.1111.110 = 448 */
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid m * 2^-9, m = 0..8 (8 is the smallest normal) */
        const double m = nearbyint(ldexp(a, 9));   /* ties to even in the default mode */
        return sign | (uint8_t)m;                  /* m = 8 encodes 0.0001.000 = 2^-6 */
    }
    int ex;
    frexp(a, &ex);                                 /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                                /* a in [2^e, 2^(e+1)) */
    double q = nearbyint(ldexp(a, 3 - e));         /* in [8, 16] */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0)) return sign | 0x7e;   /* rounded past 448 */
    return sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

static void mxfp8_block(const float* x, uint8_t* o)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        const float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    int E = -127;
    if (amax > 0.0f) {
        int ex;
        frexp((double)amax, &ex);
        E = ex - 1 - 8;
        if (E < -127) E = -127;
    }
    o[0] = (uint8_t)(E + 127);
    for (int i = 0; i < 32; i++) o[1 + i] = orc_f64_to_e4m3_rn_sat(ldexp((double)x[i], -E));
}

int orc_quantize_mxfp8(const float* x, int64_t n, uint8_t* out)
{
    if (n < 0) return ORC_EINVAL;
    if (n % 32) return ORC_ESHAPE;
    for (int64_t i = 0; i < n; i++)
        if (!isfinite(x[i])) return ORC_ERANGE;
    for (int64_t b = 0; b < n / 32; b++) mxfp8_block(x + 32 * b, out + 33 * b);
    return ORC_OK;
}

double orc_mxfp8_value(const uint8_t* blk, int i)
{
    return ldexp(orc_e4m3_to_f64(blk[1 + i]), (int)blk[0] - 127);
}
