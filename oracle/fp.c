/*
 * fp.c -- IEEE-754 binary16 and bfloat16 conversions, written out from the
 * bit encodings.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * The block formats of the "Models and formats" page ("Tensor formats") keep
 * their scales as fp16; the prefill multiply of the "Architecture" page
 * ("The package map", pkg/tensor MatMul) is fed bf16 tiles here.  Neither page
 * prints a conversion, so these follow the IEEE-754 definitions:
 *   binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 *   bfloat16: the upper 16 bits of binary32 (8 exponent bits, 7 fraction bits);
 *   rounding: to nearest, ties to even.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (ex == 31) {
        v = frac ? NAN : INFINITY;
    } else if (ex == 0) {
        v = ldexp((double)frac, -24);               /* subnormal: frac * 2^-24 */
    } else {
        v = ldexp((double)(1024 + frac), ex - 25);  /* (1.frac) * 2^(ex-15) */
    }
    return sign ? -v : v;
}

/* Round m * 2^(e-23) (m a 24-bit significand, 2^23 <= m < 2^24) to binary16. */
static uint16_t round_to_f16(uint16_t sign, int e, uint32_t m)
{
    if (e > 15) return (uint16_t)(sign | 0x7c00);          /* beyond the largest binade */
    int normal = e >= -14;
    int ulp_exp = normal ? e - 10 : -24;                   /* weight of the last kept bit */
    int s = ulp_exp - (e - 23);                            /* bits to drop, >= 13 */
    uint64_t q;
    if (s >= 63) {
        q = 0;
    } else {
        uint64_t mm = m;
        uint64_t rem = mm & ((1ull << s) - 1);
        uint64_t half = 1ull << (s - 1);
        q = mm >> s;
        if (rem > half || (rem == half && (q & 1))) q++;
    }
    uint32_t bits;
    if (normal) {
        /* q in [1024, 2048]; q == 2048 carries into the exponent, up to 0x7c00 (inf). */
        bits = ((uint32_t)(e + 15) << 10) + (uint32_t)(q - 1024);
    } else {
        /* q in [0, 1024]; 1024 is the smallest normal. */
        bits = (uint32_t)q;
    }
    return (uint16_t)(sign | bits);
}

uint16_t orc_f32_to_f16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
    uint32_t ex = (u >> 23) & 0xff;
    uint32_t frac = u & 0x7fffff;
    if (ex == 0xff) return (uint16_t)(sign | 0x7c00 | (frac ? 0x200 : 0));
    if (ex == 0) return sign;   /* binary32 subnormals are below 2^-126, far under half of 2^-24 */
    return round_to_f16(sign, (int)ex - 127, frac | 0x800000);
}

double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

uint16_t orc_f32_to_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000) == 0x7f800000 && (u & 0x7fffff)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lower = u & 0xffff;        /* the 16 bits dropped */
    uint32_t upper = u >> 16;
    if (lower > 0x8000 || (lower == 0x8000 && (upper & 1))) upper++;   /* carries into the exponent as it must */
    return (uint16_t)upper;
}
