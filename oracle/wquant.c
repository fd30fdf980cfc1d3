/*
 * wquant.c -- weight quantisers, fp32 rows to Q4_0 / Q5_0 / Q8_0 blocks.
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * "Models and formats" page, "Tensor formats": `llamay quantize` writes
 * Q4_0/1, Q5_0/1, Q8_0 and the K-quants.  The pages name the formats but not
 * the procedure that picks a block's scale.  This oracle takes the reading
 * that keeps the written files those of the GGUF ecosystem the pages read:
 *
 *   Q8_0: the symmetric 8-bit form, exactly the activation quantiser of
 *         quant.c (d = max|x| / 127, codes rounded half away from zero).
 *   Q4_0: m = the value of largest magnitude in the block, with its sign
 *         (the first such element when several tie);
 *         d = m / -8, id = (d == 0 ? 0 : 1 / d),
 *         q_i = trunc(clamp(x_i * id + 8.5, 0, 15));  w = d * (q - 8).
 *         When |d| is below 2^-128, 1 / d overflows; x_i / d (one fp32
 *         division) then stands for x_i * id, so that a zero weight still
 *         lands on code 8 (the quotient is what x_i * id approximates).
 *         The largest-magnitude element lands on code 0 (w = -8 d = m); the
 *         grid reaches +7 d on the other side, where values clamp.
 *   Q5_0: the same with d = m / -16 and q_i = trunc(clamp(x_i * id + 16.5, 0, 31)).
 *
 * Every step is one fp32 IEEE operation (this file is built without FMA
 * contraction), so the integer codes are decided in fp32 as a kernel doing
 * the same steps decides them; fp16(d) (round to nearest even) is stored and
 * is the scale every later dot product uses.  Element order is that of the
 * decoders in blocks.c: elements j and j + 16 share byte j of the nibbles
 * (low and high nibble), and Q5_0 keeps element i's fifth bit in bit i of
 * the little-endian 32-bit qh.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

/* m, the signed value of largest magnitude (the first on ties). */
static float block_extreme(const float* x)
{
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) {
            amax = a;
            m = x[i];
        }
    }
    return m;
}

/* Codes 0 .. 2^bits - 1 of one block; returns d (fp32). */
static float block_codes(const float* x, int bits, uint8_t* q)
{
    const float half = (float)(1 << (bits - 1));   /* 8 or 16 */
    const int top = (1 << bits) - 1;                /* 15 or 31 */
    float m = block_extreme(x);
    float d = m / -half;
    float id = (d == 0.0f) ? 0.0f : 1.0f / d;
    const int overflow = isinf(id);                 /* |d| below 2^-128 */
    for (int i = 0; i < 32; i++) {
        float v = overflow ? x[i] / d : x[i] * id;
        v = v + (half + 0.5f);
        /* clamp in fp32 before truncating (converting an out-of-range float
         * to an integer is undefined in C) */
        if (v > (float)top) v = (float)top;
        if (v < 0.0f) v = 0.0f;
        q[i] = (uint8_t)(int)v;                     /* truncation */
    }
    return d;
}

int orc_quantize_weights(int wtype, const float* w, int64_t n, uint8_t* out)
{
    if (wtype == ORC_Q8_0) return orc_quantize_act(ORC_Q8_0, w, n, out);
    if (wtype != ORC_Q4_0 && wtype != ORC_Q5_0) return ORC_EUNSUP;
    if (n < 0) return ORC_EINVAL;
    if (n % 32) return ORC_ESHAPE;
    const int64_t bb = orc_block_bytes(wtype);
    uint8_t q[32];
    for (int64_t b = 0; b < n / 32; b++) {
        uint8_t* o = out + b * bb;
        float d = block_codes(w + 32 * b, wtype == ORC_Q4_0 ? 4 : 5, q);
        uint16_t h = orc_f32_to_f16_rn(d);
        o[0] = (uint8_t)(h & 0xff);
        o[1] = (uint8_t)(h >> 8);
        uint8_t* qs = o + 2;
        if (wtype == ORC_Q5_0) {
            uint32_t qh = 0;
            for (int i = 0; i < 32; i++) qh |= (uint32_t)((q[i] >> 4) & 1) << i;
            for (int i = 0; i < 4; i++) o[2 + i] = (uint8_t)(qh >> (8 * i));
            qs = o + 6;
        }
        for (int j = 0; j < 16; j++) qs[j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
    }
    return ORC_OK;
}
