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
 *   Q4_1 / Q5_1, Q4_K / Q5_K, Q6_K: one pass of min/max rules per run, no
 *   search (the pages name these formats among those written but print no
 *   procedure, and say a grid search belongs with an importance matrix); see
 *   each function below.
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

/* round half away from zero of an fp32 value (roundf) as an int, after
 * clamping to [lo, hi] in fp32 (converting an out-of-range float is undefined
 * in C) */
static int round_clamp(float v, float lo, float hi)
{
    float r = roundf(v);
    if (r > hi) r = hi;
    if (r < lo) r = lo;
    return (int)r;
}

/* v * (1/s) with id = 1/s precomputed, or v / s itself when 1/s overflowed
 * (reading A18); 0 when s = 0. */
static float scaled(float v, float s, float id)
{
    if (s == 0.0f) return 0.0f;
    return isinf(id) ? v / s : v * id;
}

static void put_f16(uint8_t* o, float v)
{
    uint16_t h = orc_f32_to_f16_rn(v);
    o[0] = (uint8_t)(h & 0xff);
    o[1] = (uint8_t)(h >> 8);
}

/* Q4_1 / Q5_1 (32 w): m = min x, d = (max x - m) / (2^bits - 1); codes
 * q = trunc(clamp((x - m) * (1/d) + 0.5, 0, 2^bits - 1)); w = d*q + m. */
static void quantize_q_1(const float* x, int bits, uint8_t* o)
{
    const int top = (1 << bits) - 1;
    float mn = x[0], mx = x[0];
    for (int i = 1; i < 32; i++) {
        if (x[i] < mn) mn = x[i];
        if (x[i] > mx) mx = x[i];
    }
    const float d = (mx - mn) / (float)top;
    const float id = d == 0.0f ? 0.0f : 1.0f / d;
    uint8_t q[32];
    for (int i = 0; i < 32; i++) {
        float v = scaled(x[i] - mn, d, id) + 0.5f;
        if (v > (float)top) v = (float)top;
        if (v < 0.0f) v = 0.0f;
        q[i] = (uint8_t)(int)v;
    }
    put_f16(o, d);
    put_f16(o + 2, mn);
    uint8_t* qs = o + 4;
    if (bits == 5) {
        uint32_t qh = 0;
        for (int i = 0; i < 32; i++) qh |= (uint32_t)((q[i] >> 4) & 1) << i;
        for (int i = 0; i < 4; i++) o[4 + i] = (uint8_t)(qh >> (8 * i));
        qs = o + 8;
    }
    for (int j = 0; j < 16; j++) qs[j] = (uint8_t)((q[j] & 15) | ((q[j + 16] & 15) << 4));
}

/* Q4_K / Q5_K (256 w, eight sub-blocks of 32, codes 0..top, top = 15 or 31):
 *   lo_j = min(0, min x), s_j = (max x - lo_j) / top, z_j = -lo_j;
 *   d = max_j s_j / 63, dmin = max_j z_j / 63 (fp32);
 *   sc_j = round(s_j / d), m_j = round(z_j / dmin), clamped to 0..63;
 *   with the stored fp16 d, dmin: D_j = d*sc_j, M_j = dmin*m_j (exact) and
 *   q = round((x + M_j) / D_j) clamped to 0..top (0 when D_j = 0);
 *   w = D_j*q - M_j.  Every division is a multiplication by the fp32
 *   reciprocal (reading A18 when it overflows); rounding is half away from
 *   zero. */
static void quantize_q45k(const float* x, int bits, uint8_t* o)
{
    const int top = (1 << bits) - 1;
    float s[8], z[8], smax = 0.0f, zmax = 0.0f;
    for (int j = 0; j < 8; j++) {
        float mn = 0.0f, mx = x[32 * j];
        for (int i = 0; i < 32; i++) {
            const float v = x[32 * j + i];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        s[j] = (mx - mn) / (float)top;
        z[j] = -mn;
        if (s[j] > smax) smax = s[j];
        if (z[j] > zmax) zmax = z[j];
    }
    const float d = smax / 63.0f, dmin = zmax / 63.0f;
    const float id = d == 0.0f ? 0.0f : 1.0f / d, idm = dmin == 0.0f ? 0.0f : 1.0f / dmin;
    int sc[8], m[8];
    for (int j = 0; j < 8; j++) {
        sc[j] = round_clamp(scaled(s[j], d, id), 0.0f, 63.0f);
        m[j] = round_clamp(scaled(z[j], dmin, idm), 0.0f, 63.0f);
    }
    put_f16(o, d);
    put_f16(o + 2, dmin);
    const float dst = (float)orc_f16_to_f64(orc_f32_to_f16_rn(d));
    const float dmst = (float)orc_f16_to_f64(orc_f32_to_f16_rn(dmin));
    uint8_t* f = o + 4;
    for (int j = 0; j < 4; j++) {
        f[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        f[4 + j] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        f[8 + j] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t q[256];
    for (int j = 0; j < 8; j++) {
        const float D = dst * (float)sc[j], M = dmst * (float)m[j];
        const float iD = D == 0.0f ? 0.0f : 1.0f / D;
        for (int i = 0; i < 32; i++)
            q[32 * j + i] = (uint8_t)round_clamp(scaled(x[32 * j + i] + M, D, iD), 0.0f, (float)top);
    }
    uint8_t* qh = o + 16;                    /* Q5_K only */
    uint8_t* qs = o + (bits == 5 ? 48 : 16);
    if (bits == 5) memset(qh, 0, 32);
    for (int c = 0; c < 4; c++)
        for (int l = 0; l < 32; l++) {
            const int a = q[64 * c + l], b = q[64 * c + 32 + l];
            qs[32 * c + l] = (uint8_t)((a & 15) | ((b & 15) << 4));
            if (bits == 5) qh[l] |= (uint8_t)(((a >> 4) & 1) << (2 * c)) | (uint8_t)(((b >> 4) & 1) << (2 * c + 1));
        }
}

/* Q6_K (256 w, sixteen runs of 16, codes 0..63, w = d*sc*(q - 32)):
 *   per run j the signed value of largest magnitude m_j (the first on ties),
 *   s_j = m_j / -32; the s_j of largest magnitude s_e (the first on ties),
 *   d = s_e / -128 (fp32); sc_j = round(s_j / d) clamped to -128..127;
 *   with the stored fp16 d: D_j = d*sc_j (exact) and
 *   q = round(x / D_j) + 32 clamped to 0..63 (32 when D_j = 0).  The run
 *   extreme lands on code 0 (-32 D_j), the super-block extreme scale on -128. */
static void quantize_q6k(const float* x, uint8_t* o)
{
    float s[16], se = 0.0f;
    for (int j = 0; j < 16; j++) {
        float a = 0.0f, m = 0.0f;
        for (int i = 0; i < 16; i++) {
            const float v = x[16 * j + i];
            if (fabsf(v) > a) {
                a = fabsf(v);
                m = v;
            }
        }
        s[j] = m / -32.0f;
        if (fabsf(s[j]) > fabsf(se)) se = s[j];
    }
    const float d = se / -128.0f;
    const float id = d == 0.0f ? 0.0f : 1.0f / d;
    int sc[16];
    for (int j = 0; j < 16; j++) sc[j] = round_clamp(scaled(s[j], d, id), -128.0f, 127.0f);
    const float dst = (float)orc_f16_to_f64(orc_f32_to_f16_rn(d));
    uint8_t q[256];
    for (int j = 0; j < 16; j++) {
        const float D = dst * (float)sc[j];
        const float iD = D == 0.0f ? 0.0f : 1.0f / D;
        for (int i = 0; i < 16; i++)
            q[16 * j + i] = (uint8_t)(round_clamp(scaled(x[16 * j + i], D, iD), -32.0f, 31.0f) + 32);
    }
    uint8_t* ql = o;
    uint8_t* qh = o + 128;
    memset(o, 0, 192);
    for (int h = 0; h < 2; h++)
        for (int l = 0; l < 32; l++) {
            const int e = 128 * h + l;
            const int q0 = q[e], q1 = q[e + 32], q2 = q[e + 64], q3 = q[e + 96];
            ql[64 * h + l] = (uint8_t)((q0 & 15) | ((q2 & 15) << 4));
            ql[64 * h + l + 32] = (uint8_t)((q1 & 15) | ((q3 & 15) << 4));
            qh[32 * h + l] = (uint8_t)((q0 >> 4) | ((q1 >> 4) << 2) | ((q2 >> 4) << 4) | ((q3 >> 4) << 6));
        }
    for (int j = 0; j < 16; j++) o[192 + j] = (uint8_t)(int8_t)sc[j];
    put_f16(o + 208, d);
}

int orc_quantize_weights(int wtype, const float* w, int64_t n, uint8_t* out)
{
    if (wtype == ORC_Q8_0) return orc_quantize_act(ORC_Q8_0, w, n, out);
    if (wtype == ORC_Q4_1 || wtype == ORC_Q5_1 || wtype == ORC_Q4_K || wtype == ORC_Q5_K || wtype == ORC_Q6_K) {
        const int64_t bs = orc_block_elems(wtype), bb = orc_block_bytes(wtype);
        if (n < 0) return ORC_EINVAL;
        if (n % bs) return ORC_ESHAPE;
        for (int64_t b = 0; b < n / bs; b++) {
            if (wtype == ORC_Q4_1 || wtype == ORC_Q5_1)
                quantize_q_1(w + bs * b, wtype == ORC_Q4_1 ? 4 : 5, out + bb * b);
            else if (wtype == ORC_Q6_K)
                quantize_q6k(w + bs * b, out + bb * b);
            else
                quantize_q45k(w + bs * b, wtype == ORC_Q4_K ? 4 : 5, out + bb * b);
        }
        return ORC_OK;
    }
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
