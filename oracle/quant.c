/*
 * quant.c -- activation quantisers to 8-bit blocks.  TEST INFRASTRUCTURE ONLY
 * (see oracle.h).
 *
 * The "Architecture" page ("The package map", pkg/quant) names fused W4A8
 * kernels: 4-bit weights against 8-bit activations.  The pages do not print
 * the activation quantiser; this one takes the plainest symmetric reading,
 * identical for both block sizes:
 *
 *   per block of bs values (bs = 32 for Q8_0, 256 for Q8_K):
 *     amax = max |x_i|                      (fp32)
 *     d    = amax / 127                     (fp32, one rounding)
 *     id   = d == 0 ? 0 : 1 / d             (fp32, one rounding)
 *     q_i  = round half away from zero (x_i * id), clamped to [-127, 127]
 *   When d is below 2^-128 (amax under 127 * 2^-128), 1 / d overflows to
 *   infinity and x_i * id is no longer the scaled value (for x_i = 0 it is
 *   not even a number); the codes of such a block are then taken from the
 *   quotient x_i / d itself (fp32, one rounding), which is the plain
 *   definition q = round(x / d): zero stays zero.
 *   Q8_0 stores fp16(d) (round to nearest even) and q[32]    -> 34 bytes;
 *   Q8_K stores the fp32 d, q[256] and int16 bsums[16], the sums of q over
 *   each run of 16                                           -> 292 bytes.
 * The codes come from the fp32 d; the stored (for Q8_0, fp16-rounded) d is
 * the scale every later dot product uses.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

static void quantize_block(const float* x, int bs, float* d_out, int8_t* q)
{
    float amax = 0.0f;
    for (int i = 0; i < bs; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    float id = (d == 0.0f) ? 0.0f : 1.0f / d;
    const int overflow = isinf(id);             /* d below 2^-128 */
    for (int i = 0; i < bs; i++) {
        float v = overflow ? x[i] / d : x[i] * id;
        float r = roundf(v);                    /* halves away from zero */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
    *d_out = d;
}

int orc_quantize_act(int atype, const float* x, int64_t n, uint8_t* out)
{
    int64_t bs = orc_block_elems(atype), bb = orc_block_bytes(atype);
    if (atype == ORC_MXFP8) return orc_quantize_mxfp8(x, n, out);
    if (atype != ORC_Q8_0 && atype != ORC_Q8_K) return ORC_EUNSUP;
    if (n < 0) return ORC_EINVAL;
    if (n % bs) return ORC_ESHAPE;
    int8_t q[256];
    for (int64_t b = 0; b < n / bs; b++) {
        float d;
        uint8_t* o = out + b * bb;
        quantize_block(x + b * bs, (int)bs, &d, q);
        if (atype == ORC_Q8_0) {
            uint16_t h = orc_f32_to_f16_rn(d);
            o[0] = (uint8_t)(h & 0xff);
            o[1] = (uint8_t)(h >> 8);
            memcpy(o + 2, q, 32);
        } else {
            uint32_t u;
            memcpy(&u, &d, 4);
            for (int i = 0; i < 4; i++) o[i] = (uint8_t)(u >> (8 * i));
            memcpy(o + 4, q, 256);
            for (int g = 0; g < 16; g++) {
                int s = 0;
                for (int i = 0; i < 16; i++) s += q[16 * g + i];
                uint16_t us = (uint16_t)(int16_t)s;
                o[260 + 2 * g] = (uint8_t)(us & 0xff);
                o[261 + 2 * g] = (uint8_t)(us >> 8);
            }
        }
    }
    return ORC_OK;
}

int orc_decode_act_block(int atype, const uint8_t* blk, int32_t* q, double* d, int32_t* bsums)
{
    if (atype == ORC_Q8_0) {
        *d = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
        for (int i = 0; i < 32; i++) q[i] = (int8_t)blk[2 + i];
        return ORC_OK;
    }
    if (atype == ORC_Q8_K) {
        uint32_t u = (uint32_t)blk[0] | ((uint32_t)blk[1] << 8) | ((uint32_t)blk[2] << 16) | ((uint32_t)blk[3] << 24);
        float f;
        memcpy(&f, &u, 4);
        *d = (double)f;
        for (int i = 0; i < 256; i++) q[i] = (int8_t)blk[4 + i];
        if (bsums)
            for (int g = 0; g < 16; g++)
                bsums[g] = (int16_t)(uint16_t)(blk[260 + 2 * g] | (blk[261 + 2 * g] << 8));
        return ORC_OK;
    }
    return ORC_EUNSUP;
}
