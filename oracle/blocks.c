/*
 * blocks.c -- decode one quantised block into exact integer codes and scales.
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Formats: "Models and formats" page, section "Tensor formats" (Q4_0, Q5_0,
 * Q8_0, the K-quants Q4_K and Q6_K, MXFP4); "Architecture" page, section
 * "The package map", pkg/quant ("block layouts, dequantisation").  The pages
 * name the formats without printing their bytes; the layouts below are the
 * GGUF block conventions, read field by field, little-endian:
 *
 *   Q4_0  (18 B / 32 w): fp16 d | 16 bytes of nibbles.  Element j (j < 16) is
 *         the low nibble of byte j, element j+16 its high nibble.  w = d*(q-8).
 *   Q5_0  (22 B / 32 w): fp16 d | u32 high-bit mask | 16 bytes of nibbles.
 *         Nibbles as Q4_0; bit i of the mask is bit 4 of element i.  w = d*(q-16).
 *   Q8_0  (34 B / 32 w): fp16 d | 32 int8.  w = d*q.
 *   Q8_1  (36 B / 32 w): fp16 d | fp16 s | 32 int8.  w = d*q; s is the block's
 *         code sum times d, which only an activation block uses, so a weight
 *         ignores it.
 *   Q4_1  (20 B / 32 w): fp16 d | fp16 m | 16 bytes of nibbles, order as Q4_0.
 *         w = d*q + m (carried below as dmin = -m with sub_min = 1).
 *   Q5_1  (24 B / 32 w): fp16 d | fp16 m | u32 high-bit mask | 16 bytes of
 *         nibbles, bits and order as Q5_0.  w = d*q + m.
 *   MXFP4 (17 B / 32 w): u8 E8M0 exponent e | 16 bytes of E2M1 codes, nibble
 *         order as Q4_0.  w = 2^(e-127) * E2M1(code); e = 255 is NaN (OCP MX).
 *   Q4_K  (144 B / 256 w): fp16 d | fp16 dmin | 12 bytes of packed 6-bit
 *         sub-block scales sc[8] and mins m[8] | 128 bytes of nibbles.
 *         Sub-block j holds elements 32j..32j+31; 32-byte chunk c of the
 *         nibbles holds sub-block 2c in its low nibbles and 2c+1 in its high
 *         nibbles.  w = d*sc_j*q - dmin*m_j.
 *   Q5_K  (176 B / 256 w): fp16 d | fp16 dmin | the 12 scale/min bytes of Q4_K |
 *         32 B of fifth bits | 128 bytes of nibbles laid out as in Q4_K.  The
 *         fifth bit of element 32j+l (sub-block j) is bit j of byte l of the
 *         fifth-bit field.  w = d*sc_j*q - dmin*m_j with 5-bit q.
 *   Q2_K  (84 B / 256 w): 16 scale bytes (low nibble sc, high nibble m) |
 *         64 B of 2-bit codes | fp16 d | fp16 dmin.  Element 128n+32j+l
 *         (n < 2, j < 4, l < 32) is bits 2j..2j+1 of code byte 32n+l and uses
 *         scale byte 8n+2j+(l >= 16).  w = d*sc*q - dmin*m.
 *   Q3_K  (110 B / 256 w): 32 B high-bit mask | 64 B of 2-bit codes | 12 bytes
 *         of sixteen 6-bit scales | fp16 d.  Element 128n+32j+l takes its low
 *         bits as in Q2_K and bit 4n+j of mask byte l; its code is the low
 *         bits minus 4 when that bit is clear.  Scale s (0..15): low 4 bits
 *         from byte s (s < 8, low nibble) or byte s-8 (high nibble), high 2
 *         bits from bits 2*(s/4) of byte 8 + s%4.  w = d*(s6 - 32)*code.
 *   Q6_K  (210 B / 256 w): 128 B low nibbles | 64 B high 2-bit pairs |
 *         int8 scales[16] | fp16 d.  Element i uses scales[i/16].
 *         w = d*sc*(q-32).
 *   F32, F16, BF16: plain little-endian values, one per element ("Models and
 *         formats", "Tensor formats": read and accelerated on every backend).
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

static uint32_t rd_u16(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }
static uint32_t rd_u32(const uint8_t* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

int64_t orc_block_elems(int type)
{
    switch (type) {
    case ORC_Q4_0: case ORC_Q5_0: case ORC_Q8_0: case ORC_MXFP4: case ORC_Q4_1: case ORC_Q5_1: case ORC_Q8_1:
    case ORC_MXFP8:
        return 32;
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: case ORC_Q8_K: case ORC_Q2_K: case ORC_Q3_K: return 256;
    default: return 0;
    }
}

int64_t orc_block_bytes(int type)
{
    switch (type) {
    case ORC_Q4_0: return 18;
    case ORC_Q5_0: return 22;
    case ORC_Q8_0: return 34;
    case ORC_Q8_1: return 36;
    case ORC_Q4_1: return 20;
    case ORC_Q5_1: return 24;
    case ORC_MXFP4: return 17;
    case ORC_MXFP8: return 33;
    case ORC_Q4_K: return 144;
    case ORC_Q5_K: return 176;
    case ORC_Q2_K: return 84;
    case ORC_Q3_K: return 110;
    case ORC_Q6_K: return 210;
    case ORC_Q8_K: return 292;
    default: return 0;
    }
}

/* Nibble k (0..31) of a 16-byte nibble field in the Q4_0 element order. */
static int nibble32(const uint8_t* qs, int k)
{
    return k < 16 ? (qs[k] & 0x0f) : (qs[k - 16] >> 4);
}

/* OCP E2M1: bit 3 sign, bits 2..1 exponent E (bias 1), bit 0 mantissa M.
 * E == 0 is subnormal: 0.5*M; otherwise 2^(E-1)*(1 + M/2).  Returned doubled,
 * which makes every value an integer: {0,1,2,3,4,6,8,12} with sign. */
static int e2m1_doubled(int c)
{
    int s = (c >> 3) & 1;
    int E = (c >> 1) & 3;
    int M = c & 1;
    int mag2;
    if (E == 0) mag2 = M;                       /* 2 * 0.5*M */
    else mag2 = (2 + M) << (E - 1);             /* 2 * 2^(E-1) * (1 + M/2) */
    return s ? -mag2 : mag2;
}

/* Q4_K: the 12-byte field packs eight 6-bit scales and eight 6-bit mins.
 * Bytes 0..3: low 6 bits are sc0..sc3, top 2 bits are bits 4..5 of sc4..sc7.
 * Bytes 4..7: low 6 bits are m0..m3, top 2 bits are bits 4..5 of m4..m7.
 * Bytes 8..11: low nibble is bits 0..3 of sc4..sc7, high nibble of m4..m7. */
static void q4k_scale_min(const uint8_t* f, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = f[j] & 63;
        *m = f[4 + j] & 63;
    } else {
        int t = j - 4;
        *sc = (f[8 + t] & 0x0f) | ((f[t] >> 6) << 4);
        *m = (f[8 + t] >> 4) | ((f[4 + t] >> 6) << 4);
    }
}

int orc_decode_block(int type, const uint8_t* b, orc_block* out)
{
    memset(out, 0, sizeof(*out));
    switch (type) {
    case ORC_Q4_0: {
        out->n = 32;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        for (int i = 0; i < 32; i++) {
            out->code[i] = nibble32(b + 2, i) - 8;
            out->sub_scale[i] = 1;
        }
        return ORC_OK;
    }
    case ORC_Q5_0: {
        out->n = 32;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        uint32_t qh = rd_u32(b + 2);
        for (int i = 0; i < 32; i++) {
            int q = nibble32(b + 6, i) | (int)(((qh >> i) & 1u) << 4);
            out->code[i] = q - 16;
            out->sub_scale[i] = 1;
        }
        return ORC_OK;
    }
    case ORC_Q8_0: {
        out->n = 32;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        for (int i = 0; i < 32; i++) {
            out->code[i] = (int8_t)b[2 + i];
            out->sub_scale[i] = 1;
        }
        return ORC_OK;
    }
    case ORC_Q8_1: {
        out->n = 32;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        for (int i = 0; i < 32; i++) {
            out->code[i] = (int8_t)b[4 + i];
            out->sub_scale[i] = 1;
        }
        return ORC_OK;
    }
    case ORC_Q4_1:
    case ORC_Q5_1: {
        /* w = d*q + m with the unsigned 4- or 5-bit code q */
        out->n = 32;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        out->dmin = -orc_f16_to_f64((uint16_t)rd_u16(b + 2));
        const uint32_t qh = type == ORC_Q5_1 ? rd_u32(b + 4) : 0u;
        const uint8_t* qs = b + (type == ORC_Q5_1 ? 8 : 4);
        for (int i = 0; i < 32; i++) {
            out->code[i] = nibble32(qs, i) | (int)(((qh >> i) & 1u) << 4);
            out->sub_scale[i] = 1;
            out->sub_min[i] = 1;
        }
        return ORC_OK;
    }
    case ORC_MXFP4: {
        out->n = 32;
        int e = b[0];
        /* E8M0: 2^(e-127); the doubled code takes one more factor 1/2. */
        out->d = (e == 255) ? NAN : ldexp(1.0, e - 128);
        for (int i = 0; i < 32; i++) {
            out->code[i] = e2m1_doubled(nibble32(b + 1, i));
            out->sub_scale[i] = 1;
        }
        return ORC_OK;
    }
    case ORC_Q4_K: {
        out->n = 256;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        out->dmin = orc_f16_to_f64((uint16_t)rd_u16(b + 2));
        const uint8_t* scf = b + 4;
        const uint8_t* qs = b + 16;
        for (int j = 0; j < 8; j++) {
            int sc, m;
            q4k_scale_min(scf, j, &sc, &m);
            const uint8_t* chunk = qs + 32 * (j / 2);
            for (int l = 0; l < 32; l++) {
                int q = (j % 2 == 0) ? (chunk[l] & 0x0f) : (chunk[l] >> 4);
                out->code[32 * j + l] = q;
                out->sub_scale[32 * j + l] = sc;
                out->sub_min[32 * j + l] = m;
            }
        }
        return ORC_OK;
    }
    case ORC_Q2_K: {
        out->n = 256;
        const uint8_t* sc = b;
        const uint8_t* qs = b + 16;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b + 80));
        out->dmin = orc_f16_to_f64((uint16_t)rd_u16(b + 82));
        for (int n = 0; n < 2; n++)
            for (int j = 0; j < 4; j++)
                for (int l = 0; l < 32; l++) {
                    const int e = 128 * n + 32 * j + l;
                    const int s = sc[8 * n + 2 * j + (l >= 16)];
                    out->code[e] = (qs[32 * n + l] >> (2 * j)) & 3;
                    out->sub_scale[e] = s & 15;
                    out->sub_min[e] = s >> 4;
                }
        return ORC_OK;
    }
    case ORC_Q3_K: {
        out->n = 256;
        const uint8_t* hm = b;
        const uint8_t* qs = b + 32;
        const uint8_t* sf = b + 96;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b + 108));
        int s6[16];
        for (int s = 0; s < 16; s++) {
            const int lo = s < 8 ? (sf[s] & 15) : (sf[s - 8] >> 4);
            const int hi = (sf[8 + s % 4] >> (2 * (s / 4))) & 3;
            s6[s] = lo | (hi << 4);
        }
        for (int n = 0; n < 2; n++)
            for (int j = 0; j < 4; j++)
                for (int l = 0; l < 32; l++) {
                    const int e = 128 * n + 32 * j + l;
                    const int q = (qs[32 * n + l] >> (2 * j)) & 3;
                    const int h = (hm[l] >> (4 * n + j)) & 1;
                    out->code[e] = q - (h ? 0 : 4);
                    out->sub_scale[e] = s6[8 * n + 2 * j + (l >= 16)] - 32;
                }
        return ORC_OK;
    }
    case ORC_Q5_K: {
        out->n = 256;
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b));
        out->dmin = orc_f16_to_f64((uint16_t)rd_u16(b + 2));
        const uint8_t* scf = b + 4;
        const uint8_t* qh = b + 16;
        const uint8_t* qs = b + 48;
        for (int j = 0; j < 8; j++) {
            int sc, m;
            q4k_scale_min(scf, j, &sc, &m);
            const uint8_t* chunk = qs + 32 * (j / 2);
            for (int l = 0; l < 32; l++) {
                int q = (j % 2 == 0) ? (chunk[l] & 0x0f) : (chunk[l] >> 4);
                q |= ((qh[l] >> j) & 1) << 4;
                out->code[32 * j + l] = q;
                out->sub_scale[32 * j + l] = sc;
                out->sub_min[32 * j + l] = m;
            }
        }
        return ORC_OK;
    }
    case ORC_Q6_K: {
        out->n = 256;
        const uint8_t* ql = b;
        const uint8_t* qh = b + 128;
        const int8_t* scales = (const int8_t*)(b + 192);
        out->d = orc_f16_to_f64((uint16_t)rd_u16(b + 208));
        for (int h = 0; h < 2; h++) {
            const uint8_t* L = ql + 64 * h;
            const uint8_t* H = qh + 32 * h;
            for (int l = 0; l < 32; l++) {
                int e0 = 128 * h + l;
                int q0 = (L[l] & 0x0f) | (((H[l] >> 0) & 3) << 4);
                int q1 = (L[l + 32] & 0x0f) | (((H[l] >> 2) & 3) << 4);
                int q2 = (L[l] >> 4) | (((H[l] >> 4) & 3) << 4);
                int q3 = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
                out->code[e0] = q0 - 32;
                out->code[e0 + 32] = q1 - 32;
                out->code[e0 + 64] = q2 - 32;
                out->code[e0 + 96] = q3 - 32;
            }
        }
        for (int i = 0; i < 256; i++) out->sub_scale[i] = scales[i / 16];
        return ORC_OK;
    }
    default:
        return ORC_EUNSUP;
    }
}

double orc_block_weight(const orc_block* b, int i)
{
    /* Each product below is exact in fp64 (at most 23 significant bits), and
     * so is the difference for the scale ranges the formats can express at
     * any realistic spread of d and dmin. */
    double a = b->d * (double)b->sub_scale[i] * (double)b->code[i];
    double m = b->dmin * (double)b->sub_min[i];
    return a - m;
}

int64_t orc_plain_bytes(int type)
{
    return type == ORC_F32 ? 4 : (type == ORC_F16 || type == ORC_BF16) ? 2 : 0;
}

/* Element i of a plain weight row, exactly. */
double orc_plain_weight(int type, const uint8_t* row, int64_t i)
{
    if (type == ORC_F32) {
        float f;
        memcpy(&f, row + 4 * i, 4);
        return (double)f;
    }
    const uint16_t h = (uint16_t)(row[2 * i] | (row[2 * i + 1] << 8));
    return type == ORC_F16 ? orc_f16_to_f64(h) : orc_bf16_to_f64(h);
}

int orc_dequant(int type, const uint8_t* W, int64_t rows, int64_t cols, float* out)
{
    if (orc_plain_bytes(type)) {
        if (rows < 0 || cols < 0) return ORC_EINVAL;
        for (int64_t r = 0; r < rows; r++)
            for (int64_t c = 0; c < cols; c++)
                out[r * cols + c] = (float)orc_plain_weight(type, W + r * cols * orc_plain_bytes(type), c);
        return ORC_OK;
    }
    int64_t bs = orc_block_elems(type), bb = orc_block_bytes(type);
    if (bs == 0 || type == ORC_Q8_K) return ORC_EUNSUP;
    if (rows < 0 || cols < 0) return ORC_EINVAL;
    if (cols % bs) return ORC_ESHAPE;
    int64_t nb = cols / bs;
    orc_block blk;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t k = 0; k < nb; k++) {
            int rc = orc_decode_block(type, W + (r * nb + k) * bb, &blk);
            if (rc) return rc;
            for (int i = 0; i < bs; i++) out[r * cols + k * bs + i] = (float)orc_block_weight(&blk, i);
        }
    }
    return ORC_OK;
}
