// formats.cuh -- per-format decoding of weight "units" and their fused dot
// products with staged activations.
//
// Formats ("Models and formats" page, "Tensor formats"; GGUF block layouts):
//   Q4_0  18 B / 32 w   fp16 d | 16 B nibbles              w = d*(q-8)
//   Q5_0  22 B / 32 w   fp16 d | u32 fifth bits | 16 B     w = d*(q-16)
//   Q8_0  34 B / 32 w   fp16 d | int8[32]                  w = d*q
//   MXFP4 17 B / 32 w   E8M0 e | 16 B E2M1 codes           w = 2^(e-127)*E2M1(q)
//   Q4_K 144 B / 256 w  fp16 d | fp16 dmin | 12 B six-bit sc/m | 128 B nibbles
//                                                          w = d*sc_j*q - dmin*m_j
//   Q6_K 210 B / 256 w  128 B low nibbles | 64 B high pairs | int8 sc[16] | fp16 d
//                                                          w = d*sc*(q-32)
//   Q4_1  20 B / 32 w   fp16 d | fp16 m | 16 B nibbles     w = d*q + m
//   Q5_1  24 B / 32 w   fp16 d | fp16 m | u32 fifth bits | 16 B   w = d*q + m
//   Q8_1  36 B / 32 w   fp16 d | fp16 s (unused) | int8[32]  w = d*q
//   Q5_K 176 B / 256 w  Q4_K's d, dmin, 12 B sc/m | 32 B fifth bits | 128 B nibbles
//   Q2_K  84 B / 256 w  16 B sc|m nibbles per 16 | 64 B 2-bit codes | fp16 d | fp16 dmin
//   Q3_K 110 B / 256 w  32 B high bits | 64 B 2-bit codes | 12 B 6-bit scales | fp16 d
//   F32, F16, BF16      plain values (fp32 activations only), units of 8
// Nibble order: element j of a 32-run is the low nibble of byte j, element
// j+16 its high nibble; Q4_K 32-byte chunk c holds sub-block 2c (low) and
// 2c+1 (high); Q6_K element i uses scales[i/16].
//
// A unit is the piece of a row one lane handles at a time: one block (32 w)
// for the 32-element formats, 64 weights for the K-quants (Q4_K: one 32-byte
// nibble chunk = two sub-blocks; Q6_K: the l-half lh of half h, i.e. the 16
// consecutive elements at offsets 32g + 16lh, g = 0..3, of that half).
//
// The W4A8 ("fused W4A8 kernels", "Architecture" page, pkg/quant) product of a
// unit is exact in integers: codes are laid out as bytes that line up with the
// staged int8 activations and summed with dp4a; offsets (q-8, q-16, q-32) are
// applied through the exact activation sums.  The scales enter once per unit
// through fixed fp32 fused multiply-adds, so the reduction order of an output
// depends only on the row, never on how many vectors share the pass.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace qmv {

// ---- staged activations -------------------------------------------------------
// Layout in shared memory for G vectors (all arrays 16-byte aligned):
//   A8:  codes int8 [G][cols] (MXFP4: each 32-run interleaved as x0,x16,x1,x17,..)
//        d     f32  [G][nb]         (activation block scale)
//        sum32 i32  [G][nb]         (32-element formats: sum of the block's codes)
//        bsum  i16  [G][nb][16]     (K-quants: sums of each run of 16 codes)
//   A32: xf    f32  [G][cols]       (MXFP4 runs interleaved as above)
//        xs32  f32  [G][cols/32]    (Q4_K: sum of each 32-run, fixed order)
struct XView {
    const uint8_t* codes;
    const float* d;
    const int* sum32;
    const int16_t* bsum;
    const float* xf;
    const float* xs32;
    int cols;
    int nb;   // activation blocks per vector (= weight blocks per row)
};

// Staged 8-bit activations of the K-quants: each 256-element block takes
// kKPitch bytes, one 80-byte slot (64 codes + 16 of padding) per 64-element
// unit, so that consecutive lanes, which decode consecutive units, read 16-byte
// chunks 80 bytes apart (no shared-memory bank conflicts).  The unit slot holds
// the unit's elements in this order: Q4_K unit c = elements 64c..64c+63;
// Q6_K unit (h, lh) = elements 128h + 32g + 16lh + j for g = 0..3, j = 0..15.
// Position of 16-element run r (elements 16r..16r+15) of a block:
constexpr int kKPitch = 320;
// Staged 8-bit activations of the 32-element formats: kBPitch bytes per block
// (32 codes + 16 of padding), so that consecutive lanes' 16-byte loads land in
// distinct banks.
constexpr int kBPitch = 48;
template <int T>
__host__ __device__ constexpr int kquant_run_pos(int r)
{
    if constexpr (T == QMV_Q6_K) return 80 * (2 * (r >> 3) + (r & 1)) + 16 * ((r & 7) >> 1);   // h = r/8, g = (r%8)/2, lh = r%2
    else return 80 * (r >> 2) + 16 * (r & 3);   // unit u = elements 64u .. 64u+63 in order
}


template <int T>
struct Fmt;

// ------------------------------------------------------------------------------
// The 32-element formats share one shape: 8 code words + one scale per unit.
// ------------------------------------------------------------------------------
struct W32 {
    uint32_t c[8];   // 32 code bytes in staged-activation order
    float d;         // w = d * (code - OFF)
    __device__ __forceinline__ uint32_t code(int k) const { return c[k]; }
};

template <int T>
struct Fmt32Base {
    static constexpr int BS = 32, UE = 32, UPB = 1;
    static constexpr bool MIN = false;   // a per-block offset m (w = d*q + m)

    struct XA8 {
        uint32_t w[8];
        float d;
        int sum;
    };

    static __device__ __forceinline__ void load_x_a8(const XView& X, int v, int b, int /*sub*/, XA8& x)
    {
        const uint4* p = reinterpret_cast<const uint4*>(X.codes + ((size_t)v * X.nb + b) * kBPitch);
        const uint4 a = p[0], c = p[1];
        x.w[0] = a.x; x.w[1] = a.y; x.w[2] = a.z; x.w[3] = a.w;
        x.w[4] = c.x; x.w[5] = c.y; x.w[6] = c.z; x.w[7] = c.w;
        x.d = X.d[v * X.nb + b];
        x.sum = X.sum32[v * X.nb + b];
    }
};

template <>
struct Fmt<QMV_Q4_0> : Fmt32Base<QMV_Q4_0> {
    static constexpr int BB = 18, OFF = 8;
    static constexpr bool SIGNED = false;
    using W = W32;
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        uint32_t q[4];
        load_words<4>(blk + 2, q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.c[k] = q[k] & 0x0f0f0f0fu;
            w.c[4 + k] = (q[k] >> 4) & 0x0f0f0f0fu;
        }
        w.d = half_bits_to_float(ld_u16(blk));
    }
};

template <>
struct Fmt<QMV_Q5_0> : Fmt32Base<QMV_Q5_0> {
    static constexpr int BB = 22, OFF = 16;
    static constexpr bool SIGNED = false;
    using W = W32;
    // Four bits of the mask -> bit 4 of four bytes.  t * 0x00204081 places bit
    // j of t at bit 8j (and elsewhere, never overlapping bits 0, 8, 16, 24).
    static __device__ __forceinline__ uint32_t spread4(uint32_t t)
    {
        return ((t * 0x00204081u) & 0x01010101u) << 4;
    }
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        uint32_t q[5];
        load_words<5>(blk + 2, q);   // q[0] = fifth-bit mask, q[1..4] = nibbles
        const uint32_t qh = q[0];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.c[k] = (q[1 + k] & 0x0f0f0f0fu) | spread4((qh >> (4 * k)) & 15u);
            w.c[4 + k] = ((q[1 + k] >> 4) & 0x0f0f0f0fu) | spread4((qh >> (16 + 4 * k)) & 15u);
        }
        w.d = half_bits_to_float(ld_u16(blk));
    }
};

template <>
struct Fmt<QMV_Q8_0> : Fmt32Base<QMV_Q8_0> {
    static constexpr int BB = 34, OFF = 0;
    static constexpr bool SIGNED = true;
    using W = W32;
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        load_words<8>(blk + 2, w.c);
        w.d = half_bits_to_float(ld_u16(blk));
    }
};

// MXFP4: E2M1 codes become the doubled values {0,1,2,3,4,6,8,12} (exact
// integers) with their sign, through byte-permute tables; the doubling is
// undone by using 2^(e-128) as the block scale.
template <>
struct Fmt<QMV_MXFP4> : Fmt32Base<QMV_MXFP4> {
    static constexpr int BB = 17, OFF = 0;
    static constexpr bool SIGNED = true;
    // The block's 16 code bytes as loaded (four words, nibbles in GGUF order)
    // and the signed code words c (c[2k] from the low half of q[k], c[2k+1]
    // from its high half).  The 8-bit product with one or two vectors reads q
    // only (ints32 below), so c is never formed there; with more vectors each
    // signed word serves every vector.
    struct W {
        uint32_t q[4];
        uint32_t c[8];
        float d;
        __device__ __forceinline__ uint32_t code(int k) const { return c[k]; }
    };
    // Four nibbles (16 bits) -> four signed bytes.
    static __device__ __forceinline__ uint32_t lut4(uint32_t s)
    {
        const uint32_t sel = s & 0x7777u;
        const uint32_t pos = __byte_perm(0x03020100u, 0x0c080604u, sel);   // 0,1,2,3 | 4,6,8,12
        const uint32_t neg = __byte_perm(0xfdfeff00u, 0xf4f8fafcu, sel);   // 0,-1,-2,-3 | -4,-6,-8,-12
        // 0xff in the bytes whose nibble has its sign bit (bit 3) set: with
        // bit 3 of a selector nibble set, prmt.b32 replicates bit 7 of the
        // selected byte.  (The __byte_perm intrinsic only honours 3-bit
        // selectors, so this one is written in PTX.)
        uint32_t m;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(m) : "r"(s << 4), "r"(s), "r"(0xd9c8u));
        return (pos & ~m) | (neg & m);
    }
    static __device__ __forceinline__ float e8m0_half(uint32_t e)   // 2^(e-128)
    {
        if (e == 255u) return __int_as_float(0x7fc00000);
        if (e >= 2u) return __int_as_float(static_cast<int>((e - 1u) << 23));
        return __int_as_float(static_cast<int>(0x00400000u >> (1u - e)));
    }
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        load_words<4>(blk + 1, w.q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.c[2 * k] = lut4(w.q[k] & 0xffffu);
            w.c[2 * k + 1] = lut4(w.q[k] >> 16);
        }
        w.d = e8m0_half(blk[0]);
    }
    // Magnitudes (doubled E2M1: 0,1,2,3,4,6,8,12) of the four codes of a
    // 16-bit nibble group whose sign bit is clear, 0 where it is set: prmt.b32
    // selects byte (code & 7) of the table, and a set bit 3 of a selector
    // nibble replicates that byte's bit 7, which is 0 in every entry.  With the
    // sign bits flipped first, the same gives the negative codes' magnitudes.
    static __device__ __forceinline__ uint32_t mag4(uint32_t s)
    {
        uint32_t m;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(m) : "r"(0x03020100u), "r"(0x0c080604u), "r"(s));
        return m;
    }
};

// Q4_1 / Q5_1: unsigned codes with a per-block offset, w = d*q + m.  The
// offset enters through the exact sum of the block's activation codes.
struct W32M {
    uint32_t c[8];   // 32 code bytes
    float d, m;
    __device__ __forceinline__ uint32_t code(int k) const { return c[k]; }
};

template <>
struct Fmt<QMV_Q4_1> : Fmt32Base<QMV_Q4_1> {
    static constexpr int BB = 20, OFF = 0;
    static constexpr bool SIGNED = false, MIN = true;
    using W = W32M;
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        uint32_t q[4];
        load_words<4>(blk + 4, q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.c[k] = q[k] & 0x0f0f0f0fu;
            w.c[4 + k] = (q[k] >> 4) & 0x0f0f0f0fu;
        }
        w.d = half_bits_to_float(ld_u16(blk));
        w.m = half_bits_to_float(ld_u16(blk + 2));
    }
};

template <>
struct Fmt<QMV_Q5_1> : Fmt32Base<QMV_Q5_1> {
    static constexpr int BB = 24, OFF = 0;
    static constexpr bool SIGNED = false, MIN = true;
    using W = W32M;
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        uint32_t q[5];
        load_words<5>(blk + 4, q);   // q[0] = fifth-bit mask, q[1..4] = nibbles
        const uint32_t qh = q[0];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.c[k] = (q[1 + k] & 0x0f0f0f0fu) | Fmt<QMV_Q5_0>::spread4((qh >> (4 * k)) & 15u);
            w.c[4 + k] = ((q[1 + k] >> 4) & 0x0f0f0f0fu) | Fmt<QMV_Q5_0>::spread4((qh >> (16 + 4 * k)) & 15u);
        }
        w.d = half_bits_to_float(ld_u16(blk));
        w.m = half_bits_to_float(ld_u16(blk + 2));
    }
};

// Q8_1 as a weight: Q8_0's codes and scale; the second fp16 field (the block's
// code sum times d) serves activation blocks only and is not read.
template <>
struct Fmt<QMV_Q8_1> : Fmt32Base<QMV_Q8_1> {
    static constexpr int BB = 36, OFF = 0;
    static constexpr bool SIGNED = true;
    using W = W32;
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        load_words<8>(blk + 4, w.c);
        w.d = half_bits_to_float(ld_u16(blk));
    }
};

// ------------------------------------------------------------------------------
// Q4_K: unit = 32-byte nibble chunk c of a super-block (sub-blocks 2c, 2c+1).
// ------------------------------------------------------------------------------
template <>
struct Fmt<QMV_Q4_K> {
    static constexpr int BS = 256, BB = 144, UE = 64, UPB = 4;
    struct W {
        uint32_t lo[8], hi[8];
        int sc0, sc1, m0, m1;
        float d, dmin;
    };
    static __device__ __forceinline__ uint32_t fbyte(uint32_t f0, uint32_t f1, uint32_t f2, int i)
    {
        const uint32_t w = i < 4 ? f0 : (i < 8 ? f1 : f2);
        return (w >> (8 * (i & 3))) & 0xffu;
    }
    // Six-bit scale and min of sub-block j from the 12-byte field.
    static __device__ __forceinline__ void scale_min(uint32_t f0, uint32_t f1, uint32_t f2, int j, int& sc, int& m)
    {
        if (j < 4) {
            sc = fbyte(f0, f1, f2, j) & 63;
            m = fbyte(f0, f1, f2, j + 4) & 63;
        } else {
            const uint32_t lo4 = fbyte(f0, f1, f2, j + 4);
            sc = (lo4 & 15) | ((fbyte(f0, f1, f2, j - 4) >> 6) << 4);
            m = (lo4 >> 4) | ((fbyte(f0, f1, f2, j) >> 6) << 4);
        }
    }
    // blk is 16-byte aligned (144-byte blocks in a 16-byte aligned staging slot).
    static __device__ __forceinline__ void load(const uint8_t* blk, int c, W& w)
    {
        const uint4 h = *reinterpret_cast<const uint4*>(blk);   // d, dmin, field[0..11]
        const uint4* qp = reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
        const uint4 a = qp[0], b = qp[1];
        const uint32_t q[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            w.lo[k] = q[k] & 0x0f0f0f0fu;
            w.hi[k] = (q[k] >> 4) & 0x0f0f0f0fu;
        }
        scale_min(h.y, h.z, h.w, 2 * c, w.sc0, w.m0);
        scale_min(h.y, h.z, h.w, 2 * c + 1, w.sc1, w.m1);
        w.d = half_bits_to_float(h.x & 0xffffu);
        w.dmin = half_bits_to_float(h.x >> 16);
    }
    struct XA8 {
        uint32_t lo[8], hi[8];
        float d;
        int s0, s1;   // sums of the codes of sub-blocks 2c and 2c+1
    };
    static __device__ __forceinline__ void load_x_a8(const XView& X, int v, int b, int c, XA8& x)
    {
        const uint4* p = reinterpret_cast<const uint4*>(X.codes + ((size_t)v * X.nb + b) * kKPitch + 80 * c);
        const uint4 a0 = p[0], a1 = p[1], a2 = p[2], a3 = p[3];
        x.lo[0] = a0.x; x.lo[1] = a0.y; x.lo[2] = a0.z; x.lo[3] = a0.w;
        x.lo[4] = a1.x; x.lo[5] = a1.y; x.lo[6] = a1.z; x.lo[7] = a1.w;
        x.hi[0] = a2.x; x.hi[1] = a2.y; x.hi[2] = a2.z; x.hi[3] = a2.w;
        x.hi[4] = a3.x; x.hi[5] = a3.y; x.hi[6] = a3.z; x.hi[7] = a3.w;
        x.d = X.d[v * X.nb + b];
        const uint2 bs = *reinterpret_cast<const uint2*>(X.bsum + ((size_t)v * X.nb + b) * 16 + 4 * c);
        x.s0 = (int)(int16_t)(bs.x & 0xffffu) + (int)(int16_t)(bs.x >> 16);
        x.s1 = (int)(int16_t)(bs.y & 0xffffu) + (int)(int16_t)(bs.y >> 16);
    }
    static __device__ __forceinline__ void ints(const W& w, const XA8& x, int& S, int& Mn)
    {
        int i0 = 0, i1 = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            i0 = dp4a_us(w.lo[k], x.lo[k], i0);
            i1 = dp4a_us(w.hi[k], x.hi[k], i1);
        }
        S = w.sc0 * i0 + w.sc1 * i1;
        Mn = w.m0 * x.s0 + w.m1 * x.s1;
    }
    static __device__ __forceinline__ void acc_a8(const W& w, const XA8& x, float& acc)
    {
        int S, Mn;
        ints(w, x, S, Mn);
        acc = __fmaf_rn((float)S, w.d * x.d, acc);
        acc = __fmaf_rn(-(float)Mn, w.dmin * x.d, acc);
    }
    static __device__ __forceinline__ void acc_a32(const W& w, const XView& X, int v, int b, int c, float& acc)
    {
        const float4* xp = reinterpret_cast<const float4*>(X.xf + (size_t)v * X.cols + (size_t)b * 256 + 64 * c);
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 xa = xp[k], xb = xp[8 + k];
            p0 = __fmaf_rn(ubyte_to_float_minus(w.lo[k], 0, 8388608.f), xa.x, p0);
            p0 = __fmaf_rn(ubyte_to_float_minus(w.lo[k], 1, 8388608.f), xa.y, p0);
            p0 = __fmaf_rn(ubyte_to_float_minus(w.lo[k], 2, 8388608.f), xa.z, p0);
            p0 = __fmaf_rn(ubyte_to_float_minus(w.lo[k], 3, 8388608.f), xa.w, p0);
            p1 = __fmaf_rn(ubyte_to_float_minus(w.hi[k], 0, 8388608.f), xb.x, p1);
            p1 = __fmaf_rn(ubyte_to_float_minus(w.hi[k], 1, 8388608.f), xb.y, p1);
            p1 = __fmaf_rn(ubyte_to_float_minus(w.hi[k], 2, 8388608.f), xb.z, p1);
            p1 = __fmaf_rn(ubyte_to_float_minus(w.hi[k], 3, 8388608.f), xb.w, p1);
        }
        const float* xs = X.xs32 + (size_t)v * (X.cols / 32) + (size_t)b * 8 + 2 * c;
        acc = __fmaf_rn(p0, w.d * (float)w.sc0, acc);
        acc = __fmaf_rn(p1, w.d * (float)w.sc1, acc);
        acc = __fmaf_rn(-xs[0], w.dmin * (float)w.m0, acc);
        acc = __fmaf_rn(-xs[1], w.dmin * (float)w.m1, acc);
    }
};

// ------------------------------------------------------------------------------
// Q6_K: unit (h, lh) = elements 128h + 32g + 16lh + [0,16) for g = 0..3.
// ------------------------------------------------------------------------------
template <>
struct Fmt<QMV_Q6_K> {
    static constexpr int BS = 256, BB = 210, UE = 64, UPB = 4;
    struct W {
        uint32_t g[4][4];   // 6-bit codes (0..63) of group g, 16 elements as 4 words
        int sc[4];          // scale of group g: scales[8h + 2g + lh]
        float d;
    };
    static __device__ __forceinline__ void load(const uint8_t* blk, int sub, W& w)
    {
        const int h = sub >> 1, lh = sub & 1;
        uint32_t L0[4], L1[4], H[4], S[2];
        load_words<4>(blk + 64 * h + 16 * lh, L0);        // ql[l],    l = 16lh..16lh+15
        load_words<4>(blk + 64 * h + 32 + 16 * lh, L1);   // ql[l+32]
        load_words<4>(blk + 128 + 32 * h + 16 * lh, H);   // qh[l]
        load_words<2>(blk + 192 + 8 * h, S);              // this half's 8 int8 scales
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w.g[0][k] = (L0[k] & 0x0f0f0f0fu) | ((H[k] & 0x03030303u) << 4);
            w.g[1][k] = (L1[k] & 0x0f0f0f0fu) | ((H[k] & 0x0c0c0c0cu) << 2);
            w.g[2][k] = ((L0[k] >> 4) & 0x0f0f0f0fu) | (H[k] & 0x30303030u);
            w.g[3][k] = ((L1[k] >> 4) & 0x0f0f0f0fu) | ((H[k] & 0xc0c0c0c0u) >> 2);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int idx = 2 * g + lh;   // 0..7 within the half
            const uint32_t word = idx < 4 ? S[0] : S[1];
            w.sc[g] = (int)(int8_t)((word >> (8 * (idx & 3))) & 0xffu);
        }
        w.d = half_bits_to_float(ld_u16(blk + 208));
    }
    struct XA8 {
        uint32_t g[4][4];
        float d;
        int s[4];   // sums of the 16 codes of each group
    };
    static __device__ __forceinline__ void load_x_a8(const XView& X, int v, int b, int sub, XA8& x)
    {
        const int h = sub >> 1, lh = sub & 1;
        const uint8_t* base = X.codes + ((size_t)v * X.nb + b) * kKPitch + 80 * sub;
        const int16_t* bs = X.bsum + ((size_t)v * X.nb + b) * 16 + 8 * h + lh;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint4 a = *reinterpret_cast<const uint4*>(base + 16 * g);
            x.g[g][0] = a.x; x.g[g][1] = a.y; x.g[g][2] = a.z; x.g[g][3] = a.w;
            x.s[g] = bs[2 * g];
        }
        x.d = X.d[v * X.nb + b];
    }
    static __device__ __forceinline__ void ints(const W& w, const XA8& x, int& S, int& Mn)
    {
        S = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            int dot = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) dot = dp4a_us(w.g[g][k], x.g[g][k], dot);
            S += w.sc[g] * (dot - 32 * x.s[g]);
        }
        Mn = 0;
    }
    static __device__ __forceinline__ void acc_a8(const W& w, const XA8& x, float& acc)
    {
        int S, Mn;
        ints(w, x, S, Mn);
        acc = __fmaf_rn((float)S, w.d * x.d, acc);
    }
    static __device__ __forceinline__ void acc_a32(const W& w, const XView& X, int v, int b, int sub, float& acc)
    {
        const int h = sub >> 1, lh = sub & 1;
        const float* xb = X.xf + (size_t)v * X.cols + (size_t)b * 256 + 128 * h + 16 * lh;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4* xp = reinterpret_cast<const float4*>(xb + 32 * g);
            float p = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 xa = xp[k];
                p = __fmaf_rn(ubyte_to_float_minus(w.g[g][k], 0, 8388640.f), xa.x, p);
                p = __fmaf_rn(ubyte_to_float_minus(w.g[g][k], 1, 8388640.f), xa.y, p);
                p = __fmaf_rn(ubyte_to_float_minus(w.g[g][k], 2, 8388640.f), xa.z, p);
                p = __fmaf_rn(ubyte_to_float_minus(w.g[g][k], 3, 8388640.f), xa.w, p);
            }
            acc = __fmaf_rn(p, w.d * (float)w.sc[g], acc);
        }
    }
};

// ------------------------------------------------------------------------------
// Q5_K: Q4_K's fields plus a 32-byte field of fifth bits (bit j of byte l is the
// fifth bit of element 32j + l); units, staging and products are Q4_K's, with
// 5-bit codes.
// ------------------------------------------------------------------------------
template <>
struct Fmt<QMV_Q5_K> : Fmt<QMV_Q4_K> {
    static constexpr int BB = 176;
    // blk is 16-byte aligned (176-byte blocks in a 16-byte aligned staging slot).
    static __device__ __forceinline__ void load(const uint8_t* blk, int c, W& w)
    {
        const uint4 h = *reinterpret_cast<const uint4*>(blk);   // d, dmin, field[0..11]
        const uint4* hp = reinterpret_cast<const uint4*>(blk + 16);
        const uint4* qp = reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
        const uint4 h0 = hp[0], h1 = hp[1], a = qp[0], b = qp[1];
        const uint32_t q[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const uint32_t qh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            w.lo[k] = (q[k] & 0x0f0f0f0fu) | (((qh[k] >> (2 * c)) & 0x01010101u) << 4);
            w.hi[k] = ((q[k] >> 4) & 0x0f0f0f0fu) | (((qh[k] >> (2 * c + 1)) & 0x01010101u) << 4);
        }
        scale_min(h.y, h.z, h.w, 2 * c, w.sc0, w.m0);
        scale_min(h.y, h.z, h.w, 2 * c + 1, w.sc1, w.m1);
        w.d = half_bits_to_float(h.x & 0xffffu);
        w.dmin = half_bits_to_float(h.x >> 16);
    }
};

// ------------------------------------------------------------------------------
// Q2_K and Q3_K: 2-bit code planes.  Element 128n + 32j + l (n < 2, j < 4,
// l < 32) takes bits 2j..2j+1 of code byte 32n + l.  Unit u = elements
// 64u .. 64u+63 (n = u/2, j = 2(u%2) + j', j' < 2): four 16-element runs, each
// with its own scale (run r = 2j' + half, block run 4u + r).
// ------------------------------------------------------------------------------
struct WK2 {
    uint32_t c[2][8];   // codes of elements 64u + 32j' + 4k .. +3 as bytes
    int sc[4], m[4];    // per run: scale and min (Q3_K: signed scale, no min)
    float d, dmin;
};

struct XK2 {
    uint32_t c[2][8];
    float d;
    int s[4];   // sums of the codes of each run
};

template <int T>
struct FmtK2Base {
    static constexpr int BS = 256, UE = 64, UPB = 4;
    using W = WK2;
    using XA8 = XK2;
    static __device__ __forceinline__ void load_x_a8(const XView& X, int v, int b, int u, XA8& x)
    {
        const uint4* p = reinterpret_cast<const uint4*>(X.codes + ((size_t)v * X.nb + b) * kKPitch + 80 * u);
        const uint4 a0 = p[0], a1 = p[1], a2 = p[2], a3 = p[3];
        x.c[0][0] = a0.x; x.c[0][1] = a0.y; x.c[0][2] = a0.z; x.c[0][3] = a0.w;
        x.c[0][4] = a1.x; x.c[0][5] = a1.y; x.c[0][6] = a1.z; x.c[0][7] = a1.w;
        x.c[1][0] = a2.x; x.c[1][1] = a2.y; x.c[1][2] = a2.z; x.c[1][3] = a2.w;
        x.c[1][4] = a3.x; x.c[1][5] = a3.y; x.c[1][6] = a3.z; x.c[1][7] = a3.w;
        x.d = X.d[v * X.nb + b];
        const uint2 bs = *reinterpret_cast<const uint2*>(X.bsum + ((size_t)v * X.nb + b) * 16 + 4 * u);
        x.s[0] = (int)(int16_t)(bs.x & 0xffffu);
        x.s[1] = (int)(int16_t)(bs.x >> 16);
        x.s[2] = (int)(int16_t)(bs.y & 0xffffu);
        x.s[3] = (int)(int16_t)(bs.y >> 16);
    }
    // The integer dot of run r (16 codes) with its activation codes.
    static __device__ __forceinline__ int run_dot(const W& w, const XA8& x, int r)
    {
        int dot = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) dot = dp4a_us(w.c[r >> 1][4 * (r & 1) + k], x.c[r >> 1][4 * (r & 1) + k], dot);
        return dot;
    }
    // sum over run r of (code - off) * x, fp32 in a fixed order
    template <int OFFC>
    static __device__ __forceinline__ float run_a32(const W& w, const float* xr, int r)
    {
        const float4* xp = reinterpret_cast<const float4*>(xr + 16 * r);
        float p = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t c = w.c[r >> 1][4 * (r & 1) + k];
            const float4 xa = xp[k];
            p = __fmaf_rn(ubyte_to_float_minus(c, 0, 8388608.f + OFFC), xa.x, p);
            p = __fmaf_rn(ubyte_to_float_minus(c, 1, 8388608.f + OFFC), xa.y, p);
            p = __fmaf_rn(ubyte_to_float_minus(c, 2, 8388608.f + OFFC), xa.z, p);
            p = __fmaf_rn(ubyte_to_float_minus(c, 3, 8388608.f + OFFC), xa.w, p);
        }
        return p;
    }
};

template <>
struct Fmt<QMV_Q2_K> : FmtK2Base<QMV_Q2_K> {
    static constexpr int BB = 84;
    static __device__ __forceinline__ void load(const uint8_t* blk, int u, W& w)
    {
        const int n = u >> 1, j0 = 2 * (u & 1);
        uint32_t q[8], sm[1];
        load_words<8>(blk + 16 + 32 * n, q);
        load_words<1>(blk + 8 * n + 2 * j0, sm);   // scale|min bytes of runs 4u .. 4u+3
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            w.c[0][k] = (q[k] >> (2 * j0)) & 0x03030303u;
            w.c[1][k] = (q[k] >> (2 * j0 + 2)) & 0x03030303u;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t byte = (sm[0] >> (8 * r)) & 0xffu;
            w.sc[r] = (int)(byte & 15u);
            w.m[r] = (int)(byte >> 4);
        }
        w.d = half_bits_to_float(ld_u16(blk + 80));
        w.dmin = half_bits_to_float(ld_u16(blk + 82));
    }
    static __device__ __forceinline__ void ints(const W& w, const XA8& x, int& S, int& Mn)
    {
        S = 0;
        Mn = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            S += w.sc[r] * run_dot(w, x, r);
            Mn += w.m[r] * x.s[r];
        }
    }
    static __device__ __forceinline__ void acc_a8(const W& w, const XA8& x, float& acc)
    {
        int S, Mn;
        ints(w, x, S, Mn);
        acc = __fmaf_rn((float)S, w.d * x.d, acc);
        acc = __fmaf_rn(-(float)Mn, w.dmin * x.d, acc);
    }
    static __device__ __forceinline__ void acc_a32(const W& w, const XView& X, int v, int b, int u, float& acc)
    {
        const float* xr = X.xf + (size_t)v * X.cols + (size_t)b * 256 + 64 * u;
        const float* xs = X.xs32 + (size_t)v * (X.cols / 16) + (size_t)b * 16 + 4 * u;   // sums of 16
#pragma unroll
        for (int r = 0; r < 4; ++r) acc = __fmaf_rn(run_a32<0>(w, xr, r), w.d * (float)w.sc[r], acc);
#pragma unroll
        for (int r = 0; r < 4; ++r) acc = __fmaf_rn(-xs[r], w.dmin * (float)w.m[r], acc);
    }
};

template <>
struct Fmt<QMV_Q3_K> : FmtK2Base<QMV_Q3_K> {
    static constexpr int BB = 110;
    // Six-bit scale s (0..15): low 4 bits from byte s (low nibble, s < 8) or
    // byte s-8 (high nibble), high 2 bits from bits 2*(s/4) of byte 8 + s%4.
    static __device__ __forceinline__ int scale6(const uint32_t (&f)[3], int s)
    {
        const uint32_t lo = s < 8 ? (f[s >> 2] >> (8 * (s & 3))) & 15u : (f[(s - 8) >> 2] >> (8 * ((s - 8) & 3) + 4)) & 15u;
        const uint32_t hi = (f[2] >> (8 * (s & 3) + 2 * (s >> 2))) & 3u;
        return (int)(lo | (hi << 4)) - 32;
    }
    static __device__ __forceinline__ void load(const uint8_t* blk, int u, W& w)
    {
        const int n = u >> 1, j0 = 2 * (u & 1);
        uint32_t q[8], hm[8], f[3];
        load_words<8>(blk + 32 + 32 * n, q);
        load_words<8>(blk, hm);
        load_words<3>(blk + 96, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            // code + 4 = low bits | high bit << 2, in 0..7
            w.c[0][k] = ((q[k] >> (2 * j0)) & 0x03030303u) | (((hm[k] >> (4 * n + j0)) & 0x01010101u) << 2);
            w.c[1][k] = ((q[k] >> (2 * j0 + 2)) & 0x03030303u) | (((hm[k] >> (4 * n + j0 + 1)) & 0x01010101u) << 2);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) w.sc[r] = scale6(f, 4 * u + r);
        w.d = half_bits_to_float(ld_u16(blk + 108));
    }
    static __device__ __forceinline__ void ints(const W& w, const XA8& x, int& S, int& Mn)
    {
        S = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) S += w.sc[r] * (run_dot(w, x, r) - 4 * x.s[r]);
        Mn = 0;
    }
    static __device__ __forceinline__ void acc_a8(const W& w, const XA8& x, float& acc)
    {
        int S, Mn;
        ints(w, x, S, Mn);
        acc = __fmaf_rn((float)S, w.d * x.d, acc);
    }
    static __device__ __forceinline__ void acc_a32(const W& w, const XView& X, int v, int b, int u, float& acc)
    {
        const float* xr = X.xf + (size_t)v * X.cols + (size_t)b * 256 + 64 * u;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc = __fmaf_rn(run_a32<4>(w, xr, r), w.d * (float)w.sc[r], acc);
    }
};

// ------------------------------------------------------------------------------
// Plain weights (F32, F16, BF16) with fp32 activations: a unit is 8 weights
// (16 or 32 bytes, 16-byte aligned when rows are multiples of 8 elements).
// ------------------------------------------------------------------------------
struct WP {
    float w[8];
};

template <int T>
struct FmtPlain {
    static constexpr int BS = 8, UE = 8, UPB = 1;
    static constexpr int BB = T == QMV_F32 ? 32 : 16;
    using W = WP;
    using XA8 = int;   // no 8-bit activation form
    static __device__ __forceinline__ void load(const uint8_t* blk, int, W& w)
    {
        if constexpr (T == QMV_F32) {
            const float4 a = reinterpret_cast<const float4*>(blk)[0], b = reinterpret_cast<const float4*>(blk)[1];
            w.w[0] = a.x; w.w[1] = a.y; w.w[2] = a.z; w.w[3] = a.w;
            w.w[4] = b.x; w.w[5] = b.y; w.w[6] = b.z; w.w[7] = b.w;
        } else {
            const uint4 a = *reinterpret_cast<const uint4*>(blk);
            const uint32_t h[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (T == QMV_F16) {
                    w.w[2 * k] = half_bits_to_float(h[k] & 0xffffu);
                    w.w[2 * k + 1] = half_bits_to_float(h[k] >> 16);
                } else {
                    w.w[2 * k] = __uint_as_float(h[k] << 16);
                    w.w[2 * k + 1] = __uint_as_float(h[k] & 0xffff0000u);
                }
            }
        }
    }
    static __device__ __forceinline__ void acc_a32(const W& w, const XView& X, int v, int b, int, float& acc)
    {
        const float4* xp = reinterpret_cast<const float4*>(X.xf + (size_t)v * X.cols + (size_t)b * 8);
        const float4 a = xp[0], c = xp[1];
        float p = __fmul_rn(w.w[0], a.x);
        p = __fmaf_rn(w.w[1], a.y, p);
        p = __fmaf_rn(w.w[2], a.z, p);
        p = __fmaf_rn(w.w[3], a.w, p);
        p = __fmaf_rn(w.w[4], c.x, p);
        p = __fmaf_rn(w.w[5], c.y, p);
        p = __fmaf_rn(w.w[6], c.z, p);
        p = __fmaf_rn(w.w[7], c.w, p);
        acc = __fadd_rn(acc, p);
    }
};
template <> struct Fmt<QMV_F32> : FmtPlain<QMV_F32> {};
template <> struct Fmt<QMV_F16> : FmtPlain<QMV_F16> {};
template <> struct Fmt<QMV_BF16> : FmtPlain<QMV_BF16> {};

// ---- the 32-element formats' products ------------------------------------------
// SPLIT (MXFP4, one or two vectors): the sum of the positive codes' products
// minus that of the negative codes', the same integer as the signed codes'
// dot: two byte permutes and a xor per four codes instead of the signed
// table's six operations, for a second dp4a -- cheaper while few vectors share
// each block (MXFP4 14336 x 4096, one vector: 23.3 -> 21.3 us; eight vectors
// keep the signed words: 43.7 against 55.8 us).
template <int T, bool SPLIT = false>
__device__ __forceinline__ void ints32(const typename Fmt<T>::W& w, const typename Fmt<T>::XA8& x, int& S, int& Mn)
{
    int dot = 0;
    if constexpr (T == QMV_MXFP4 && SPLIT) {
        int neg = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t s = (k & 1) ? w.q[k >> 1] >> 16 : w.q[k >> 1];   // prmt reads the low 16 bits
            dot = dp4a_us(Fmt<T>::mag4(s), x.w[k], dot);
            neg = dp4a_us(Fmt<T>::mag4(s ^ 0x8888u), x.w[k], neg);
        }
        dot -= neg;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            dot = Fmt<T>::SIGNED ? dp4a_ss(w.c[k], x.w[k], dot) : dp4a_us(w.c[k], x.w[k], dot);
    }
    S = dot - Fmt<T>::OFF * x.sum;
    Mn = Fmt<T>::MIN ? x.sum : 0;
}

template <int T, bool SPLIT = false>
__device__ __forceinline__ void acc32_a8(const typename Fmt<T>::W& w, const typename Fmt<T>::XA8& x, float& acc)
{
    int S, Mn;
    ints32<T, SPLIT>(w, x, S, Mn);
    acc = __fmaf_rn((float)S, w.d * x.d, acc);
    if constexpr (Fmt<T>::MIN) acc = __fmaf_rn((float)Mn, w.m * x.d, acc);
}

template <int T>
__device__ __forceinline__ void acc32_a32(const typename Fmt<T>::W& w, const XView& X, int v, int b, float& acc)
{
    // Unsigned codes minus OFF; signed codes are biased by 128 first.
    constexpr float kOff = 8388608.f + (Fmt<T>::SIGNED ? 128.f : (float)Fmt<T>::OFF);
    const float4* xp = reinterpret_cast<const float4*>(X.xf + (size_t)v * X.cols + (size_t)b * 32);
    float p = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t c = Fmt<T>::SIGNED ? (w.code(k) ^ 0x80808080u) : w.code(k);
        const float4 xa = xp[k];
        p = __fmaf_rn(ubyte_to_float_minus(c, 0, kOff), xa.x, p);
        p = __fmaf_rn(ubyte_to_float_minus(c, 1, kOff), xa.y, p);
        p = __fmaf_rn(ubyte_to_float_minus(c, 2, kOff), xa.z, p);
        p = __fmaf_rn(ubyte_to_float_minus(c, 3, kOff), xa.w, p);
    }
    acc = __fmaf_rn(p, w.d, acc);
    if constexpr (Fmt<T>::MIN) acc = __fmaf_rn(X.xs32[(size_t)v * (X.cols / 32) + b], w.m, acc);   // m * sum x
}

// Uniform entry points over all formats.
template <int T>
struct Ops {
    using F = Fmt<T>;
    using W = typename F::W;
    using XA8 = typename F::XA8;
    static __device__ __forceinline__ void ints(const W& w, const XA8& x, int& S, int& Mn)
    {
        if constexpr (F::BS == 32) ints32<T>(w, x, S, Mn);
        else if constexpr (F::BS == 256) F::ints(w, x, S, Mn);
    }
    // FEW: one or two vectors share each decoded block
    template <bool FEW = false>
    static __device__ __forceinline__ void acc_a8(const W& w, const XA8& x, float& acc)
    {
        if constexpr (F::BS == 32) acc32_a8<T, FEW>(w, x, acc);
        else if constexpr (F::BS == 256) F::acc_a8(w, x, acc);
    }
    static __device__ __forceinline__ void acc_a32(const W& w, const XView& X, int v, int b, int sub, float& acc)
    {
        if constexpr (F::BS == 32) acc32_a32<T>(w, X, v, b, acc);
        else F::acc_a32(w, X, v, b, sub, acc);
    }
};

// ---- staging activations into shared memory -----------------------------------------
// Position of element i (0..31) of a 32-run in the staged order of format T.
template <int T>
__device__ __forceinline__ int staged_pos(int i)
{
    if constexpr (T == QMV_MXFP4) return i < 16 ? 2 * i : 2 * (i - 16) + 1;
    else return i;
}

// Bytes of staged activation codes for g vectors (8-bit staging).
__host__ __device__ inline size_t xcode_bytes(int T, int g, int cols)
{
    return kq_rt(T) ? (size_t)g * (cols / 256) * kKPitch : (size_t)g * (cols / 32) * kBPitch;
}

// Bytes of staged activations for g vectors of `cols` elements.
__host__ __device__ inline size_t xhat_bytes(int T, bool a8, int g, int cols)
{
    const int bs = kq_rt(T) ? 256 : 32;
    const size_t nb = (size_t)cols / bs;
    auto r16 = [](size_t v) { return (v + 15) & ~size_t(15); };
    if (a8) {
        size_t s = r16(xcode_bytes(T, g, cols)) + r16((size_t)g * nb * 4);
        s += (bs == 32) ? r16((size_t)g * nb * 4) : r16((size_t)g * nb * 32);
        return s;
    }
    size_t s = r16((size_t)g * cols * 4);
    if (xsum_run_rt(T)) s += r16((size_t)g * (cols / xsum_run_rt(T)) * 4);
    return s;
}

template <int T>
__device__ __forceinline__ XView carve_xview(uint8_t* base, bool a8, int g, int cols)
{
    constexpr int bs = Fmt<T>::BS;
    const int nb = cols / bs;
    auto r16 = [](size_t v) { return (v + 15) & ~size_t(15); };
    XView X{};
    X.cols = cols;
    X.nb = nb;
    if (a8) {
        X.codes = base;
        uint8_t* p = base + r16(xcode_bytes(T, g, cols));
        X.d = reinterpret_cast<const float*>(p);
        p += r16((size_t)g * nb * 4);
        if (bs == 32) X.sum32 = reinterpret_cast<const int*>(p);
        else X.bsum = reinterpret_cast<const int16_t*>(p);
    } else {
        X.xf = reinterpret_cast<const float*>(base);
        X.xs32 = reinterpret_cast<const float*>(base + r16((size_t)g * cols * 4));
    }
    return X;
}

// Quantise-while-staging: TPB threads per activation block, each loading its
// 32/TPB (or 256/TPB) consecutive values at once; the block's amax and code
// sums are xor-shuffles over the TPB lanes, which are consecutive lanes of one
// warp (the loop runs over whole warps: nth is a multiple of 32).  Scale,
// codes and sums are those of the activation quantiser.  Small activations
// (one decode vector of a few thousand elements) would otherwise be quantised
// by a few dozen threads, each over a whole block, on the critical path of
// every launch.
template <int T, bool NATURAL, int TPB, typename Row>
__device__ __forceinline__ void stage_quant32(uint8_t* codes, float* d, uint8_t* tail, const Row& row, int nbk,
                                              int nb, int tid, int nth)
{
    if constexpr (TPB == 1) {
        // One block per thread: an amax pass, then a quantising pass over the
        // same (cached) values; measured faster here than holding the block
        // in registers.
        for (int i = tid; i < nbk; i += nth) {
            const float4* xp = reinterpret_cast<const float4*>(row(i / nb)) + (size_t)(i % nb) * 8;
            float amax = 0.f;
            for (int k = 0; k < 8; ++k) {
                const float4 w = xp[k];
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w))));
            }
            float dd, id;
            act_scale(amax, dd, id);
            uint8_t* dst = codes + (size_t)i * (NATURAL ? 32 : kBPitch);
            // The quantising pass, in two copies so that the common one holds
            // no division: TINY for the rare block whose 1/d overflows (its
            // codes are round(x / d), see tiny_scale_divide).
            auto pass = [&](auto tiny) {
                int sum = 0;
                for (int k = 0; k < 8; ++k) {
                    float4 wv[1] = {xp[k]};
                    float idk = id;
                    if constexpr (decltype(tiny)::value) tiny_scale_divide(wv, dd, idk);
                    const float4 w = wv[0];
                    const int8_t q0 = quant1(w.x, idk), q1 = quant1(w.y, idk), q2 = quant1(w.z, idk),
                                 q3 = quant1(w.w, idk);
                    dst[NATURAL ? 4 * k + 0 : staged_pos<T>(4 * k + 0)] = (uint8_t)q0;
                    dst[NATURAL ? 4 * k + 1 : staged_pos<T>(4 * k + 1)] = (uint8_t)q1;
                    dst[NATURAL ? 4 * k + 2 : staged_pos<T>(4 * k + 2)] = (uint8_t)q2;
                    dst[NATURAL ? 4 * k + 3 : staged_pos<T>(4 * k + 3)] = (uint8_t)q3;
                    sum += q0 + q1 + q2 + q3;
                }
                return sum;
            };
            const int sum = isinf(id) ? pass(std::true_type{}) : pass(std::false_type{});
            d[i] = __half2float(__float2half_rn(dd));   // Q8_0 keeps its scale in fp16
            reinterpret_cast<int*>(tail)[i] = sum;
        }
        return;
    }
    constexpr int E = 32 / TPB, NF4 = E / 4;
    const int lane = tid & 31, total = nbk * TPB;
    for (int i0 = tid - lane; i0 < total; i0 += nth) {
        const int i = i0 + lane, blk = i / TPB, part = i % TPB;
        const bool valid = i < total;    // the same for the TPB lanes of a block
        float4 w[NF4];
        float amax = 0.f;
#pragma unroll
        for (int f = 0; f < NF4; ++f) w[f] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            const float4* xp = reinterpret_cast<const float4*>(row(blk / nb)) + (size_t)(blk % nb) * 8 + part * NF4;
#pragma unroll
            for (int f = 0; f < NF4; ++f) w[f] = xp[f];
        }
#pragma unroll
        for (int f = 0; f < NF4; ++f)
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(w[f].x), fabsf(w[f].y)), fmaxf(fabsf(w[f].z), fabsf(w[f].w))));
#pragma unroll
        for (int o = 1; o < TPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        float dd, id;
        act_scale(amax, dd, id);
        tiny_scale_divide(w, dd, id);
        uint8_t* dst = codes + (size_t)blk * (NATURAL ? 32 : kBPitch);
        int sum = 0;
#pragma unroll
        for (int f = 0; f < NF4; ++f) {
            const int8_t q0 = quant1(w[f].x, id), q1 = quant1(w[f].y, id), q2 = quant1(w[f].z, id),
                         q3 = quant1(w[f].w, id);
            sum += q0 + q1 + q2 + q3;
            const int e = part * E + 4 * f;
            if (!valid) continue;
            if (NATURAL || T != QMV_MXFP4) {
                reinterpret_cast<uint32_t*>(dst)[e >> 2] = (uint32_t)(uint8_t)q0 | ((uint32_t)(uint8_t)q1 << 8) |
                                                           ((uint32_t)(uint8_t)q2 << 16) |
                                                           ((uint32_t)(uint8_t)q3 << 24);
            } else {
                dst[staged_pos<T>(e + 0)] = (uint8_t)q0;
                dst[staged_pos<T>(e + 1)] = (uint8_t)q1;
                dst[staged_pos<T>(e + 2)] = (uint8_t)q2;
                dst[staged_pos<T>(e + 3)] = (uint8_t)q3;
            }
        }
#pragma unroll
        for (int o = 1; o < TPB; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (valid && part == 0) {
            d[blk] = __half2float(__float2half_rn(dd));   // Q8_0 keeps its scale in fp16
            reinterpret_cast<int*>(tail)[blk] = sum;
        }
    }
}

template <int T, bool NATURAL, int TPB, typename Row>
__device__ __forceinline__ void stage_quant256(uint8_t* codes, float* d, uint8_t* tail, const Row& row, int nbk,
                                               int nb, int tid, int nth)
{
    static_assert(TPB == 8 || TPB == 16 || TPB == 32, "256-element blocks: 8, 16 or 32 threads each");
    constexpr int E = 256 / TPB, NF4 = E / 4;
    const int lane = tid & 31, total = nbk * TPB;
    for (int i0 = tid - lane; i0 < total; i0 += nth) {
        const int i = i0 + lane, blk = i / TPB, part = i % TPB;
        const bool valid = i < total;
        float4 w[NF4];
        float amax = 0.f;
#pragma unroll
        for (int f = 0; f < NF4; ++f) w[f] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            const float4* xp = reinterpret_cast<const float4*>(row(blk / nb)) + (size_t)(blk % nb) * 64 + part * NF4;
#pragma unroll
            for (int f = 0; f < NF4; ++f) w[f] = xp[f];
        }
#pragma unroll
        for (int f = 0; f < NF4; ++f)
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(w[f].x), fabsf(w[f].y)), fmaxf(fabsf(w[f].z), fabsf(w[f].w))));
#pragma unroll
        for (int o = 1; o < TPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        float dd, id;
        act_scale(amax, dd, id);
        tiny_scale_divide(w, dd, id);
        uint8_t* dst = codes + (size_t)blk * (NATURAL ? 256 : kKPitch);
        int16_t* bsum = reinterpret_cast<int16_t*>(tail) + (size_t)blk * 16;
        int s16 = 0;   // running sum of the current 16-group
#pragma unroll
        for (int f = 0; f < NF4; ++f) {
            const int8_t q0 = quant1(w[f].x, id), q1 = quant1(w[f].y, id), q2 = quant1(w[f].z, id),
                         q3 = quant1(w[f].w, id);
            s16 += q0 + q1 + q2 + q3;
            const int e = part * E + 4 * f, r = e >> 4;
            if (valid)
                reinterpret_cast<uint32_t*>(dst + (NATURAL ? 16 * r : kquant_run_pos<T>(r)))[(e & 15) >> 2] =
                    (uint32_t)(uint8_t)q0 | ((uint32_t)(uint8_t)q1 << 8) | ((uint32_t)(uint8_t)q2 << 16) |
                    ((uint32_t)(uint8_t)q3 << 24);
            if constexpr (E >= 16) {
                if ((f & 3) == 3) {   // a whole 16-group in this thread
                    if (valid) bsum[r] = (int16_t)s16;
                    s16 = 0;
                }
            }
        }
        if constexpr (E == 8) {   // a 16-group spans two lanes
            s16 += __shfl_xor_sync(0xffffffffu, s16, 1);
            if (valid && (part & 1) == 0) bsum[(part * E) >> 4] = (int16_t)s16;
        }
        if (valid && part == 0) d[blk] = dd;
    }
}

// Stage g activation vectors with threads tid = 0..nth-1 of the block, whole
// warps (nth a multiple of 32; the caller synchronises afterwards).  Vector v is row idx[v] (v when idx is
// NULL) of the caller's activations, whose rows are xrow bytes apart: fp32
// [cols] (A32, or A8 with quant_x) or Q8_0/Q8_K blocks [nb] (A8).  With
// quant_x the fp32 activations are quantised here with the exact steps of the
// activation quantiser, so the staged bytes equal those staged from
// qmv_quantize_act's output.
template <int T, bool NATURAL = false>
__device__ void stage_xhat(uint8_t* base, bool a8, bool quant_x, const void* x, size_t xrow, const int* idx, int g,
                           int cols, int tid, int nth)
{
    constexpr int bs = Fmt<T>::BS;
    const int nb = cols / bs;
    auto r16 = [](size_t v) { return (v + 15) & ~size_t(15); };
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    auto row = [&](int v) { return xb + (size_t)(idx ? idx[v] : v) * xrow; };
    if (a8 && quant_x) {
        uint8_t* codes = base;
        float* d = reinterpret_cast<float*>(base + r16(xcode_bytes(T, g, cols)));
        uint8_t* tail = base + r16(xcode_bytes(T, g, cols)) + r16((size_t)g * nb * 4);
        // As many threads per block as one pass of the CTA's threads allows (a
        // block's activations then arrive with one round of loads), or two
        // passes if the second is at least half full (else the CTA would wait
        // a whole pass for a few threads).
        const int nbk = g * nb;
        auto fits = [&](int t) { return nbk * t <= nth || (nbk * t <= 2 * nth && 2 * nbk * t >= 3 * nth); };
        if constexpr (bs == 32) {
            if (fits(8)) stage_quant32<T, NATURAL, 8>(codes, d, tail, row, nbk, nb, tid, nth);
            else if (fits(4)) stage_quant32<T, NATURAL, 4>(codes, d, tail, row, nbk, nb, tid, nth);
            else if (fits(2)) stage_quant32<T, NATURAL, 2>(codes, d, tail, row, nbk, nb, tid, nth);
            else stage_quant32<T, NATURAL, 1>(codes, d, tail, row, nbk, nb, tid, nth);
        } else {
            if (nbk * 32 <= nth) stage_quant256<T, NATURAL, 32>(codes, d, tail, row, nbk, nb, tid, nth);
            else if (nbk * 16 <= nth) stage_quant256<T, NATURAL, 16>(codes, d, tail, row, nbk, nb, tid, nth);
            else stage_quant256<T, NATURAL, 8>(codes, d, tail, row, nbk, nb, tid, nth);
        }
    } else if (a8) {
        uint8_t* codes = base;
        float* d = reinterpret_cast<float*>(base + r16(xcode_bytes(T, g, cols)));
        uint8_t* tail = base + r16(xcode_bytes(T, g, cols)) + r16((size_t)g * nb * 4);
        if constexpr (bs == 32) {
            // Q8_0 blocks: fp16 d | int8[32], 34 bytes, 2-byte aligned.
            int* sum = reinterpret_cast<int*>(tail);
            for (int i = tid; i < g * nb; i += nth) {
                const int v = i / nb, b = i % nb;
                const uint16_t* h = reinterpret_cast<const uint16_t*>(row(v) + (size_t)b * 34);
                uint8_t q[32];
                int s = 0;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint32_t two = h[1 + k];
                    q[2 * k] = two & 0xffu;
                    q[2 * k + 1] = two >> 8;
                    s += (int)(int8_t)(two & 0xffu) + (int)(int8_t)(two >> 8);
                }
                uint8_t* dst = codes + (size_t)i * (NATURAL ? 32 : kBPitch);   // vector v, block b: i = v*nb + b
#pragma unroll
                for (int k = 0; k < 32; ++k) dst[NATURAL ? k : staged_pos<T>(k)] = q[k];
                d[i] = half_bits_to_float(h[0]);
                sum[i] = s;
            }
        } else {
            // Q8_K blocks: f32 d | int8[256] | int16 bsums[16], 292 bytes, 4-byte aligned.
            int16_t* bsum = reinterpret_cast<int16_t*>(tail);
            for (int i = tid; i < g * nb * 73; i += nth) {
                const int blkno = i / 73, wd = i % 73;
                const int v = blkno / nb, b = blkno % nb;
                const uint32_t val = reinterpret_cast<const uint32_t*>(row(v) + (size_t)b * 292)[wd];
                if (wd == 0) d[blkno] = __uint_as_float(val);
                else if (wd <= 64) {
                    const int w = wd - 1;   // code word w: elements 4w..4w+3, run w / 4
                    if (NATURAL) reinterpret_cast<uint32_t*>(codes + (size_t)blkno * 256)[w] = val;
                    else reinterpret_cast<uint32_t*>(codes + (size_t)blkno * kKPitch + kquant_run_pos<T>(w >> 2))[w & 3] = val;
                }
                else reinterpret_cast<uint32_t*>(bsum + (size_t)blkno * 16)[wd - 65] = val;
            }
        }
    } else {
        float* xf = reinterpret_cast<float*>(base);
        const int c4 = cols / 4;
        for (int i = tid; i < g * c4; i += nth) {
            const int v = i / c4, j = i % c4;
            const float4 w = reinterpret_cast<const float4*>(row(v))[j];
            if constexpr (T == QMV_MXFP4) {
                const int e = 4 * i, run = e & ~31;
                xf[run + staged_pos<T>((e + 0) & 31)] = w.x;
                xf[run + staged_pos<T>((e + 1) & 31)] = w.y;
                xf[run + staged_pos<T>((e + 2) & 31)] = w.z;
                xf[run + staged_pos<T>((e + 3) & 31)] = w.w;
            } else {
                reinterpret_cast<float4*>(xf)[i] = w;
            }
        }
    }
}

// A8 staging in natural element order (the tensor-core engine's B fragments).
template <int T>
__device__ __forceinline__ void stage_xhat_a8_natural(uint8_t* base, bool quant_x, const void* x, size_t xrow, int g,
                                                      int cols, int tid, int nth)
{
    stage_xhat<T, true>(base, true, quant_x, x, xrow, nullptr, g, cols, tid, nth);
}

// Sums of each run of R staged fp32 activations (R = xsum_run_rt(T): the
// formats whose weights carry a per-run offset), in a fixed order; run after
// the staging is visible to these threads.
template <int T>
__device__ void stage_xsum32(uint8_t* base, int g, int cols, int tid, int nth)
{
    constexpr int R = xsum_run_rt(T);
    if constexpr (R > 0) {
        auto r16 = [](size_t v) { return (v + 15) & ~size_t(15); };
        const float* xf = reinterpret_cast<const float*>(base);
        float* xs = reinterpret_cast<float*>(base + r16((size_t)g * cols * 4));
        for (int i = tid; i < g * cols / R; i += nth) {
            float s = 0.f;
            for (int k = 0; k < R; ++k) s += xf[(size_t)i * R + k];
            xs[i] = s;
        }
    }
}

}  // namespace qmv
