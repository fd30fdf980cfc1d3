// mma_units.cuh -- weight codes and activations as int8 MMA fragments.
//
// The W4A8 product ("Architecture" page, "The package map": the fused W4A8
// kernels of pkg/quant) on the int8 tensor-core path of sm_103a:
// mma.sync.m16n8k32 (k16 for Q6_K's 16-element sub-blocks) .s8.s8.s32.
// A = 16 weight rows x 32 codes, B = 32 activation codes x 8 vectors, D =
// exact int32 block dots.  (The tcgen05 int8 kind is not available on
// sm_103a; these warp-level MMAs are.)
//
// Fragment layouts (groupID g = lane/4, q = lane%4):
//   A k32: a0 row g, k 4q..4q+3; a1 row g+8; a2 row g, k 16+4q..; a3 row g+8
//   A k16: a0 row g, k 4q..4q+3; a1 row g+8
//   B k32: b0 k 4q..4q+3, column g; b1 k 16+4q..    B k16: b0 only
//   D: d0 (row g, col 2q), d1 (row g, col 2q+1), d2 (row g+8, col 2q), d3 (row g+8, col 2q+1)
// Weight codes are laid out so that byte j of a fragment register is the code
// of element k+j, in natural element order; unsigned codes (Q4_0 0..15, Q5_0
// 0..31, Q4_K 0..15, Q6_K 0..63) enter as non-negative s8 and their offsets
// (8, 16, 32) are removed through exact activation sums afterwards.
#pragma once

#include "formats.cuh"

namespace qmv {

__device__ __forceinline__ void mma_k32(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_k16(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// Word of 4 bytes at any byte address of shared memory.
__device__ __forceinline__ uint32_t ld_word(const uint8_t* p)
{
    uint32_t w[1];
    load_words<1>(p, w);
    return w[0];
}

// The four low (or high) nibbles of a byte word as four nibble selectors.
__device__ __forceinline__ uint32_t nibbles_to_sel(uint32_t bytes4)
{
    const uint32_t t = bytes4 | (bytes4 >> 4);          // byte0 = n0 | n1<<4, byte2 = n2 | n3<<4
    return __byte_perm(t, 0u, 0x0020u) & 0xffffu;       // [byte0, byte2]
}

// ---- per-format A fragments of one 32-element block (rows g and g+8) ---------
// blk0 / blk1: the block of row g and of row g+8 in shared memory.
template <int T>
struct MmaA32;

template <>
struct MmaA32<QMV_Q4_0> {
    static constexpr int OFF = 8;
    static __device__ __forceinline__ void load(const uint8_t* blk0, const uint8_t* blk1, int q, uint32_t (&a)[4],
                                                float& d0, float& d1)
    {
        const uint32_t w0 = ld_word(blk0 + 2 + 4 * q), w1 = ld_word(blk1 + 2 + 4 * q);
        a[0] = w0 & 0x0f0f0f0fu;
        a[1] = w1 & 0x0f0f0f0fu;
        a[2] = (w0 >> 4) & 0x0f0f0f0fu;
        a[3] = (w1 >> 4) & 0x0f0f0f0fu;
        d0 = half_bits_to_float(ld_u16(blk0));
        d1 = half_bits_to_float(ld_u16(blk1));
    }
};

template <>
struct MmaA32<QMV_Q5_0> {
    static constexpr int OFF = 16;
    static __device__ __forceinline__ void load(const uint8_t* blk0, const uint8_t* blk1, int q, uint32_t (&a)[4],
                                                float& d0, float& d1)
    {
        const uint32_t h0 = ld_word(blk0 + 2), h1 = ld_word(blk1 + 2);
        const uint32_t w0 = ld_word(blk0 + 6 + 4 * q), w1 = ld_word(blk1 + 6 + 4 * q);
        a[0] = (w0 & 0x0f0f0f0fu) | Fmt<QMV_Q5_0>::spread4((h0 >> (4 * q)) & 15u);
        a[1] = (w1 & 0x0f0f0f0fu) | Fmt<QMV_Q5_0>::spread4((h1 >> (4 * q)) & 15u);
        a[2] = ((w0 >> 4) & 0x0f0f0f0fu) | Fmt<QMV_Q5_0>::spread4((h0 >> (16 + 4 * q)) & 15u);
        a[3] = ((w1 >> 4) & 0x0f0f0f0fu) | Fmt<QMV_Q5_0>::spread4((h1 >> (16 + 4 * q)) & 15u);
        d0 = half_bits_to_float(ld_u16(blk0));
        d1 = half_bits_to_float(ld_u16(blk1));
    }
};

template <>
struct MmaA32<QMV_Q8_0> {
    static constexpr int OFF = 0;
    static __device__ __forceinline__ void load(const uint8_t* blk0, const uint8_t* blk1, int q, uint32_t (&a)[4],
                                                float& d0, float& d1)
    {
        a[0] = ld_word(blk0 + 2 + 4 * q);
        a[1] = ld_word(blk1 + 2 + 4 * q);
        a[2] = ld_word(blk0 + 18 + 4 * q);
        a[3] = ld_word(blk1 + 18 + 4 * q);
        d0 = half_bits_to_float(ld_u16(blk0));
        d1 = half_bits_to_float(ld_u16(blk1));
    }
};

template <>
struct MmaA32<QMV_MXFP4> {
    static constexpr int OFF = 0;
    static __device__ __forceinline__ void load(const uint8_t* blk0, const uint8_t* blk1, int q, uint32_t (&a)[4],
                                                float& d0, float& d1)
    {
        const uint32_t w0 = ld_word(blk0 + 1 + 4 * q), w1 = ld_word(blk1 + 1 + 4 * q);
        using M = Fmt<QMV_MXFP4>;
        a[0] = M::lut4(nibbles_to_sel(w0 & 0x0f0f0f0fu));
        a[1] = M::lut4(nibbles_to_sel(w1 & 0x0f0f0f0fu));
        a[2] = M::lut4(nibbles_to_sel((w0 >> 4) & 0x0f0f0f0fu));
        a[3] = M::lut4(nibbles_to_sel((w1 >> 4) & 0x0f0f0f0fu));
        d0 = M::e8m0_half(blk0[0]);
        d1 = M::e8m0_half(blk1[0]);
    }
};

}  // namespace qmv

namespace qmv {

// Q4_K six-bit scales and mins of all 8 sub-blocks as packed bytes:
// sc03/m03 hold sub-blocks 0..3, sc47/m47 sub-blocks 4..7 (byte j = sub-block j).
struct Q4kScales {
    uint32_t sc03, sc47, m03, m47;
    __device__ __forceinline__ int sc(int j) const { return (int)(((j < 4 ? sc03 : sc47) >> (8 * (j & 3))) & 0xffu); }
    __device__ __forceinline__ int m(int j) const { return (int)(((j < 4 ? m03 : m47) >> (8 * (j & 3))) & 0xffu); }
};

__device__ __forceinline__ Q4kScales q4k_scales(uint32_t f0, uint32_t f1, uint32_t f2)
{
    Q4kScales s;
    s.sc03 = f0 & 0x3f3f3f3fu;
    s.m03 = f1 & 0x3f3f3f3fu;
    s.sc47 = (f2 & 0x0f0f0f0fu) | ((f0 >> 2) & 0x30303030u);
    s.m47 = ((f2 >> 4) & 0x0f0f0f0fu) | ((f1 >> 2) & 0x30303030u);
    return s;
}

}  // namespace qmv
