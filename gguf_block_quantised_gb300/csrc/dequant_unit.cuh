// dequant_unit.cuh -- one decoding unit of a weight block as fp32 values in
// element order, for the prefill kernels that turn weight tiles into bf16
// tensor-core operands.  The values are the matvec kernels' (formats.cuh unit
// decoders): w = d*q (exact), d*q + m or d*sc*q - dmin*m (one fp32 rounding).
#pragma once

#include <cuda_bf16.h>

#include "formats.cuh"

namespace qmv {

// Element index of byte j of code word k of a 32-element unit (MXFP4 keeps its
// nibble pairs: low nibble = element p/2, high = 16 + p/2).
template <int T>
__device__ __forceinline__ constexpr int unit_elem(int k, int j)
{
    if constexpr (T == QMV_MXFP4) {
        const int p = 4 * k + j;
        return (p & 1) ? 16 + (p >> 1) : (p >> 1);
    } else {
        return 4 * k + j;
    }
}

// The UE values of unit `s` of the block at blk, in the unit's own element
// order (Q6_K: group g's 16 elements at 16g..16g+15).
template <int T>
__device__ __forceinline__ void unit_values(const uint8_t* blk, int s, float (&v)[Fmt<T>::UE])
{
    using F = Fmt<T>;
    typename F::W w;
    F::load(blk, s, w);
    if constexpr (plain_rt(T)) {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = w.w[k];
    } else if constexpr (F::BS == 32) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t byte = (w.code(k) >> (8 * j)) & 0xffu;
                const int q = F::SIGNED ? (int)(int8_t)byte : (int)byte - F::OFF;
                if constexpr (F::MIN) v[unit_elem<T>(k, j)] = __fmaf_rn(w.d, (float)q, w.m);   // one rounding
                else v[unit_elem<T>(k, j)] = w.d * (float)q;   // exact: <= 24 significant bits
            }
    } else if constexpr (T == QMV_Q4_K || T == QMV_Q5_K) {
        constexpr uint32_t mask = T == QMV_Q5_K ? 31u : 15u;
        const float D0 = w.d * (float)w.sc0, D1 = w.d * (float)w.sc1;       // exact
        const float M0 = w.dmin * (float)w.m0, M1 = w.dmin * (float)w.m1;   // exact
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[4 * k + j] = __fmaf_rn(D0, (float)((w.lo[k] >> (8 * j)) & mask), -M0);
                v[32 + 4 * k + j] = __fmaf_rn(D1, (float)((w.hi[k] >> (8 * j)) & mask), -M1);
            }
    } else if constexpr (T == QMV_Q2_K || T == QMV_Q3_K) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float D = w.d * (float)w.sc[r];   // exact
            const float M = T == QMV_Q2_K ? w.dmin * (float)w.m[r] : 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = (int)((w.c[r >> 1][4 * (r & 1) + (i >> 2)] >> (8 * (i & 3))) & 0xffu);
                v[16 * r + i] = T == QMV_Q2_K ? __fmaf_rn(D, (float)c, -M) : D * (float)(c - 4);
            }
        }
    } else {   // Q6_K
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float D = w.d * (float)w.sc[g];   // exact
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j) v[16 * g + 4 * k + j] = D * (float)((int)((w.g[g][k] >> (8 * j)) & 63u) - 32);
        }
    }
}

// Two fp32 values in one 64-bit register for the packed f32x2 instructions.
__device__ __forceinline__ uint64_t pk2(float lo, float hi)
{
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

// (D*q - M) for the two codes packed in bytes j0, j1 of `codes` (each 0..15),
// exactly as two fp32 fused multiply-adds: 0x4B0000qq is the float 2^23 + q,
// so subtracting 2^23 gives q exactly.
__device__ __forceinline__ uint32_t dq2_bf16(uint32_t codes, uint32_t sel, uint64_t D2, uint64_t negM2)
{
    const uint32_t f0 = __byte_perm(codes, 0x4B000000u, sel & 0xffffu);          // bytes: code, 0, 0, 0x4B
    const uint32_t f1 = __byte_perm(codes, 0x4B000000u, sel >> 16);
    uint64_t v = ((uint64_t)f1 << 32) | f0, q, w;
    const uint64_t two23 = pk2(-8388608.f, -8388608.f);
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(v), "l"(two23));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(w) : "l"(D2), "l"(q), "l"(negM2));
    const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float((uint32_t)w), __uint_as_float((uint32_t)(w >> 32)));
    return *reinterpret_cast<const uint32_t*>(&b);
}

// Bytes [p, p + 4*NW) of shared memory as NW little-endian words, p any byte
// address: 16-byte loads from p rounded down to 16 (the rows of the tiles are
// laid out so that eight consecutive rows' 16-byte loads hit distinct banks),
// then the words are realigned in registers.  Reads up to 15 + 16 bytes past
// the window.
template <int NW>
__device__ __forceinline__ void smem_window(const uint8_t* p, uint32_t (&x)[NW])
{
    const uint32_t a = smem_u32(p);
    const uint4* b = reinterpret_cast<const uint4*>(p - (a & 15u));
    const uint32_t sh = a & 15u, q = sh >> 2, fs = 8u * (sh & 3u);
    constexpr int NV = (4 * NW + 15 + 15) / 16;
    uint32_t u[4 * NV + 3];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const uint4 c = b[v];
        u[4 * v] = c.x; u[4 * v + 1] = c.y; u[4 * v + 2] = c.z; u[4 * v + 3] = c.w;
    }
#pragma unroll
    for (int i = 4 * NV; i < 4 * NV + 3; ++i) u[i] = 0u;
    uint32_t w[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) w[i] = q == 0 ? u[i] : q == 1 ? u[i + 1] : q == 2 ? u[i + 2] : u[i + 3];
#pragma unroll
    for (int i = 0; i < NW; ++i) x[i] = __funnelshift_r(w[i], w[i + 1], fs);
}

}  // namespace qmv
