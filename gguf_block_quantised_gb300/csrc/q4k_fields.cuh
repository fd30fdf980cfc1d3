// q4k_fields.cuh -- the six-bit scales and mins of a Q4_K super-block, as
// packed bytes, for the tensor-core kernels that dequantise whole tiles.
//
// Q4_K ("Models and formats" page, "Tensor formats"; GGUF layout): a 12-byte
// field after d and dmin packs eight 6-bit scales and eight 6-bit mins; bytes
// 0..3 hold sc0..sc3 in their low 6 bits and bits 4..5 of sc4..sc7 on top,
// bytes 4..7 the same for the mins, bytes 8..11 the low nibbles of sc4..sc7
// (low) and m4..m7 (high).
#pragma once

#include "common.cuh"

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
