// quant_w.cu -- fp32 weights -> Q4_0 / Q5_0 blocks ("Models and formats" page,
// "Tensor formats": the quantiser writes Q4_0/1, Q5_0/1, Q8_0 and the
// K-quants).  Q8_0 weights are the symmetric 8-bit form and run the
// activation quantiser (quant_act.cu).
//
// Per 32-element block: m = the signed value of largest magnitude (the first
// on ties); d = m / -half (half = 8 or 16); id = 1/d (0 when d = 0); code =
// trunc(clamp(x*id + half + 0.5, 0, 2*half - 1)), with x/d in place of x*id
// when |d| is below 2^-128 and 1/d overflows.  The largest-magnitude
// element lands on code 0.  Every step is one IEEE fp32 rounding (__fdiv_rn,
// __fmul_rn, __fadd_rn; no contraction), so the codes do not depend on the
// thread layout.  The block stores fp16(d), for Q5_0 the fifth bits (bit i
// for element i), then the nibbles: byte j holds element j (low) and j + 16
// (high).
//
// Eight threads per block, one float4 each (coalesced 16-byte loads); the
// extreme is an xor reduction of (|x|, index) over the eight lanes.  The pass
// reads 4 bytes and writes 0.56 or 0.69 bytes per weight: bound by HBM.
#include "common.cuh"

namespace qmv {

template <int BITS>
__global__ void __launch_bounds__(256) k_quant_w(const float4* __restrict__ x, uint8_t* __restrict__ out,
                                                 int64_t nblk)
{
    constexpr int BB = BITS == 4 ? 18 : 22;
    constexpr float kHalf = (float)(1 << (BITS - 1));
    constexpr float kTop = (float)((1 << BITS) - 1);
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t blk = i >> 3;
    const int part = (int)(i & 7);
    const bool valid = blk < nblk;           // the same for the eight lanes of a block
    const float4 w = valid ? x[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    float v[4] = {w.x, w.y, w.z, w.w};

    // The first element of largest magnitude: strictly larger magnitudes win,
    // and among equal ones the lower index (an all-zero block keeps +0).
    float a = 0.f, m = 0.f;
    int idx = 32;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (fabsf(v[k]) > a) {
            a = fabsf(v[k]);
            m = v[k];
            idx = 4 * part + k;
        }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const float oa = __shfl_xor_sync(0xffffffffu, a, o);
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (oa > a || (oa == a && oi < idx)) {
            a = oa;
            m = om;
            idx = oi;
        }
    }
    const float d = __fdiv_rn(m, -kHalf);
    float id = d == 0.f ? 0.f : __fdiv_rn(1.f, d);
    tiny_scale_divide(v, d, id);   // |d| below 2^-128: the codes come from x / d
    uint32_t codes = 0, hi_bits = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float t = __fadd_rn(__fmul_rn(v[k], id), kHalf + 0.5f);
        t = fmaxf(fminf(t, kTop), 0.f);
        const uint32_t c = (uint32_t)__float2int_rz(t);
        codes |= (c & 15u) << (8 * k);
        hi_bits |= ((c >> 4) & 1u) << (4 * part + k);
    }
    // Byte j of the nibbles pairs element j (thread j/4) with element j + 16
    // (thread 4 + j/4).
    const uint32_t other = __shfl_xor_sync(0xffffffffu, codes, 4);
    if constexpr (BITS == 5) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) hi_bits |= __shfl_xor_sync(0xffffffffu, hi_bits, o);
    }
    if (!valid) return;
    // Blocks are 18 or 22 bytes and the output 2-byte aligned: 16-bit stores.
    uint16_t* o = reinterpret_cast<uint16_t*>(out + blk * BB);
    if (part == 0) {
        *reinterpret_cast<__half*>(o) = __float2half_rn(d);
        if constexpr (BITS == 5) {
            o[1] = (uint16_t)(hi_bits & 0xffffu);
            o[2] = (uint16_t)(hi_bits >> 16);
        }
    }
    if (part < 4) {
        const uint32_t b = (codes & 0x0f0f0f0fu) | ((other & 0x0f0f0f0fu) << 4);   // bytes 4*part .. 4*part+3
        uint16_t* qs = o + (BITS == 5 ? 3 : 1) + 2 * part;
        qs[0] = (uint16_t)(b & 0xffffu);
        qs[1] = (uint16_t)(b >> 16);
    }
}

}  // namespace qmv

int qmv_launch_quantize(int atype, const float* x, void* xq, int64_t n, bool pdl, cudaStream_t st);

// Returns 0, or -1 on a launch failure.
int qmv_launch_quantize_weights(int wtype, const float* W, int64_t n, void* out, cudaStream_t st)
{
    using namespace qmv;
    if (wtype == QMV_Q8_0) return qmv_launch_quantize(QMV_Q8_0, W, out, n, false, st);
    const int64_t nblk = n / 32;
    if (nblk == 0) return 0;
    const int64_t threads = nblk * 8;
    const dim3 grid((unsigned)((threads + 255) / 256));
    const float4* x = reinterpret_cast<const float4*>(W);
    uint8_t* o = static_cast<uint8_t*>(out);
    if (wtype == QMV_Q4_0) k_quant_w<4><<<grid, 256, 0, st>>>(x, o, nblk);
    else k_quant_w<5><<<grid, 256, 0, st>>>(x, o, nblk);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
