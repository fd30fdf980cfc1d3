// quant_act.cu -- fp32 activations -> Q8_0 / Q8_K blocks (the "A8" of the
// fused W4A8 kernels, "Architecture" page, "The package map", pkg/quant).
//
// Per block: amax = max|x|; d = amax/127; id = 1/d (0 when d = 0);
// q = round-half-away-from-zero(x*id) clamped to +-127, or of x/d when d is
// below 2^-128 and 1/d overflows.  Every step is one IEEE fp32 rounding
// (__fdiv_rn, __fmul_rn, roundf), so the codes do not depend on the thread
// layout and equal those of the plain definition.  Q8_0
// stores fp16(d) (round to nearest even); Q8_K stores the fp32 d and the
// int16 sums of each run of 16 codes.
//
// One warp per block.  This kernel moves ~5 bytes per element in total and is
// a small fraction of any multiply it feeds.
#include "common.cuh"
#include "runtime.cuh"

namespace qmv {

// Q8_0: lane i owns element i of the block.
__global__ void k_quant_q8_0(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblk)
{
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();
    if (b >= nblk) return;
    float v[1] = {x[b * 32 + lane]};
    const float amax = warp_max(fabsf(v[0]));
    float d, id;
    act_scale(amax, d, id);
    tiny_scale_divide(v, d, id);
    const int8_t q = quant1(v[0], id);
    uint8_t* o = out + b * 34;
    o[2 + lane] = (uint8_t)q;
    if (lane == 0) *reinterpret_cast<__half*>(o) = __float2half_rn(d);
}

// Q8_K: lane i owns elements 8i..8i+7.
__global__ void k_quant_q8_k(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblk)
{
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();
    if (b >= nblk) return;
    const float4* xp = reinterpret_cast<const float4*>(x + b * 256 + lane * 8);
    const float4 a = xp[0], c = xp[1];
    float v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
    const float amax = warp_max(m);
    float d, id;
    act_scale(amax, d, id);
    tiny_scale_divide(v, d, id);
    uint32_t w0 = 0, w1 = 0;
    int s = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int8_t q = quant1(v[k], id);
        s += q;
        if (k < 4) w0 |= (uint32_t)(uint8_t)q << (8 * k);
        else w1 |= (uint32_t)(uint8_t)q << (8 * (k - 4));
    }
    uint8_t* o = out + b * 292;
    uint32_t* qw = reinterpret_cast<uint32_t*>(o + 4 + lane * 8);
    qw[0] = w0;
    qw[1] = w1;
    const int pair = s + __shfl_xor_sync(0xffffffffu, s, 1);   // lanes 2g, 2g+1 cover run g of 16
    if ((lane & 1) == 0) reinterpret_cast<int16_t*>(o + 260)[lane >> 1] = (int16_t)pair;
    if (lane == 0) *reinterpret_cast<float*>(o) = d;
}

// MXFP8: eight threads per 32-element block, four elements each; blocks are
// 33 bytes (E8M0 scale | 32 E4M3 codes).
__global__ void k_quant_mxfp8(const float* __restrict__ x, uint8_t* __restrict__ out, int64_t nblk)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t b = g >> 3;
    const int sub = (int)(g & 7);
    pdl_trigger();
    pdl_wait();
    if (b >= nblk) return;   // whole groups of eight leave together
    const float4 v = reinterpret_cast<const float4*>(x + b * 32)[sub];
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    const unsigned group = 0xffu << (threadIdx.x & 24);   // this block's eight lanes
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(group, m, o, 8));
    const int E = mx_scale_exp(m);
    uint8_t* o = out + b * 33;
    o[1 + 4 * sub] = (uint8_t)mx_e4m3(v.x, E);
    o[2 + 4 * sub] = (uint8_t)mx_e4m3(v.y, E);
    o[3 + 4 * sub] = (uint8_t)mx_e4m3(v.z, E);
    o[4 + 4 * sub] = (uint8_t)mx_e4m3(v.w, E);
    if (sub == 0) o[0] = (uint8_t)(E + 127);
}

}  // namespace qmv

int qmv_launch_quantize(int atype, const float* x, void* xq, int64_t n, bool pdl, cudaStream_t st)
{
    using namespace qmv;
    const int bs = atype == QMV_Q8_K ? 256 : 32;
    const int64_t nblk = n / bs;
    if (nblk == 0) return 0;
    if (atype == QMV_MXFP8) {
        const int64_t threads = nblk * 8;
        return launch_ex(k_quant_mxfp8, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, pdl, x,
                         static_cast<uint8_t*>(xq), nblk) == cudaSuccess
                   ? 0
                   : -1;
    }
    const int warps = 8;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((nblk + warps - 1) / warps));
    cfg.blockDim = dim3(warps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    uint8_t* out = static_cast<uint8_t*>(xq);
    const cudaError_t e = atype == QMV_Q8_0 ? cudaLaunchKernelEx(&cfg, k_quant_q8_0, x, out, nblk)
                                            : cudaLaunchKernelEx(&cfg, k_quant_q8_k, x, out, nblk);
    return e == cudaSuccess ? 0 : -1;
}
