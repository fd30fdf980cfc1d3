// quant_w.cu -- weights (fp32 or bf16) -> Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0 and
// Q4_K / Q5_K / Q6_K blocks ("Models and formats" page, "Tensor formats": the
// quantiser writes Q4_0/1, Q5_0/1, Q8_0 and the K-quants).
//
// The pages print no procedure; each format follows the plainest reading,
// one pass of min/max rules per run with no search:
//   Q4_0 / Q5_0: m = the signed value of largest magnitude (the first on
//     ties); d = m / -half (half = 8 or 16); code = trunc(clamp(x/d + half +
//     0.5, 0, 2*half - 1)).  The largest-magnitude element lands on code 0.
//   Q8_0: the symmetric 8-bit form of the activation quantiser, d = amax/127,
//     code = round(x/d).
//   Q4_1 / Q5_1: m = min x, d = (max x - m) / (2^bits - 1), code =
//     trunc(clamp((x - m)/d + 0.5, 0, 2^bits - 1)); w = d*q + m.
//   Q4_K / Q5_K: per 32-element sub-block lo = min(0, min x), s = (max x - lo)
//     / top, z = -lo; d = max s / 63, dmin = max z / 63; six-bit sc = round(s/d),
//     m = round(z/dmin); codes round((x + dmin*m) / (d*sc)) on the stored fp16
//     scales, clamped to 0..top.
//   Q6_K: per 16-element run the signed extreme e, s = e / -32; the s of
//     largest magnitude s_e, d = s_e / -128; int8 sc = round(s/d); codes
//     round(x / (d*sc)) + 32, clamped to 0..63.
// Every division is a multiplication by the fp32 reciprocal (the quotient
// itself when the reciprocal overflows), rounding is half away from zero, and
// every step is one IEEE fp32 rounding (__fdiv_rn, __fmul_rn, __fadd_rn; no
// contraction), so the codes do not depend on the thread layout.  Blocks are
// written with 16-bit stores (the output is 2-byte aligned).
//
// 32-element formats: eight threads per block, four weights each (one 16-byte
// fp32 or 8-byte bf16 load); the block's extremes are xor reductions over the
// eight lanes.  K-quants: one warp per 256-element super-block, eight weights
// per lane; the codes go through shared memory to be packed.  Each pass reads
// 4 (fp32) or 2 (bf16) bytes and writes the block bytes per weight: bound by
// HBM.
#include <type_traits>

#include "common.cuh"

namespace qmv {

// Four consecutive input weights starting at element 4*i.
template <bool BF>
__device__ __forceinline__ void load4(const void* x, int64_t i, float (&v)[4])
{
    if constexpr (BF) {
        const uint2 u = reinterpret_cast<const uint2*>(x)[i];
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const float4 f = reinterpret_cast<const float4*>(x)[i];
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
}

__device__ __forceinline__ uint32_t f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
__device__ __forceinline__ float f16_round(float v) { return __half2float(__float2half_rn(v)); }

// round half away from zero, clamped to [lo, hi], as an int
__device__ __forceinline__ int round_clamp(float v, float lo, float hi)
{
    return (int)fminf(fmaxf(roundf(v), lo), hi);
}

// v * (1/s) with id = 1/s (v / s when 1/s overflowed); 0 when s = 0
__device__ __forceinline__ float scaled(float v, float s, float id)
{
    if (s == 0.f) return 0.f;
    return isinf(id) ? __fdiv_rn(v, s) : __fmul_rn(v, id);
}

// ---- the 32-element formats: eight threads per block --------------------------------
// One block's share of thread `part` (weights 4*part .. +3 in v); every lane of
// the warp calls it (the reductions are shuffles over the block's eight lanes).
template <int T>
__device__ __forceinline__ void quant_w32_item(float (&v)[4], int64_t blk, int part, bool valid,
                                               uint8_t* __restrict__ out)
{
    constexpr bool Q0 = T == QMV_Q4_0 || T == QMV_Q5_0, Q1 = T == QMV_Q4_1 || T == QMV_Q5_1, Q8 = T == QMV_Q8_0;
    constexpr int BITS = (T == QMV_Q4_0 || T == QMV_Q4_1) ? 4 : 5;
    constexpr int BB = T == QMV_Q4_0 ? 18 : T == QMV_Q5_0 ? 22 : T == QMV_Q4_1 ? 20 : T == QMV_Q5_1 ? 24 : 34;
    constexpr float kHalf = (float)(1 << (BITS - 1));
    constexpr float kTop = (float)((1 << BITS) - 1);

    float d = 0.f, id = 0.f, mn = 0.f;
    uint32_t codes = 0, hi_bits = 0;
    if constexpr (Q0) {
        // The first element of largest magnitude: strictly larger magnitudes
        // win, and among equal ones the lower index (an all-zero block keeps +0).
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
        d = __fdiv_rn(m, -kHalf);
        id = d == 0.f ? 0.f : __fdiv_rn(1.f, d);
        tiny_scale_divide(v, d, id);   // |d| below 2^-128: the codes come from x / d
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float t = __fadd_rn(__fmul_rn(v[k], id), kHalf + 0.5f);
            t = fmaxf(fminf(t, kTop), 0.f);
            const uint32_t c = (uint32_t)__float2int_rz(t);
            codes |= (c & 15u) << (8 * k);
            hi_bits |= ((c >> 4) & 1u) << (4 * part + k);
        }
    } else if constexpr (Q1) {
        // min and max, the first element on ties (+0 and -0 compare equal, and
        // the one met first is kept, as a scan from element 0 keeps it)
        float lo = v[0], hi = v[0];
        int li = 4 * part, hj = 4 * part;
#pragma unroll
        for (int k = 1; k < 4; ++k) {
            if (v[k] < lo) { lo = v[k]; li = 4 * part + k; }
            if (v[k] > hi) { hi = v[k]; hj = 4 * part + k; }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const float ol = __shfl_xor_sync(0xffffffffu, lo, o), oh = __shfl_xor_sync(0xffffffffu, hi, o);
            const int oli = __shfl_xor_sync(0xffffffffu, li, o), ohj = __shfl_xor_sync(0xffffffffu, hj, o);
            if (ol < lo || (ol == lo && oli < li)) { lo = ol; li = oli; }
            if (oh > hi || (oh == hi && ohj < hj)) { hi = oh; hj = ohj; }
        }
        mn = lo;
        d = __fdiv_rn(__fsub_rn(hi, lo), kTop);
        id = d == 0.f ? 0.f : __fdiv_rn(1.f, d);
        float u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) u[k] = __fsub_rn(v[k], mn);
        tiny_scale_divide(u, d, id);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float t = __fadd_rn(d == 0.f ? 0.f : __fmul_rn(u[k], id), 0.5f);
            t = fmaxf(fminf(t, kTop), 0.f);
            const uint32_t c = (uint32_t)__float2int_rz(t);
            codes |= (c & 15u) << (8 * k);
            hi_bits |= ((c >> 4) & 1u) << (4 * part + k);
        }
    } else {   // Q8_0
        float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        act_scale(a, d, id);
        tiny_scale_divide(v, d, id);
#pragma unroll
        for (int k = 0; k < 4; ++k) codes |= (uint32_t)(uint8_t)quant1(v[k], id) << (8 * k);
    }
    // Byte j of the nibbles pairs element j (thread j/4) with element j + 16
    // (thread 4 + j/4).
    const uint32_t other = __shfl_xor_sync(0xffffffffu, codes, 4);
    if constexpr (BITS == 5 && !Q8) {
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) hi_bits |= __shfl_xor_sync(0xffffffffu, hi_bits, o);
    }
    if (!valid) return;
    uint16_t* o = reinterpret_cast<uint16_t*>(out + blk * BB);
    if constexpr (Q8) {
        if (part == 0) o[0] = (uint16_t)f16_bits(d);
        o[1 + 2 * part] = (uint16_t)(codes & 0xffffu);
        o[2 + 2 * part] = (uint16_t)(codes >> 16);
        return;
    } else {
        constexpr int HEAD = (Q1 ? 2 : 1) + (BITS == 5 ? 2 : 0);   // 16-bit words before the nibbles
        if (part == 0) {
            o[0] = (uint16_t)f16_bits(d);
            if constexpr (Q1) o[1] = (uint16_t)f16_bits(mn);
            if constexpr (BITS == 5) {
                o[HEAD - 2] = (uint16_t)(hi_bits & 0xffffu);
                o[HEAD - 1] = (uint16_t)(hi_bits >> 16);
            }
        }
        if (part < 4) {
            const uint32_t b = (codes & 0x0f0f0f0fu) | ((other & 0x0f0f0f0fu) << 4);   // bytes 4*part .. +3
            uint16_t* qs = o + HEAD + 2 * part;
            qs[0] = (uint16_t)(b & 0xffffu);
            qs[1] = (uint16_t)(b >> 16);
        }
    }
}

// Each thread takes ITEMS blocks a grid apart, all its loads issued first (more
// bytes in flight per thread: a bf16 thread reads only 8 bytes per block).
template <int T, bool BF, int ITEMS>
__global__ void __launch_bounds__(256) k_quant_w32(const void* __restrict__ x, uint8_t* __restrict__ out,
                                                   int64_t nblk)
{
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;   // a multiple of 8: blocks stay whole
    float v[ITEMS][4];
    bool valid[ITEMS];
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        const int64_t i = i0 + j * stride;
        valid[j] = (i >> 3) < nblk;   // the same for the eight lanes of a block
#pragma unroll
        for (int k = 0; k < 4; ++k) v[j][k] = 0.f;
        if (valid[j]) load4<BF>(x, i, v[j]);
    }
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        const int64_t i = i0 + j * stride;
        quant_w32_item<T>(v[j], i >> 3, (int)(i & 7), valid[j], out);
    }
}

// ---- the K-quants: one warp per 256-element super-block -------------------------------
constexpr int kKWarps = 8;

template <int T, bool BF>
__global__ void __launch_bounds__(32 * kKWarps) k_quant_wk(const void* __restrict__ x, uint8_t* __restrict__ out,
                                                           int64_t nblk)
{
    constexpr int BB = T == QMV_Q4_K ? 144 : T == QMV_Q5_K ? 176 : 210;
    __shared__ __align__(16) uint8_t sq[kKWarps][256];    // codes of the super-block
    __shared__ __align__(16) uint8_t sb[kKWarps][224];    // the packed block
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t blk = (int64_t)blockIdx.x * kKWarps + w;
    if (blk >= nblk) return;   // warp-uniform
    float v[8];
    {
        float a[4], b[4];
        load4<BF>(x, blk * 64 + 2 * lane, a);
        load4<BF>(x, blk * 64 + 2 * lane + 1, b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = a[k];
            v[4 + k] = b[k];
        }
    }
    uint8_t* q = sq[w];
    uint8_t* o = sb[w];
    if constexpr (T == QMV_Q4_K || T == QMV_Q5_K) {
        constexpr float top = T == QMV_Q4_K ? 15.f : 31.f;
        // sub-block j = lane / 4: lo = min(0, min x), hi = max x
        float lo = 0.f, hi = v[0];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (v[k] < lo) lo = v[k];
            if (v[k] > hi) hi = v[k];
        }
#pragma unroll
        for (int o2 = 1; o2 < 4; o2 <<= 1) {
            const float ol = __shfl_xor_sync(0xffffffffu, lo, o2), oh = __shfl_xor_sync(0xffffffffu, hi, o2);
            if (ol < lo) lo = ol;
            if (oh > hi) hi = oh;
        }
        const float s = __fdiv_rn(__fsub_rn(hi, lo), top), z = -lo;
        // the largest s and z over the sub-blocks, from +0 (a -0 never wins)
        float smax = s > 0.f ? s : 0.f, zmax = z > 0.f ? z : 0.f;
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, smax, o2), oz = __shfl_xor_sync(0xffffffffu, zmax, o2);
            if (os > smax) smax = os;
            if (oz > zmax) zmax = oz;
        }
        const float d = __fdiv_rn(smax, 63.f), dmin = __fdiv_rn(zmax, 63.f);
        const float id = d == 0.f ? 0.f : __fdiv_rn(1.f, d), idm = dmin == 0.f ? 0.f : __fdiv_rn(1.f, dmin);
        const int sc = round_clamp(scaled(s, d, id), 0.f, 63.f), m = round_clamp(scaled(z, dmin, idm), 0.f, 63.f);
        const float D = __fmul_rn(f16_round(d), (float)sc), M = __fmul_rn(f16_round(dmin), (float)m);   // exact
        const float iD = D == 0.f ? 0.f : __fdiv_rn(1.f, D);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            q[8 * lane + k] = (uint8_t)round_clamp(scaled(__fadd_rn(v[k], M), D, iD), 0.f, top);
        // scale field: lane 4j holds sub-block j's sc, m
        int scj[8], mj[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            scj[j] = __shfl_sync(0xffffffffu, sc, 4 * j);
            mj[j] = __shfl_sync(0xffffffffu, m, 4 * j);
        }
        __syncwarp();
        if (lane == 0) {
            *reinterpret_cast<uint16_t*>(o) = (uint16_t)f16_bits(d);
            *reinterpret_cast<uint16_t*>(o + 2) = (uint16_t)f16_bits(dmin);
        }
        if (lane < 4) {
            const int j = lane;
            o[4 + j] = (uint8_t)((scj[j] & 63) | ((scj[j + 4] >> 4) << 6));
            o[8 + j] = (uint8_t)((mj[j] & 63) | ((mj[j + 4] >> 4) << 6));
            o[12 + j] = (uint8_t)((scj[j + 4] & 15) | ((mj[j + 4] & 15) << 4));
        }
        // nibbles: byte 32c + l = code 64c + l (low) | code 64c + 32 + l (high);
        // Q5_K fifth bits: bit 2c (2c+1) of byte l from code 64c + l (64c + 32 + l)
        const int l = lane;
        uint32_t qh = 0;
        uint8_t* qs = o + (T == QMV_Q5_K ? 48 : 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t a = q[64 * c + l], b = q[64 * c + 32 + l];
            qs[32 * c + l] = (uint8_t)((a & 15u) | ((b & 15u) << 4));
            qh |= ((a >> 4) & 1u) << (2 * c) | ((b >> 4) & 1u) << (2 * c + 1);
        }
        if constexpr (T == QMV_Q5_K) o[16 + l] = (uint8_t)qh;
    } else {   // Q6_K: run j = lane / 2
        float a = 0.f, e = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (fabsf(v[k]) > a) {
                a = fabsf(v[k]);
                e = v[k];
            }
        {   // the pair's first element of largest magnitude: lane 2j's elements come first
            const float oa = __shfl_xor_sync(0xffffffffu, a, 1), oe = __shfl_xor_sync(0xffffffffu, e, 1);
            const bool first = (lane & 1) == 0;
            if (oa > a || (oa == a && !first)) {
                a = oa;
                e = oe;
            }
        }
        const float s = __fdiv_rn(e, -32.f);
        // the s of largest magnitude, the first run on ties, from +0
        float sa = fabsf(s), se = s;
        int sj = lane >> 1;
        if (!(sa > 0.f)) { sa = 0.f; se = 0.f; sj = 16; }
#pragma unroll
        for (int o2 = 2; o2 < 32; o2 <<= 1) {
            const float oa = __shfl_xor_sync(0xffffffffu, sa, o2), os = __shfl_xor_sync(0xffffffffu, se, o2);
            const int oj = __shfl_xor_sync(0xffffffffu, sj, o2);
            if (oa > sa || (oa == sa && oj < sj)) {
                sa = oa;
                se = os;
                sj = oj;
            }
        }
        const float d = __fdiv_rn(se, -128.f);
        const float id = d == 0.f ? 0.f : __fdiv_rn(1.f, d);
        const int sc = round_clamp(scaled(s, d, id), -128.f, 127.f);
        const float D = __fmul_rn(f16_round(d), (float)sc);
        const float iD = D == 0.f ? 0.f : __fdiv_rn(1.f, D);
#pragma unroll
        for (int k = 0; k < 8; ++k) q[8 * lane + k] = (uint8_t)(round_clamp(scaled(v[k], D, iD), -32.f, 31.f) + 32);
        __syncwarp();
        // ql[64h + l], ql[64h + 32 + l], qh[32h + l] from codes 128h + l + {0, 32, 64, 96}
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t q0 = q[128 * h + lane], q1 = q[128 * h + lane + 32], q2 = q[128 * h + lane + 64],
                           q3 = q[128 * h + lane + 96];
            o[64 * h + lane] = (uint8_t)((q0 & 15u) | ((q2 & 15u) << 4));
            o[64 * h + 32 + lane] = (uint8_t)((q1 & 15u) | ((q3 & 15u) << 4));
            o[128 + 32 * h + lane] = (uint8_t)((q0 >> 4) | ((q1 >> 4) << 2) | ((q2 >> 4) << 4) | ((q3 >> 4) << 6));
        }
        if ((lane & 1) == 0) o[192 + (lane >> 1)] = (uint8_t)(int8_t)sc;
        if (lane == 0) *reinterpret_cast<uint16_t*>(o + 208) = (uint16_t)f16_bits(d);
    }
    __syncwarp();
    // the block out, 16 bits at a time
    uint16_t* dst = reinterpret_cast<uint16_t*>(out + blk * BB);
    const uint16_t* srcw = reinterpret_cast<const uint16_t*>(o);
    for (int k = lane; k < BB / 2; k += 32) dst[k] = srcw[k];
}

template <int T, bool BF>
static int launch_w32(const void* W, int64_t n, void* out, cudaStream_t st)
{
    const int64_t nblk = n / 32;
    if (nblk == 0) return 0;
    constexpr int ITEMS = BF ? 4 : 2;
    const int64_t threads = (nblk * 8 + ITEMS - 1) / ITEMS;
    k_quant_w32<T, BF, ITEMS><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(W, static_cast<uint8_t*>(out),
                                                                                nblk);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <int T, bool BF>
static int launch_wk(const void* W, int64_t n, void* out, cudaStream_t st)
{
    const int64_t nblk = n / 256;
    if (nblk == 0) return 0;
    k_quant_wk<T, BF><<<(unsigned)((nblk + kKWarps - 1) / kKWarps), 32 * kKWarps, 0, st>>>(
        W, static_cast<uint8_t*>(out), nblk);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <bool BF>
static int launch_w(int wtype, const void* W, int64_t n, void* out, cudaStream_t st)
{
    switch (wtype) {
    case QMV_Q4_0: return launch_w32<QMV_Q4_0, BF>(W, n, out, st);
    case QMV_Q5_0: return launch_w32<QMV_Q5_0, BF>(W, n, out, st);
    case QMV_Q8_0: return launch_w32<QMV_Q8_0, BF>(W, n, out, st);
    case QMV_Q4_1: return launch_w32<QMV_Q4_1, BF>(W, n, out, st);
    case QMV_Q5_1: return launch_w32<QMV_Q5_1, BF>(W, n, out, st);
    case QMV_Q4_K: return launch_wk<QMV_Q4_K, BF>(W, n, out, st);
    case QMV_Q5_K: return launch_wk<QMV_Q5_K, BF>(W, n, out, st);
    case QMV_Q6_K: return launch_wk<QMV_Q6_K, BF>(W, n, out, st);
    default: return -3;
    }
}

}  // namespace qmv

// Returns 0, -3 (type) or -1 on a launch failure.  bf16: the weights are
// bfloat16 values instead of fp32.
int qmv_launch_quantize_weights(int wtype, bool bf16, const void* W, int64_t n, void* out, cudaStream_t st)
{
    return bf16 ? qmv::launch_w<true>(wtype, W, n, out, st) : qmv::launch_w<false>(wtype, W, n, out, st);
}
