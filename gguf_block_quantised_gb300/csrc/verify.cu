// verify.cu -- dequantisation to fp32 and the per-block integer dots of the
// fused W4A8 product ("Architecture" page, "The package map": pkg/quant owns
// "block layouts, dequantisation, and the fused W4A8 kernels every one of them
// is tested against").
//
// Both kernels decode with the same per-format unit routines (formats.cuh) the
// matvec kernels use, so checking these outputs bit for bit checks the integer
// path of every matvec.  They read blocks with byte loads into a 16-byte
// aligned local copy; speed is not their purpose.
#include "formats.cuh"

namespace qmv {

template <int T>
__device__ __forceinline__ void copy_block(const uint8_t* src, uint8_t* dst)
{
#pragma unroll 4
    for (int i = 0; i < Fmt<T>::BB; ++i) dst[i] = src[i];
#pragma unroll
    for (int i = Fmt<T>::BB; i < Fmt<T>::BB + 8; ++i) dst[i] = 0;
}

// Element index of byte j of code word k of unit `sub`.
template <int T>
__device__ __forceinline__ int elem_of(int sub, int k, int j)
{
    if constexpr (T == QMV_MXFP4) {
        const int p = 4 * k + j;
        return (p & 1) ? 16 + (p >> 1) : (p >> 1);
    } else {
        return 4 * k + j;
    }
}

template <int T>
__global__ void k_dequant(const uint8_t* __restrict__ W, int64_t rows, int cols, float* __restrict__ out)
{
    using F = Fmt<T>;
    const int nb = cols / F::BS;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * nb) return;
    const int64_t r = i / nb;
    const int b = (int)(i % nb);
    __align__(16) uint8_t buf[Fmt<T>::BB + 24];
    copy_block<T>(W + i * F::BB, buf);
    float* o = out + r * cols + (int64_t)b * F::BS;
    for (int sub = 0; sub < F::UPB; ++sub) {
        typename F::W w;
        F::load(buf, sub, w);
        if constexpr (plain_rt(T)) {
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = w.w[k];
        } else if constexpr (F::BS == 32) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t byte = (w.code(k) >> (8 * j)) & 0xffu;
                    const int q = F::SIGNED ? (int)(int8_t)byte : (int)byte - F::OFF;
                    if constexpr (F::MIN) o[elem_of<T>(sub, k, j)] = __fmaf_rn(w.d, (float)q, w.m);   // one rounding
                    else o[elem_of<T>(sub, k, j)] = w.d * (float)q;   // exact: <= 24 significant bits
                }
        } else if constexpr (T == QMV_Q4_K || T == QMV_Q5_K) {
            constexpr uint32_t mask = T == QMV_Q5_K ? 31u : 15u;
            const float D0 = w.d * (float)w.sc0, D1 = w.d * (float)w.sc1;       // exact
            const float M0 = w.dmin * (float)w.m0, M1 = w.dmin * (float)w.m1;   // exact
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    o[64 * sub + 4 * k + j] = __fmaf_rn(D0, (float)((w.lo[k] >> (8 * j)) & mask), -M0);
                    o[64 * sub + 32 + 4 * k + j] = __fmaf_rn(D1, (float)((w.hi[k] >> (8 * j)) & mask), -M1);
                }
        } else if constexpr (T == QMV_Q2_K || T == QMV_Q3_K) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float D = w.d * (float)w.sc[r];   // exact
                const float M = T == QMV_Q2_K ? w.dmin * (float)w.m[r] : 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = (int)((w.c[r >> 1][4 * (r & 1) + (i >> 2)] >> (8 * (i & 3))) & 0xffu);
                    o[64 * sub + 16 * r + i] = T == QMV_Q2_K ? __fmaf_rn(D, (float)c, -M) : D * (float)(c - 4);
                }
            }
        } else {   // Q6_K
            const int h = sub >> 1, lh = sub & 1;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float D = w.d * (float)w.sc[g];   // exact
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[128 * h + 32 * g + 16 * lh + 4 * k + j] =
                            D * (float)((int)((w.g[g][k] >> (8 * j)) & 63u) - 32);
            }
        }
    }
}

// One thread per (vector, row, block).
template <int T>
__global__ void k_block_dots(const uint8_t* __restrict__ W, int64_t rows, int cols, const uint8_t* __restrict__ xq,
                             int n_vec, int32_t* __restrict__ out)
{
    using F = Fmt<T>;
    using O = Ops<T>;
    const int nb = cols / F::BS;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n_vec * rows * nb) return;
    const int b = (int)(i % nb);
    const int64_t r = (i / nb) % rows;
    const int v = (int)(i / ((int64_t)nb * rows));
    __align__(16) uint8_t buf[Fmt<T>::BB + 24];
    copy_block<T>(W + (r * nb + b) * F::BB, buf);

    // Stage this activation block in the matvec kernels' shared-memory layout.
    __align__(16) uint8_t codes[F::BS == 32 ? kBPitch : kKPitch];
    float d;
    int sum32 = 0;
    __align__(16) int16_t bsum[16];
    XView X{};
    X.cols = F::BS;
    X.nb = 1;
    X.codes = codes;
    X.d = &d;
    if constexpr (F::BS == 32) {
        const uint8_t* a = xq + ((int64_t)v * nb + b) * 34;
        d = half_bits_to_float((uint32_t)a[0] | ((uint32_t)a[1] << 8));
        for (int k = 0; k < 32; ++k) {
            codes[staged_pos<T>(k)] = a[2 + k];
            sum32 += (int)(int8_t)a[2 + k];
        }
        X.sum32 = &sum32;
    } else {
        const uint8_t* a = xq + ((int64_t)v * nb + b) * 292;
        uint32_t u = (uint32_t)a[0] | ((uint32_t)a[1] << 8) | ((uint32_t)a[2] << 16) | ((uint32_t)a[3] << 24);
        d = __uint_as_float(u);
        for (int k = 0; k < 256; ++k) codes[kquant_run_pos<T>(k >> 4) + (k & 15)] = a[4 + k];
        for (int g = 0; g < 16; ++g) bsum[g] = (int16_t)((uint32_t)a[260 + 2 * g] | ((uint32_t)a[261 + 2 * g] << 8));
        X.bsum = bsum;
    }
    int S = 0, Mn = 0;
    for (int sub = 0; sub < F::UPB; ++sub) {
        typename F::W w;
        typename F::XA8 x;
        F::load(buf, sub, w);
        F::load_x_a8(X, 0, 0, sub, x);
        int s, m;
        O::ints(w, x, s, m);
        S += s;
        Mn += m;
    }
    out[2 * i] = S;
    out[2 * i + 1] = Mn;
}

template <int T>
static int launch_dequant_t(const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t st)
{
    const int64_t n = rows * (cols / Fmt<T>::BS);
    if (n == 0) return 0;
    k_dequant<T><<<(unsigned)((n + 127) / 128), 128, 0, st>>>(static_cast<const uint8_t*>(W), rows, (int)cols, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

template <int T>
static int launch_dots_t(const void* W, int64_t rows, int64_t cols, const void* xq, int n_vec, int32_t* out,
                         cudaStream_t st)
{
    const int64_t n = (int64_t)n_vec * rows * (cols / Fmt<T>::BS);
    if (n == 0) return 0;
    k_block_dots<T><<<(unsigned)((n + 127) / 128), 128, 0, st>>>(static_cast<const uint8_t*>(W), rows, (int)cols,
                                                                   static_cast<const uint8_t*>(xq), n_vec, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace qmv

int qmv_launch_dequant(int t, const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t st)
{
    using namespace qmv;
    switch (t) {
    case QMV_Q4_0: return launch_dequant_t<QMV_Q4_0>(W, rows, cols, out, st);
    case QMV_Q5_0: return launch_dequant_t<QMV_Q5_0>(W, rows, cols, out, st);
    case QMV_Q8_0: return launch_dequant_t<QMV_Q8_0>(W, rows, cols, out, st);
    case QMV_MXFP4: return launch_dequant_t<QMV_MXFP4>(W, rows, cols, out, st);
    case QMV_Q4_K: return launch_dequant_t<QMV_Q4_K>(W, rows, cols, out, st);
    case QMV_Q6_K: return launch_dequant_t<QMV_Q6_K>(W, rows, cols, out, st);
    case QMV_Q4_1: return launch_dequant_t<QMV_Q4_1>(W, rows, cols, out, st);
    case QMV_Q5_1: return launch_dequant_t<QMV_Q5_1>(W, rows, cols, out, st);
    case QMV_Q8_1: return launch_dequant_t<QMV_Q8_1>(W, rows, cols, out, st);
    case QMV_Q2_K: return launch_dequant_t<QMV_Q2_K>(W, rows, cols, out, st);
    case QMV_Q3_K: return launch_dequant_t<QMV_Q3_K>(W, rows, cols, out, st);
    case QMV_Q5_K: return launch_dequant_t<QMV_Q5_K>(W, rows, cols, out, st);
    case QMV_F32: return launch_dequant_t<QMV_F32>(W, rows, cols, out, st);
    case QMV_F16: return launch_dequant_t<QMV_F16>(W, rows, cols, out, st);
    case QMV_BF16: return launch_dequant_t<QMV_BF16>(W, rows, cols, out, st);
    default: return -3;
    }
}

int qmv_launch_block_dots(int t, const void* W, int64_t rows, int64_t cols, const void* xq, int n_vec,
                          int32_t* out, cudaStream_t st)
{
    using namespace qmv;
    switch (t) {
    case QMV_Q4_0: return launch_dots_t<QMV_Q4_0>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q5_0: return launch_dots_t<QMV_Q5_0>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q8_0: return launch_dots_t<QMV_Q8_0>(W, rows, cols, xq, n_vec, out, st);
    case QMV_MXFP4: return launch_dots_t<QMV_MXFP4>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q4_K: return launch_dots_t<QMV_Q4_K>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q6_K: return launch_dots_t<QMV_Q6_K>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q4_1: return launch_dots_t<QMV_Q4_1>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q5_1: return launch_dots_t<QMV_Q5_1>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q8_1: return launch_dots_t<QMV_Q8_1>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q2_K: return launch_dots_t<QMV_Q2_K>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q3_K: return launch_dots_t<QMV_Q3_K>(W, rows, cols, xq, n_vec, out, st);
    case QMV_Q5_K: return launch_dots_t<QMV_Q5_K>(W, rows, cols, xq, n_vec, out, st);
    default: return -3;
    }
}
