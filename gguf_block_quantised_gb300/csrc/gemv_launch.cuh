// gemv_launch.cuh -- plan and launch the decode matvec kernels of one format.
#pragma once

#include "gemv.cuh"
#include "runtime.cuh"

namespace qmv {

constexpr int kChunkTargetBytes = 2560;          // per row segment of a stage
constexpr size_t kXhatMaxBytes = 96 * 1024;      // staged activations per CTA
constexpr size_t kSmemTwoPerSm = 112 * 1024;     // two CTAs per SM
constexpr size_t kSmemOnePerSm = 227 * 1024;

inline int act_block_bytes(int wtype)
{
    return (wtype == QMV_Q4_K || wtype == QMV_Q6_K) ? 292 : 34;
}

template <int T>
inline bool plan_gemv(bool a8, int64_t rows, int64_t cols, int n_vec, GemvPlan& pl)
{
    using F = Fmt<T>;
    const int nb = (int)(cols / F::BS);
    if ((int64_t)nb * F::BB <= kChunkTargetBytes) {
        pl.kb = nb;
    } else {
        const int unit_blocks = 32 / F::UPB;   // 32 lane-units per K-chunk step
        const int m = kChunkTargetBytes / (unit_blocks * F::BB);
        pl.kb = min(nb, (m > 0 ? m : 1) * unit_blocks);
    }
    pl.n_chunks = (nb + pl.kb - 1) / pl.kb;
    pl.seg_cap = (uint32_t)(((size_t)pl.kb * F::BB + 48 + 15) & ~size_t(15));
    const size_t stage = (size_t)pl.seg_cap * kGemvRows;
    int g = n_vec < 16 ? n_vec : 16;
    if (g < 1) g = 1;
    while (g > 1 && xhat_bytes(T, a8, g, (int)cols) > kXhatMaxBytes) --g;
    pl.group = g;
    pl.xhat_bytes = (uint32_t)xhat_bytes(T, a8, g, (int)cols);
    const size_t base = 128 + ((pl.xhat_bytes + 127) & ~size_t(127));
    int S = base < kSmemTwoPerSm ? (int)((kSmemTwoPerSm - base) / stage) : 0;
    if (S < 3) S = base < kSmemOnePerSm ? (int)((kSmemOnePerSm - base) / stage) : 0;
    if (S < 2) return false;
    if (S > kMaxStages) S = kMaxStages;
    pl.stages = S;
    pl.smem = (uint32_t)(base + S * stage);
    return true;
}

template <int T, bool A8, int NV>
inline int launch_gemv_nv(const GemvParams& p, const GemvPlan& pl, cudaStream_t st)
{
    auto* k = &k_gemv<T, A8, NV>;
    const int occ = prepare_kernel(k, kGemvThreads, pl.smem);
    const int64_t n_tiles = (p.rows + kGemvRows - 1) / kGemvRows;
    int64_t grid = (int64_t)num_sms() * occ;
    if (grid > n_tiles) grid = n_tiles;
    k<<<(unsigned)grid, kGemvThreads, pl.smem, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

template <int T, bool A8>
inline int launch_gemv_group(const GemvParams& p, const GemvPlan& pl, cudaStream_t st)
{
    if (p.nv <= 1) return launch_gemv_nv<T, A8, 1>(p, pl, st);
    if (p.nv <= 2) return launch_gemv_nv<T, A8, 2>(p, pl, st);
    if (p.nv <= 4) return launch_gemv_nv<T, A8, 4>(p, pl, st);
    if (p.nv <= 8) return launch_gemv_nv<T, A8, 8>(p, pl, st);
    return launch_gemv_nv<T, A8, 16>(p, pl, st);
}

// Returns 0, -2 (shape beyond the shared-memory plan) or -6 (launch failure).
template <int T>
inline int launch_gemv_t(bool a8, const void* W, int64_t rows, int64_t cols, const void* x, float* y, int n_vec,
                         cudaStream_t st)
{
    using F = Fmt<T>;
    if (rows == 0 || n_vec == 0) return 0;
    GemvPlan pl;
    if (!plan_gemv<T>(a8, rows, cols, n_vec, pl)) return -2;
    GemvParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.rows = rows;
    p.nb = (int)(cols / F::BS);
    p.rb = (int64_t)p.nb * F::BB;
    p.total = rows * p.rb;
    p.cols = (int)cols;
    p.kb = pl.kb;
    p.n_chunks = pl.n_chunks;
    p.stages = pl.stages;
    p.seg_cap = pl.seg_cap;
    p.xhat_bytes = pl.xhat_bytes;
    p.status = status_word();
    const size_t xrow = a8 ? (size_t)p.nb * act_block_bytes(T) : (size_t)cols * 4;
    for (int v0 = 0; v0 < n_vec; v0 += pl.group) {
        p.nv = min(pl.group, n_vec - v0);
        p.x = static_cast<const uint8_t*>(x) + (size_t)v0 * xrow;
        p.y = y + (int64_t)v0 * rows;
        const int rc = a8 ? launch_gemv_group<T, true>(p, pl, st) : launch_gemv_group<T, false>(p, pl, st);
        if (rc) return rc;
    }
    return 0;
}

}  // namespace qmv

#define QMV_GEMV_INSTANTIATE(T, NAME)                                                                     \
    int NAME(bool a8, const void* W, int64_t rows, int64_t cols, const void* x, float* y, int n_vec,      \
             cudaStream_t st)                                                                              \
    {                                                                                                      \
        return qmv::launch_gemv_t<T>(a8, W, rows, cols, x, y, n_vec, st);                                  \
    }
