// gemv_launch.cuh -- plan and launch the decode matvec kernels of one format.
#pragma once

#include "gemv.cuh"
#include "moe.cuh"
#include "runtime.cuh"

namespace qmv {

// Bytes of one row segment of a stage.  Longer segments give each consumer
// lane more units per pipeline item (fewer barrier round trips per byte);
// Q4_K keeps shorter ones, whose stages are small enough for two CTAs per SM
// with two rows per warp on its long rows.
template <int T>
constexpr int chunk_target_bytes()
{
    return T == QMV_Q4_K ? 2560 : 4096;
}
constexpr size_t kXhatMaxBytes = 176 * 1024;     // staged activations per CTA
constexpr size_t kSmemTwoPerSm = 112 * 1024;     // two CTAs per SM
constexpr size_t kSmemOnePerSm = 227 * 1024;

inline int act_block_bytes(int wtype)
{
    return kq_rt(wtype) ? 292 : 34;
}

// Rows a consumer warp decodes at once: fewer as the vector count (and with
// it the accumulator count RIF x NV) grows.  K-quants with more than four
// vectors decode two rows at once when a row is one K-chunk (each staged
// activation load then serves two rows: Q6_K 128256 x 4096 with 16 vectors
// 0.65 -> 0.48 ms), one when rows span several chunks (a multi-chunk row keeps
// its warp's rows in registers, and single rows give twice the tiles there).
template <int T, int NV>
constexpr int rows_in_flight(bool multi_chunk = false)
{
    return Fmt<T>::BS != 256 ? (NV <= 2 ? 4 : 2) : (NV <= 4 || !multi_chunk ? 2 : 1);
}

inline int rows_in_flight_rt(int T, int nv, bool multi_chunk)
{
    const bool b32 = !kq_rt(T);
    const int NV = nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 8 ? 8 : 16;
    return b32 ? (NV <= 2 ? 4 : 2) : (NV <= 4 || !multi_chunk ? 2 : 1);
}

template <int T>
inline bool plan_gemv(bool a8, int64_t rows, int64_t cols, int n_vec, GemvPlan& pl, int max_rpw = 4,
                      int64_t min_tiles = 0)
{
    using F = Fmt<T>;
    const int nb = (int)(cols / F::BS);
    constexpr int kChunkTargetBytes = chunk_target_bytes<T>();
    if ((int64_t)nb * F::BB <= kChunkTargetBytes) {
        pl.kb = nb;
    } else {
        const int unit_blocks = 32 / F::UPB;   // 32 lane-units per K-chunk step
        const int m = kChunkTargetBytes / (unit_blocks * F::BB);
        pl.kb = min(nb, (m > 0 ? m : 1) * unit_blocks);
    }
    pl.n_chunks = (nb + pl.kb - 1) / pl.kb;
    pl.seg_cap = (uint32_t)(((size_t)pl.kb * F::BB + 48 + 15) & ~size_t(15));
    // Largest vector group whose staged activations fit next to at least two
    // stages (three when two CTAs share an SM); then fewer rows per warp.
    int g = n_vec < 16 ? n_vec : 16;
    if (g < 1) g = 1;
    for (;;) {
        // Accumulators stay in registers across K-chunks only for one row
        // group, so a multi-chunk row gives each warp as many rows as this
        // group's kernel decodes at once (smaller groups decode at least as many).
        // With 8-bit activations and one or two vectors (up to eight for the
        // 32-element formats) the kernel's registers allow two CTAs per SM, and tiles that let two CTAs share an SM (three
        // stages each) are preferred over larger tiles with one CTA per SM;
        // otherwise the largest tile wins, with two CTAs per SM if it fits.
        const int rif = rows_in_flight_rt(T, g, pl.n_chunks > 1);
        const bool prefer_two = a8 && (g <= 2 || (F::BS == 32 && g <= 8));   // as two_ctas_per_sm()
        bool found = false;
        for (int pass = prefer_two ? 0 : 2; pass < 3 && !found; ++pass) {
            // Rows per warp: at most the rows the kernel decodes at once when a
            // row spans several chunks (the accumulators then stay in registers
            // across chunks); fewer while the matrix would give fewer than
            // min_tiles tiles (small matrices spread over more SMs).
            int rpw0 = pl.n_chunks > 1 ? rif : max_rpw;
            while (rpw0 > 1 && (rows + kConsumerWarps * rpw0 - 1) / (kConsumerWarps * rpw0) < min_tiles) rpw0 /= 2;
            for (int rpw = rpw0; rpw >= 1; rpw /= 2) {
                const size_t xb = xhat_bytes(T, a8, g, (int)cols);
                if (xb > kXhatMaxBytes && g > 1) break;
                const size_t stage = (size_t)pl.seg_cap * kConsumerWarps * rpw;
                const size_t base = 256 + ((xb + 127) & ~size_t(127));
                // pass 0: two per SM only (tiles of two or more rows per warp may
                // run two stages each: four per SM); 1: one per SM; 2: two if it
                // fits, else one
                int S2 = base < kSmemTwoPerSm ? (int)((kSmemTwoPerSm - base) / stage) : 0;
                int S1 = base < kSmemOnePerSm ? (int)((kSmemOnePerSm - base) / stage) : 0;
                int S = pass == 0 ? (S2 >= (rpw >= 2 ? 2 : 3) ? S2 : 0) : pass == 1 ? S1 : (S2 >= 3 ? S2 : S1);
                if (S >= 2) {
                    if (S > kMaxStages) S = kMaxStages;
                    pl.group = g;
                    pl.rpw = rpw;
                    pl.xhat_bytes = (uint32_t)xb;
                    pl.stages = S;
                    pl.smem = (uint32_t)(base + S * stage);
                    found = true;
                    break;
                }
            }
        }
        if (found) return true;
        if (g == 1) return false;
        --g;
    }

}

template <int T, bool A8, int NV>
inline int launch_gemv_nv(GemvParams p, const GemvPlan& pl, bool pdl, cudaStream_t st)
{
    auto* k = p.n_chunks > 1 ? &k_gemv<T, A8, NV, rows_in_flight<T, NV>(true)>
                             : &k_gemv<T, A8, NV, rows_in_flight<T, NV>(false)>;
    const int occ = prepare_kernel(k, kGemvThreads, pl.smem);
    const int64_t tr = kConsumerWarps * pl.rpw;
    const int64_t n_tiles = (p.rows + tr - 1) / tr;
    int64_t grid = (int64_t)num_sms() * occ;
    if (grid > n_tiles) grid = n_tiles;
    return launch_ex(k, dim3((unsigned)grid), dim3(kGemvThreads), pl.smem, st, pdl, p) == cudaSuccess ? 0 : -6;
}

template <int T, bool A8>
inline int launch_gemv_group(const GemvParams& p, const GemvPlan& pl, bool pdl, cudaStream_t st)
{
    if (p.nv <= 1) return launch_gemv_nv<T, A8, 1>(p, pl, pdl, st);
    if (p.nv <= 2) return launch_gemv_nv<T, A8, 2>(p, pl, pdl, st);
    if (p.nv <= 4) return launch_gemv_nv<T, A8, 4>(p, pl, pdl, st);
    if (p.nv <= 8) return launch_gemv_nv<T, A8, 8>(p, pl, pdl, st);
    return launch_gemv_nv<T, A8, 16>(p, pl, pdl, st);
}

// Returns 0, -2 (shape beyond the shared-memory plan) or -6 (launch failure).
// quant_x: A8 from fp32 activations quantised in the kernel.  pdl: launch as a
// programmatic dependent of the previous kernel on the stream.
template <int T>
inline int launch_gemv_t(bool a8, bool quant_x, bool pdl, const void* W, int64_t rows, int64_t cols, const void* x,
                         float* y, int n_vec, cudaStream_t st)
{
    using F = Fmt<T>;
    if (rows == 0 || n_vec == 0) return 0;
    if constexpr (plain_rt(T)) {
        if (a8) return -3;   // plain weights take fp32 activations only
    }
    GemvPlan pl;
    // Small matrices get shorter tiles so that more SMs take part (the tile
    // shape does not enter the arithmetic of any output).
    if (!plan_gemv<T>(a8, rows, cols, n_vec, pl, 4, (int64_t)num_sms())) return -2;
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
    p.rpw = pl.rpw;
    // One bulk copy per row (into its own slot): measured faster on the lm_head
    // than one large copy of a whole tile of consecutive rows.
    p.quant_x = quant_x ? 1 : 0;
    p.xhat_bytes = pl.xhat_bytes;
    p.status = status_word();
    p.wait_ns = wait_limit_ns(QMV_WAIT_LIMIT_NS);
    const size_t xrow = (a8 && !quant_x) ? (size_t)p.nb * act_block_bytes(T) : (size_t)cols * 4;
    for (int v0 = 0; v0 < n_vec; v0 += pl.group) {
        p.nv = min(pl.group, n_vec - v0);
        p.x = static_cast<const uint8_t*>(x) + (size_t)v0 * xrow;
        p.y = y + (int64_t)v0 * rows;
        int rc;
        if constexpr (plain_rt(T)) rc = launch_gemv_group<T, false>(p, pl, pdl, st);
        else rc = a8 ? launch_gemv_group<T, true>(p, pl, pdl, st) : launch_gemv_group<T, false>(p, pl, pdl, st);
        if (rc) return rc;
    }
    return 0;
}

// ---- mixture of experts -----------------------------------------------------------
template <int T, bool A8, int NV>
inline int launch_moe_nv(const MoeParams& mp, const GemvPlan& pl, int grid_y, int active, int waves,
                         cudaStream_t st)
{
    auto* k = &k_moe_gemv<T, A8, NV, rows_in_flight<T, NV>()>;
    const size_t smem = pl.smem + 256;
    const int occ = prepare_kernel(k, kGemvThreads, smem);
    const int64_t tr = kConsumerWarps * pl.rpw;
    const int64_t n_tiles = (mp.g.rows + tr - 1) / tr;
    int64_t gx = ((int64_t)num_sms() * occ * waves + active - 1) / active;
    if (gx > n_tiles) gx = n_tiles;
    if (gx < 1) gx = 1;
    return launch_ex(k, dim3((unsigned)gx, (unsigned)grid_y), dim3(kGemvThreads), smem, st, true, mp) ==
                   cudaSuccess
               ? 0
               : -6;
}

// Expert matvecs for grouped (token, slot) pairs.  x rows are xrow bytes
// apart; pair p reads row p / kdiv and writes out[p*rows ..].
template <int T>
inline int launch_moe_t(bool a8, bool quant_x, const void* W3d, int n_expert, int64_t rows, int64_t cols,
                        const int* offsets, const int* active_list, const int* perm, const int32_t* ids,
                        bool self_group, int n_pairs, int n_tok, const void* x, size_t xrow, int kdiv, float* out,
                        const float* bias, cudaStream_t st)
{
    using F = Fmt<T>;
    if (rows == 0 || n_pairs == 0) return 0;
    if constexpr (plain_rt(T)) {
        if (a8) return -3;
    }
    GemvPlan pl;
    // Small tiles (as many rows per warp as the kernel decodes at once) so an
    // expert's rows spread over many SMs; the stage ring is sized for that tile.
    // The k slots of a token normally go to k different experts, so an expert
    // holds at most n_tok pairs: the vector group is sized for that (an expert
    // with more pairs takes several groups).
    // Groups of at most 8 pairs: the 8-vector kernel fits two CTAs per SM (the
    // 16-vector one, 157 registers, one), which more than pays for streaming an
    // expert's rows once more when it holds over 8 pairs (gpt-oss layer, A/B:
    // 16 tokens 0.507 -> 0.272 ms, 64 tokens 0.968 -> 0.699, 1024 tokens 10.7 -> 7.4).
    const int cap = n_tok < n_pairs ? n_tok : n_pairs;
    const int gmax = cap < 8 ? (cap > 0 ? cap : 1) : 8;
    if (!plan_gemv<T>(a8, rows, cols, gmax, pl, rows_in_flight_rt(T, gmax, false))) return -2;
    MoeParams mp{};
    GemvParams& p = mp.g;
    p.W = static_cast<const uint8_t*>(W3d);
    p.rows = rows;
    p.nb = (int)(cols / F::BS);
    p.rb = (int64_t)p.nb * F::BB;
    p.total = rows * p.rb;
    p.cols = (int)cols;
    p.kb = pl.kb;
    p.n_chunks = pl.n_chunks;
    p.stages = pl.stages;
    p.seg_cap = pl.seg_cap;
    p.rpw = pl.rpw;
    p.quant_x = quant_x ? 1 : 0;
    p.xhat_bytes = pl.xhat_bytes;
    p.status = status_word();
    p.wait_ns = wait_limit_ns(QMV_WAIT_LIMIT_NS);
    p.x = x;
    mp.expert_bytes = p.total;
    mp.offsets = offsets;
    mp.active = active_list;
    mp.perm = perm;
    mp.xrow = xrow;
    mp.kdiv = kdiv;
    mp.out = out;
    mp.bias = bias;
    mp.group = pl.group;
    mp.ids = ids;
    mp.n_pairs = n_pairs;
    mp.n_expert = n_expert;
    mp.self_group = self_group ? 1 : 0;
    // Grid rows map onto the experts that received pairs (at most this many).
    // When every expert takes one group of pairs (decode) the work per expert
    // is even and one wave of CTAs covers it; otherwise two waves of smaller
    // shares balance experts with more pairs.
    const int active = n_pairs < n_expert ? n_pairs : n_expert;
    const int g = pl.group;
    const int waves = cap <= g ? 1 : 2;
    if constexpr (!plain_rt(T)) {
        if (a8) {
            if (g <= 1) return launch_moe_nv<T, true, 1>(mp, pl, active, active, waves, st);
            if (g <= 2) return launch_moe_nv<T, true, 2>(mp, pl, active, active, waves, st);
            if (g <= 4) return launch_moe_nv<T, true, 4>(mp, pl, active, active, waves, st);
            if (g <= 8) return launch_moe_nv<T, true, 8>(mp, pl, active, active, waves, st);
            return launch_moe_nv<T, true, 16>(mp, pl, active, active, waves, st);
        }
    }
    if (g <= 1) return launch_moe_nv<T, false, 1>(mp, pl, active, active, waves, st);
    if (g <= 2) return launch_moe_nv<T, false, 2>(mp, pl, active, active, waves, st);
    if (g <= 4) return launch_moe_nv<T, false, 4>(mp, pl, active, active, waves, st);
    if (g <= 8) return launch_moe_nv<T, false, 8>(mp, pl, active, active, waves, st);
    return launch_moe_nv<T, false, 16>(mp, pl, active, active, waves, st);
}

}  // namespace qmv

#define QMV_MOE_INSTANTIATE(T, NAME)                                                                        \
    int NAME(bool a8, bool quant_x, const void* W3d, int n_expert, int64_t rows, int64_t cols,                 \
             const int* offsets, const int* active, const int* perm, const int32_t* ids, bool self_group,      \
             int n_pairs, int n_tok, const void* x, size_t xrow, int kdiv, float* out, const float* bias,       \
             cudaStream_t st)                                                                                   \
    {                                                                                                           \
        return qmv::launch_moe_t<T>(a8, quant_x, W3d, n_expert, rows, cols, offsets, active, perm, ids,        \
                                    self_group, n_pairs, n_tok, x, xrow, kdiv, out, bias, st);                  \
    }

#define QMV_GEMV_INSTANTIATE(T, NAME)                                                                     \
    int NAME(bool a8, bool quant_x, bool pdl, const void* W, int64_t rows, int64_t cols, const void* x,   \
             float* y, int n_vec, cudaStream_t st)                                                         \
    {                                                                                                      \
        return qmv::launch_gemv_t<T>(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st);                    \
    }
