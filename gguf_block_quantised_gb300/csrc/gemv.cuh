// gemv.cuh -- decode matrix-vector kernels over GGUF block rows (sm_103a).
//
// "Architecture" page, "The package map": pkg/tensor MatVec is the decode
// multiply; "The two phases": decode is bound by memory, the weights being
// read once per token ("Loading a file").  "A request, end to end": decode is
// batched so that N sequences read the weights once.
//
// Design for GB300 (persistent CTAs over row tiles; one producer warp and
// eight consumer warps per CTA):
//  * A tile is 8*rpw rows (rpw = 2 or 4 rows per consumer warp) x one K-chunk.
//    Each row's chunk is a contiguous byte range; the producer warp moves the
//    16-byte-aligned superset of each into its own shared-memory slot with one
//    TMA bulk copy (cp.async.bulk) per row, completing on the stage's "full"
//    mbarrier.  A ring of S stages keeps ~100 KB in flight per SM so the HBM
//    stream never waits on the unpacking.  GGUF blocks are 18/22/34/17/210
//    bytes and rarely 16-byte aligned; staging the aligned superset and
//    unpacking at byte granularity from shared memory keeps the global traffic
//    fully coalesced without a repacked copy of the weights.
//  * Consumers release a stage by arriving on its "empty" mbarrier; there is
//    no block-wide barrier in the steady state.
//  * Activations are staged once per CTA in shared memory in a layout that
//    lines up with the unpacked code bytes (int8 + scales + sums for A8, fp32
//    for A32).
//  * A consumer warp decodes one unit of RIF rows at once (RIF = 4 for the
//    32-element formats, 2 for the K-quants) and reuses each vector's staged
//    activations for all of them; lane l owns units u = l, l+32, l+64, ...
//  * Reduction order per output: lane l accumulates its units in increasing
//    order with fp32 fused multiply-adds, then a fixed xor-butterfly sums the
//    32 lanes.  Nothing in that order depends on n_vec, on the tile shape or
//    on which warp holds the row, so decode is batch-invariant bit for bit.
//  * Every mbarrier wait is bounded; on timeout the warp flags the device
//    status word and returns, and the producer lets its copies land (bounded)
//    before leaving.
#pragma once

#include "formats.cuh"

namespace qmv {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = 32 * (kConsumerWarps + 1);   // + one producer warp
constexpr int kMaxStages = 8;

struct GemvParams {
    const uint8_t* W;
    int64_t rows;
    int64_t rb;         // bytes per row
    int64_t total;      // rows * rb
    const void* x;      // activations of the first vector of this group
    float* y;           // outputs of the first vector of this group, y[v*rows + r]
    int cols;
    int nb;             // blocks per row
    int nv;             // vectors in this group
    int kb;             // blocks per K-chunk
    int n_chunks;
    int stages;
    int rpw;            // rows per consumer warp per tile (1, 2 or 4)
    int quant_x;        // A8 only: x is fp32, quantised while staging
    uint32_t seg_cap;   // bytes per row slot of a stage
    uint32_t xhat_bytes;
    unsigned* status;
    unsigned long long wait_ns;   // limit of the pipeline waits (QMV_WAIT_LIMIT_NS unless overridden)
};

__device__ __forceinline__ int64_t floor16(int64_t v) { return v & ~int64_t(15); }
__device__ __forceinline__ int64_t ceil16(int64_t v) { return (v + 15) & ~int64_t(15); }

// Producer warp: arm `bar` and issue the bulk copies of one work item (tile,
// chunk): lane i copies row i's chunk (its 16-byte aligned superset) into its
// slot.  The ragged end of the matrix past its last 16-byte boundary is stored
// with plain loads before the arrive, whose release orders them for the
// consumers.
template <int BB>
__device__ __forceinline__ void gemv_produce(const GemvParams& p, int64_t tile, int chunk, uint8_t* buf,
                                             uint64_t* bar)
{
    const int lane = threadIdx.x & 31;
    const int tr = kConsumerWarps * p.rpw;
    const int64_t lim = floor16(p.total);
    const int c0 = chunk * p.kb;
    const int c1 = min(p.nb, c0 + p.kb);
    uint32_t bytes = 0;
    int64_t a = 0;
    const int64_t r = tile * tr + lane;
    if (lane < tr && r < p.rows) {
        const int64_t s = r * p.rb + (int64_t)c0 * BB;
        const int64_t e = r * p.rb + (int64_t)c1 * BB;
        a = floor16(s);
        const int64_t ea = min(ceil16(e), lim);
        if (ea > a) bytes = (uint32_t)(ea - a);
        uint8_t* slot = buf + (size_t)lane * p.seg_cap;
        for (int64_t k = max(lim, a); k < e; ++k) slot[k - a] = p.W[k];   // only the matrix's last row
    }
    uint32_t total = bytes;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    // Order this buffer's earlier generic-proxy accesses (consumer reads,
    // tail stores) before the async-proxy writes that refill it.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (bytes) bulk_g2s(buf + (size_t)lane * p.seg_cap, p.W + a, bytes, bar);
}

// Consumer: rows r0 + j (j < RIF) of one warp, one K-chunk, all vectors.
template <int T, bool A8, int NV, int RIF>
__device__ __forceinline__ void gemv_rows(const GemvParams& p, const XView& X, const uint8_t* slot0, int64_t r0,
                                          int nrows, int c0, int c1, float (&acc)[RIF][NV])
{
    using F = Fmt<T>;
    using O = Ops<T>;
    const int lane = threadIdx.x & 31;
    const uint8_t* rowp[RIF];
#pragma unroll
    for (int j = 0; j < RIF; ++j)
        rowp[j] = slot0 + (size_t)j * p.seg_cap +
                  (((uint32_t)(r0 + j) * (uint32_t)p.rb + (uint32_t)c0 * (uint32_t)F::BB) & 15u);
    const int u0 = c0 * F::UPB, u1 = c1 * F::UPB;
#pragma unroll 1
    for (int u = u0 + lane; u < u1; u += 32) {
        const int b = u / F::UPB, sub = u % F::UPB;
        const int bo = (b - c0) * F::BB;
        typename F::W w[RIF];
#pragma unroll
        for (int j = 0; j < RIF; ++j)
            if (j < nrows) F::load(rowp[j] + bo, sub, w[j]);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            if (v < p.nv) {
                if constexpr (A8) {
                    typename F::XA8 xu;
                    F::load_x_a8(X, v, b, sub, xu);
#pragma unroll
                    for (int j = 0; j < RIF; ++j)
                        if (j < nrows) O::template acc_a8<(NV <= 2)>(w[j], xu, acc[j][v]);
                } else {
#pragma unroll
                    for (int j = 0; j < RIF; ++j)
                        if (j < nrows) O::acc_a32(w[j], X, v, b, sub, acc[j][v]);
                }
            }
        }
    }
}

// Sum each of RIF per-lane partials over the warp.  The result for every row
// is the value of the fixed xor-butterfly tree (16, 8, 4, 2, 1) over its 32
// partials -- the same bits a plain butterfly gives, since each level adds the
// same two operands -- but the first levels also spread the rows over the
// lanes so that fewer shuffles are needed.  Row j's total ends up in lane
// 8j (RIF = 4), 16j (RIF = 2) or 0 (RIF = 1).
template <int RIF>
__device__ __forceinline__ float warp_sum_rows(const float (&v)[RIF])
{
    const int lane = threadIdx.x & 31;
    if constexpr (RIF == 4) {
        const bool hi = lane & 16;
        const float s0 = __shfl_xor_sync(0xffffffffu, hi ? v[0] : v[2], 16);
        const float s1 = __shfl_xor_sync(0xffffffffu, hi ? v[1] : v[3], 16);
        const float a = (hi ? v[2] : v[0]) + s0;
        const float b = (hi ? v[3] : v[1]) + s1;
        const bool h8 = lane & 8;
        const float t = __shfl_xor_sync(0xffffffffu, h8 ? a : b, 8);
        float c = (h8 ? b : a) + t;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        return c;
    } else if constexpr (RIF == 2) {
        const bool hi = lane & 16;
        const float t = __shfl_xor_sync(0xffffffffu, hi ? v[0] : v[1], 16);
        float c = (hi ? v[1] : v[0]) + t;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        return c;
    } else {
        return warp_sum(v[0]);
    }
}

// Decode with 8-bit activations and one or two vectors (up to eight for the
// 32-element formats): registers for two CTAs per SM, at most 96 per thread
// since the register file is split per scheduler and two 9-warp CTAs put five
// warps on some schedulers.  (The K-quant decoders otherwise take ~165 and
// leave one 9-warp CTA per SM, too few warps to keep the weight stream in
// flight; beyond these vector counts the two-CTA bound would spill.)
template <int T, bool A8, int NV>
constexpr bool two_ctas_per_sm()
{
    return A8 && (NV <= 2 || (Fmt<T>::BS == 32 && NV <= 8));
}

template <int T, bool A8, int NV, int RIF>
__global__ void __launch_bounds__(kGemvThreads, two_ctas_per_sm<T, A8, NV>() ? 2 : 1) k_gemv(const GemvParams p)
{
    using F = Fmt<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    uint8_t* xs = smem + 256;
    uint8_t* stage0 = xs + ((p.xhat_bytes + 127) & ~127u);
    const int tr = kConsumerWarps * p.rpw;
    const uint32_t stage_bytes = p.seg_cap * (uint32_t)tr;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_tiles = (p.rows + tr - 1) / tr;
    const int my_tiles = (blockIdx.x < n_tiles) ? (int)((n_tiles - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
    const int n_items = my_tiles * p.n_chunks;
    const int S = p.stages;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_trigger();
    const bool producer = warp == kConsumerWarps;
    const size_t xrow = (A8 && !p.quant_x) ? (size_t)p.nb * (F::BS == 32 ? 34 : 292) : (size_t)p.cols * 4;
    // The activation rows into L2 first, then the weights: neither waits for
    // the grids before this one (the activations are read after the wait).
    // Otherwise the activation loads queue behind the stage ring's copies.
    if (producer) {
        prefetch_l2_lines(p.x, (size_t)p.nv * xrow, lane);
        int64_t tile = blockIdx.x;
        int chunk = 0;
        for (int it = 0; it < S && it < n_items; ++it) {
            gemv_produce<F::BB>(p, tile, chunk, stage0 + (size_t)it * stage_bytes, &full[it]);
            if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
        }
    }
    pdl_wait();
    {
        stage_xhat<T>(xs, A8, p.quant_x != 0, p.x, xrow, nullptr, p.nv, p.cols, tid, kGemvThreads);
        __syncthreads();
        if (!A8) {
            stage_xsum32<T>(xs, p.nv, p.cols, tid, kGemvThreads);
            __syncthreads();
        }
    }

    if (producer) {
        int64_t tile = blockIdx.x + (int64_t)(S / p.n_chunks) * gridDim.x;
        int chunk = S % p.n_chunks;
        int s = 0;
        uint32_t ph = 0;   // phase parity of empty[s] to wait for
        bool ok = true;
        int it = S;
        for (; it < n_items; ++it) {
            ok = mbar_wait_bounded(&empty[s], ph, p.status, p.wait_ns);
            if (!ok) break;
            gemv_produce<F::BB>(p, tile, chunk, stage0 + (size_t)s * stage_bytes, &full[s]);
            if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
            if (++s == S) { s = 0; ph ^= 1u; }
        }
        // Let the copies still in flight land (bounded) before the block can
        // leave: the last S issued items, one per stage and each its stage's
        // latest phase.  Normally they have landed already; after a consumer
        // gave up they may not have, whatever the number of items.
        const int issued = min(it, n_items);
        if (lane == 0)
            for (int j = max(0, issued - S); j < issued; ++j)
                mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), p.status, 100000000ull);
        (void)ok;
        return;
    }

    const XView X = carve_xview<T>(xs, A8, p.nv, p.cols);
    float acc[RIF][NV];
    int64_t tile = blockIdx.x;
    int chunk = 0, s = 0;
    uint32_t ph = 0;
    for (int it = 0; it < n_items; ++it) {
        if (!mbar_wait_bounded(&full[s], ph, p.status, p.wait_ns)) return;
        const uint8_t* buf = stage0 + (size_t)s * stage_bytes;
        const int c0 = chunk * p.kb;
        const int c1 = min(p.nb, c0 + p.kb);
        for (int g = 0; g < p.rpw; g += RIF) {
            const int64_t r0 = tile * tr + (int64_t)warp * p.rpw + g;
            const int nrows = (int)min((int64_t)min(RIF, p.rpw - g), p.rows - r0);
            if (nrows <= 0) break;
            // Accumulators live across K-chunks only when one group covers all of
            // the warp's rows (rpw <= RIF), which the planner guarantees whenever
            // a row spans several chunks.
            if (chunk == 0) {
#pragma unroll
                for (int j = 0; j < RIF; ++j)
#pragma unroll
                    for (int v = 0; v < NV; ++v) acc[j][v] = 0.f;
            }
            gemv_rows<T, A8, NV, RIF>(p, X, buf + (size_t)(warp * p.rpw + g) * p.seg_cap, r0, nrows, c0, c1, acc);
            if (chunk == p.n_chunks - 1) {
                const int row = RIF == 4 ? (lane >> 3) : (RIF == 2 ? (lane >> 4) : 0);
                const bool writer = (lane & (32 / RIF - 1)) == 0;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    if (v < p.nv) {
                        float col[RIF];
#pragma unroll
                        for (int j = 0; j < RIF; ++j) col[j] = acc[j][v];
                        const float sum = warp_sum_rows<RIF>(col);
                        if (writer && row < nrows) p.y[(int64_t)v * p.rows + r0 + row] = sum;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
        if (++s == S) { s = 0; ph ^= 1u; }
    }
}

// ---- host side -------------------------------------------------------------------
struct GemvPlan {
    int kb, n_chunks, stages, group, grid, rpw;
    uint32_t seg_cap, xhat_bytes, smem;
};

}  // namespace qmv

// Defined in gemv_host.cu; launches one format's kernels.
int qmv_launch_gemv(int wtype, bool a8, const void* W, int64_t rows, int64_t cols, const void* x, float* y,
                    int n_vec, cudaStream_t stream);
