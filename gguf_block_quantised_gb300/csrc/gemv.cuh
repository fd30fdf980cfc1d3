// gemv.cuh -- decode matrix-vector kernels over GGUF block rows (sm_103a).
//
// "Architecture" page, "The package map": pkg/tensor MatVec is the decode
// multiply; "The two phases": decode is bound by memory, the weights being
// read once per token ("Loading a file").  "A request, end to end": decode is
// batched so that N sequences read the weights once.
//
// Design for GB300 (one CTA = 8 warps, persistent over row tiles):
//  * A tile is 16 rows x one K-chunk.  Each row's chunk is a contiguous byte
//    range; a single thread-level TMA bulk copy (cp.async.bulk) moves each
//    16-byte-aligned superset into its own shared-memory slot, completing on
//    the stage's mbarrier.  A ring of S stages keeps many tiles in flight per
//    SM, so the HBM stream never waits on the unpacking.  GGUF blocks are
//    18/22/34/17/210 bytes and rarely 16-byte aligned; staging the aligned
//    superset and unpacking at byte granularity from shared memory keeps the
//    global traffic fully coalesced without a repacked copy of the weights.
//  * Activations are staged once per CTA in shared memory in a layout that
//    lines up with the unpacked code bytes (int8 + scales + sums for A8, fp32
//    for A32).
//  * Warp w owns rows 2w and 2w+1 of the tile; lane l owns the units
//    u = l, l+32, l+64, ... of every row it touches.  It decodes one unit of
//    both rows and reuses each vector's staged activations for the two.
//  * Reduction order per output: lane l accumulates its units in increasing
//    order with fp32 fused multiply-adds, then a fixed xor-butterfly sums the
//    32 lanes.  Nothing in that order depends on n_vec, so decode is
//    batch-invariant bit for bit.
//  * Every mbarrier wait is bounded; on timeout the CTA flags the device
//    status word, drains its own copies (bounded again) and returns.
#pragma once

#include "formats.cuh"

namespace qmv {

constexpr int kGemvThreads = 256;
constexpr int kGemvRows = 16;   // rows per tile: 8 warps x 2
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
    uint32_t seg_cap;   // bytes per row slot of a stage
    uint32_t xhat_bytes;
    unsigned* status;
};

__device__ __forceinline__ int64_t floor16(int64_t v) { return v & ~int64_t(15); }
__device__ __forceinline__ int64_t ceil16(int64_t v) { return (v + 15) & ~int64_t(15); }

// Issue the bulk copies of work item `item` (tile, chunk) into stage slot
// `buf`; called by all lanes of warp 0.  Returns nothing; lane 0 arms `bar`.
template <int BB>
__device__ __forceinline__ void gemv_issue(const GemvParams& p, int64_t tile, int chunk, uint8_t* buf,
                                           uint64_t* bar)
{
    const int lane = threadIdx.x & 31;
    const int64_t r = tile * kGemvRows + lane;
    const int64_t lim = floor16(p.total);
    uint32_t bytes = 0;
    int64_t a = 0;
    if (lane < kGemvRows && r < p.rows) {
        const int c0 = chunk * p.kb;
        const int c1 = min(p.nb, c0 + p.kb);
        const int64_t s = r * p.rb + (int64_t)c0 * BB;
        const int64_t e = r * p.rb + (int64_t)c1 * BB;
        a = floor16(s);
        const int64_t ea = min(ceil16(e), lim);
        bytes = (uint32_t)(ea - a);
    }
    uint32_t total = bytes;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    // Order earlier generic-proxy accesses of this buffer (reads, and the
    // ragged-tail stores) before the async-proxy writes that refill it.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (bytes) bulk_g2s(buf + (size_t)lane * p.seg_cap, p.W + a, bytes, bar);
}

template <int T, bool A8, int NV>
__global__ void __launch_bounds__(kGemvThreads, 2) k_gemv(const GemvParams p)
{
    using F = Fmt<T>;
    using O = Ops<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint8_t* xs = smem + 128;
    uint8_t* stage0 = xs + ((p.xhat_bytes + 127) & ~127u);
    const uint32_t stage_bytes = p.seg_cap * kGemvRows;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_tiles = (p.rows + kGemvRows - 1) / kGemvRows;
    const int64_t my_tiles = (blockIdx.x < n_tiles) ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t n_items = my_tiles * p.n_chunks;
    const int S = p.stages;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        for (int s = 0; s < S && s < n_items; ++s)
            gemv_issue<F::BB>(p, blockIdx.x + (int64_t)(s / p.n_chunks) * gridDim.x, s % p.n_chunks,
                              stage0 + (size_t)s * stage_bytes, &full[s]);
    }
    stage_xhat<T>(xs, A8, p.x, p.nv, p.cols);   // overlaps the first copies; ends with a barrier
    const XView X = carve_xview<T>(xs, A8, p.nv, p.cols);

    float accA[NV], accB[NV];
    for (int64_t it = 0; it < n_items; ++it) {
        const int s = (int)(it % S);
        const uint32_t parity = (uint32_t)((it / S) & 1);
        const int64_t tile = blockIdx.x + (it / p.n_chunks) * gridDim.x;
        const int chunk = (int)(it % p.n_chunks);
        uint8_t* buf = stage0 + (size_t)s * stage_bytes;

        const bool ok = mbar_wait_bounded(&full[s], parity, p.status);
        if (__syncthreads_or(!ok)) {
            // Drain this CTA's other copies in flight (bounded) before leaving.
            if (tid == 0)
                for (int64_t j = it + 1; j < it + S && j < n_items; ++j)
                    mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), p.status, 100000000ull);
            return;
        }
        const int64_t r0 = tile * kGemvRows;
        const int c0 = chunk * p.kb;
        const int c1 = min(p.nb, c0 + p.kb);
        // The ragged end of the matrix (fewer than 16 bytes past the last
        // 16-byte boundary) is fetched with plain loads.
        {
            const int64_t lim = floor16(p.total);
            const int64_t rl = p.rows - 1;
            if (c1 == p.nb && r0 + kGemvRows > rl && p.total > lim) {
                const int64_t s0 = rl * p.rb + (int64_t)c0 * F::BB;
                const int64_t a = floor16(s0);
                uint8_t* slot = buf + (size_t)(rl - r0) * p.seg_cap;
                for (int64_t i = lim + tid; i < p.total; i += kGemvThreads) slot[i - a] = p.W[i];
            }
            __syncthreads();
        }
        if (chunk == 0) {
#pragma unroll
            for (int v = 0; v < NV; ++v) { accA[v] = 0.f; accB[v] = 0.f; }
        }
        const int64_t rA = r0 + 2 * warp, rB = rA + 1;
        const bool vA = rA < p.rows, vB = rB < p.rows;
        if (vA) {
            const uint8_t* slotA = buf + (size_t)(2 * warp) * p.seg_cap;
            const uint8_t* slotB = slotA + p.seg_cap;
            const int offA = (int)((rA * p.rb + (int64_t)c0 * F::BB) & 15);
            const int offB = (int)((rB * p.rb + (int64_t)c0 * F::BB) & 15);
            const int u0 = c0 * F::UPB, u1 = c1 * F::UPB;
#pragma unroll 1
            for (int u = u0 + lane; u < u1; u += 32) {
                const int b = u / F::UPB, sub = u % F::UPB;
                const int bo = (b - c0) * F::BB;
                typename F::W wA, wB;
                F::load(slotA + offA + bo, sub, wA);
                if (vB) F::load(slotB + offB + bo, sub, wB);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    if (v < p.nv) {
                        if constexpr (A8) {
                            typename F::XA8 xu;
                            F::load_x_a8(X, v, b, sub, xu);
                            O::acc_a8(wA, xu, accA[v]);
                            if (vB) O::acc_a8(wB, xu, accB[v]);
                        } else {
                            O::acc_a32(wA, X, v, b, sub, accA[v]);
                            if (vB) O::acc_a32(wB, X, v, b, sub, accB[v]);
                        }
                    }
                }
            }
            if (chunk == p.n_chunks - 1) {
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    if (v < p.nv) {
                        const float sA = warp_sum(accA[v]);
                        const float sB = warp_sum(accB[v]);
                        if (lane == 0) {
                            p.y[(int64_t)v * p.rows + rA] = sA;
                            if (vB) p.y[(int64_t)v * p.rows + rB] = sB;
                        }
                    }
                }
            }
        }
        __syncthreads();   // every warp is done with stage s
        const int64_t nxt = it + S;
        if (warp == 0 && nxt < n_items)
            gemv_issue<F::BB>(p, blockIdx.x + (nxt / p.n_chunks) * gridDim.x, (int)(nxt % p.n_chunks), buf,
                              &full[s]);
    }
}

// ---- host side -------------------------------------------------------------------
struct GemvPlan {
    int kb, n_chunks, stages, group, grid;
    uint32_t seg_cap, xhat_bytes, smem;
};

}  // namespace qmv

// Defined in gemv_host.cu; launches one format's kernels.
int qmv_launch_gemv(int wtype, bool a8, const void* W, int64_t rows, int64_t cols, const void* x, float* y,
                    int n_vec, cudaStream_t stream);
