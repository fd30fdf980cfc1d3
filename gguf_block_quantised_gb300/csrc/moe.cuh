// moe.cuh -- mixture-of-experts matvec over a stacked 3-D expert tensor.
//
// "Models and formats" page, "Architectures": a router picks k of n experts
// per token and the experts are stored as stacked 3-D tensors; gpt-oss puts a
// bias on every expert projection.  The (token, slot) pairs are grouped by
// expert beforehand (k_moe_group, a stable counting sort), so each expert's
// rows stream through shared memory once per group of up to 16 of its pairs,
// with those pairs' activations gathered into the staged vectors.  The
// arithmetic per output is exactly the decode matvec's (same units, same
// fixed reduction order), so an expert's output for a pair does not depend on
// which other pairs were routed with it.
#pragma once

#include "gemv.cuh"

namespace qmv {

struct MoeParams {
    GemvParams g;            // geometry of one expert's matrix; g.W = expert 0
    int64_t expert_bytes;    // rows * rb
    const int* offsets;      // [n_expert + 1] pair ranges per expert
    const int* active;       // [0] = number of experts with pairs, [1..] their ids (grid row y -> active[1 + y])
    const int* perm;         // pair indices (t*k + s) grouped by expert, stable
    size_t xrow;             // bytes between activation rows
    int kdiv;                // activation row of pair p = p / kdiv (k: shared per token, 1: per slot)
    float* out;              // output row of pair p at out + p*rows
    const float* bias;       // [n_expert][rows] added to every output (NULL: none)
    int group;               // pairs staged at once (<= the kernel's NV, <= 16)
    // self-grouping (at most 32 pairs, decode): offsets/active/perm are unused;
    // each CTA sorts the pairs' expert ids itself
    const int32_t* ids;      // [n_pairs] expert of each pair
    int n_pairs, n_expert, self_group;
};

// The grouping of at most 32 pairs by one warp: the experts that received
// pairs, in id order, and for the y-th of them its pairs in pair order (the
// stable counting sort of k_moe_group, restricted to one expert).  Ids out of
// range set the status word and their pairs are left out.
struct SmallGroup {
    int n_active, e, cnt;
    int perm[32];
};

__device__ __forceinline__ void small_group(const MoeParams& mp, int y, SmallGroup& g)
{
    const int lane = threadIdx.x & 31;
    const int e = lane < mp.n_pairs ? mp.ids[lane] : -1;
    const bool valid = e >= 0 && e < mp.n_expert;
    if (lane < mp.n_pairs && !valid) atomicOr(mp.g.status, QMV_DEV_BAD_EXPERT);
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
    const uint32_t same = __match_any_sync(0xffffffffu, valid ? e : -1) & vmask;
    const bool first = valid && (__ffs(same) - 1) == lane;   // first pair of its expert
    const uint32_t firsts = __ballot_sync(0xffffffffu, first);
    // rank of this lane's expert among the distinct experts, by id
    int rank = 0;
    for (uint32_t f = firsts; f; f &= f - 1) {
        const int q = __ffs(f) - 1;
        const int eq = __shfl_sync(0xffffffffu, e, q);
        rank += (valid && eq < e) ? 1 : 0;
    }
    const uint32_t mine = __ballot_sync(0xffffffffu, first && rank == y);
    if (lane == 0) {
        g.n_active = __popc(firsts);
        g.e = -1;
        g.cnt = 0;
    }
    __syncwarp();
    if (mine) {
        const int leader = __ffs(mine) - 1;
        const uint32_t pairs = __shfl_sync(0xffffffffu, same, leader);
        if (lane == leader) {
            g.e = e;
            g.cnt = __popc(pairs);
        }
        if ((pairs >> lane) & 1u) g.perm[__popc(pairs & ((1u << lane) - 1u))] = lane;
    }
}

template <int T, bool A8, int NV, int RIF>
__global__ void __launch_bounds__(kGemvThreads, two_ctas_per_sm<T, A8, NV>() ? 2 : 1) k_moe_gemv(const MoeParams mp)
{
    using F = Fmt<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    // bytes 0..259 hold the barriers, pair_of, xrow_of and the abort flag (below);
    // the self-grouping result sits in the free bytes before the staged vectors at 512
    SmallGroup& sg = *reinterpret_cast<SmallGroup*>(smem + 320);
    static_assert(320 + sizeof(SmallGroup) <= 512, "self-grouping scratch");
    pdl_wait();   // the grouping (or the ids) comes from the kernel before this one
    if (mp.self_group) {
        if (threadIdx.x < 32) small_group(mp, (int)blockIdx.y, sg);
        __syncthreads();
    }
    if ((int)blockIdx.y >= (mp.self_group ? sg.n_active : mp.active[0])) return;   // uniform for the whole block
    const int e = mp.self_group ? sg.e : mp.active[1 + blockIdx.y];
    const int o0 = mp.self_group ? 0 : mp.offsets[e];
    const int cnt = mp.self_group ? sg.cnt : mp.offsets[e + 1] - o0;
    GemvParams p = mp.g;
    const int tr = kConsumerWarps * p.rpw;
    const int64_t n_tiles = (p.rows + tr - 1) / tr;
    if (cnt <= 0 || blockIdx.x >= n_tiles) return;   // uniform for the whole block
    p.W = mp.g.W + (size_t)e * mp.expert_bytes;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    int* pair_of = reinterpret_cast<int*>(empty + kMaxStages);   // [16] (smem bytes 128..319)
    int* xrow_of = pair_of + 16;                                  // [16]
    volatile int* abort_flag = xrow_of + 16;
    uint8_t* xs = smem + 512;
    uint8_t* stage0 = xs + ((p.xhat_bytes + 127) & ~127u);
    const uint32_t stage_bytes = p.seg_cap * (uint32_t)(kConsumerWarps * p.rpw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int my_tiles = (int)((n_tiles - 1 - blockIdx.x) / gridDim.x) + 1;
    const int G = mp.group;   // <= NV
    const int n_groups = (cnt + G - 1) / G;
    const int per_group = my_tiles * p.n_chunks;
    const int n_items = n_groups * per_group;
    const int S = p.stages;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // A timed-out wait sets abort_flag; every later wait then fails at once, and
    // the consumers keep meeting at their named barriers until the loop ends,
    // so no warp is left waiting on one that gave up.
    auto wait_or_abort = [&](uint64_t* bar, uint32_t parity) {
        if (*abort_flag) return false;
        if (mbar_wait_bounded(bar, parity, p.status, p.wait_ns)) return true;
        *abort_flag = 1;
        return false;
    };

    if (warp == kConsumerWarps) {
        // Producer: the expert's row tiles, once per group of pairs.
        int64_t tile = blockIdx.x;
        int chunk = 0, in_group = 0;
        bool ok = true;
        int it = 0;
        for (; it < n_items; ++it) {
            const int s = it % S;
            if (it >= S) {
                ok = wait_or_abort(&empty[s], (uint32_t)(((it / S) - 1) & 1));
                if (!ok) break;
            }
            gemv_produce<F::BB>(p, tile, chunk, stage0 + (size_t)s * stage_bytes, &full[s]);
            if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
            if (++in_group == per_group) { in_group = 0; chunk = 0; tile = blockIdx.x; }
        }
        // Let the copies still in flight land (bounded) before the block can
        // leave: the last S issued items, each its stage's latest phase.
        if (lane == 0)
            for (int j = max(0, it - S); j < it; ++j)
                mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), p.status, 100000000ull);
        (void)ok;
        return;
    }

    // Consumers (8 warps, named barrier 1).
    auto cbar = [] { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); };
    float acc[RIF][NV];
    int s = 0;
    uint32_t ph = 0;
    for (int grp = 0; grp < n_groups; ++grp) {
        const int gv = min(G, cnt - grp * G);
        cbar();   // everyone is done with the previous group's activations
        if (tid < gv) {
            const int pr = mp.self_group ? sg.perm[grp * G + tid] : mp.perm[o0 + grp * G + tid];
            pair_of[tid] = pr;
            xrow_of[tid] = pr / mp.kdiv;
        }
        cbar();
        stage_xhat<T>(xs, A8, p.quant_x != 0, p.x, mp.xrow, xrow_of, gv, p.cols, tid, kConsumerWarps * 32);
        cbar();
        if (!A8) {
            stage_xsum32<T>(xs, gv, p.cols, tid, kConsumerWarps * 32);
            cbar();
        }
        p.nv = gv;
        const XView X = carve_xview<T>(xs, A8, gv, p.cols);
        int64_t tile = blockIdx.x;
        int chunk = 0;
        for (int it = 0; it < per_group; ++it) {
            if (!__all_sync(0xffffffffu, wait_or_abort(&full[s], ph))) {
                if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
                if (++s == S) { s = 0; ph ^= 1u; }
                continue;
            }
            const uint8_t* buf = stage0 + (size_t)s * stage_bytes;
            const int c0 = chunk * p.kb;
            const int c1 = min(p.nb, c0 + p.kb);
            for (int g = 0; g < p.rpw; g += RIF) {
                const int64_t r0 = tile * tr + (int64_t)warp * p.rpw + g;
                const int nrows = (int)min((int64_t)min(RIF, p.rpw - g), p.rows - r0);
                if (nrows <= 0) break;
                if (chunk == 0) {
#pragma unroll
                    for (int j = 0; j < RIF; ++j)
#pragma unroll
                        for (int v = 0; v < NV; ++v) acc[j][v] = 0.f;
                }
                gemv_rows<T, A8, NV, RIF>(p, X, buf + (size_t)(warp * p.rpw + g) * p.seg_cap, r0, nrows, c0, c1,
                                          acc);
                if (chunk == p.n_chunks - 1) {
                    const int row = RIF == 4 ? (lane >> 3) : (RIF == 2 ? (lane >> 4) : 0);
                    const bool writer = (lane & (32 / RIF - 1)) == 0;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        if (v < gv) {
                            float col[RIF];
#pragma unroll
                            for (int j = 0; j < RIF; ++j) col[j] = acc[j][v];
                            const float sum = warp_sum_rows<RIF>(col);
                            if (writer && row < nrows) {
                                const int64_t r = r0 + row;
                                float out = sum;
                                if (mp.bias) out += mp.bias[(int64_t)e * p.rows + r];
                                mp.out[(int64_t)pair_of[v] * p.rows + r] = out;
                            }
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
}

}  // namespace qmv
