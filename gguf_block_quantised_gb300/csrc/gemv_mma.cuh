// gemv_mma.cuh -- the W4A8 decode matvec on the int8 tensor path.
//
// Same producer warp, stage ring and staged activations as the dp4a engine in
// gemv.cuh; the consumers differ.  The eight consumer warps form (8/wk) row
// groups x wk K-splits: a row group owns 16 weight rows, a K-split a
// contiguous share of each K-chunk's blocks.  Per 32-element block (16 for
// Q6_K sub-blocks) one mma.sync per 8 vectors gives the exact int32 block
// dots of 16 rows; the scales enter per block (per super-block for the
// K-quants, whose sub-block scales are first applied in integers).
//
// Reduction order of output (r, v): its K-split partial sums its blocks in
// increasing order with fp32 fused multiply-adds; the wk partials are added in
// K-split order.  wk depends only on the matrix shape, never on the number of
// vectors, so decode is bit-identical whatever n_vec is.
#pragma once

#include "gemv.cuh"
#include "mma_units.cuh"

namespace qmv {

// One row group / K-split's share of one stage: blocks [b0, b1) of rows
// 16*rg .. 16*rg+15 (slot pointers s0 = row g, s1 = row g+8 of that group).
template <int T, int NT>
__device__ __forceinline__ void mma_rows(const GemvParams& p, const XView& X, const uint8_t* s0, const uint8_t* s1,
                                         int c0, int b0, int b1, float (&acc)[NT][4])
{
    using F = Fmt<T>;
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    if constexpr (F::BS == 32) {
        for (int b = b0; b < b1; ++b) {
            const int bo = (b - c0) * F::BB;
            uint32_t a[4];
            float dw0, dw1;
            MmaA32<T>::load(s0 + bo, s1 + bo, q, a, dw0, dw1);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int vb = 8 * t + g;   // this lane's B column
                uint32_t bb0 = 0, bb1 = 0;
                if (vb < p.nv) {
                    const uint8_t* xc = X.codes + (size_t)vb * X.cols + (size_t)b * 32 + 4 * q;
                    bb0 = *reinterpret_cast<const uint32_t*>(xc);
                    bb1 = *reinterpret_cast<const uint32_t*>(xc + 16);
                }
                int d[4] = {0, 0, 0, 0};
                mma_k32(d, a, bb0, bb1);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = 8 * t + 2 * q + (e & 1);
                    if (v < p.nv) {
                        const int isum = d[e] - MmaA32<T>::OFF * X.sum32[v * X.nb + b];
                        acc[t][e] = __fmaf_rn((float)isum, (e < 2 ? dw0 : dw1) * X.d[v * X.nb + b], acc[t][e]);
                    }
                }
            }
        }
    } else if constexpr (T == QMV_Q4_K) {
        for (int b = b0; b < b1; ++b) {
            const int bo = (b - c0) * F::BB;
            const uint4 h0 = *reinterpret_cast<const uint4*>(s0 + bo);
            const uint4 h1 = *reinterpret_cast<const uint4*>(s1 + bo);
            const Q4kScales k0 = q4k_scales(h0.y, h0.z, h0.w), k1 = q4k_scales(h1.y, h1.z, h1.w);
            int S[NT][4], Mn[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[t][e] = Mn[t][e] = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint8_t* q0 = s0 + bo + 16 + 32 * c + 4 * q;
                const uint8_t* q1 = s1 + bo + 16 + 32 * c + 4 * q;
                const uint32_t w0l = *reinterpret_cast<const uint32_t*>(q0);
                const uint32_t w0h = *reinterpret_cast<const uint32_t*>(q0 + 16);
                const uint32_t w1l = *reinterpret_cast<const uint32_t*>(q1);
                const uint32_t w1h = *reinterpret_cast<const uint32_t*>(q1 + 16);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int j = 2 * c + half, sh = 4 * half;
                    const uint32_t a[4] = {(w0l >> sh) & 0x0f0f0f0fu, (w1l >> sh) & 0x0f0f0f0fu,
                                           (w0h >> sh) & 0x0f0f0f0fu, (w1h >> sh) & 0x0f0f0f0fu};
                    const int sc0 = k0.sc(j), sc1 = k1.sc(j), m0 = k0.m(j), m1 = k1.m(j);
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const int vb = 8 * t + g;
                        uint32_t bb0 = 0, bb1 = 0;
                        if (vb < p.nv) {
                            const uint8_t* xc = X.codes + (size_t)vb * X.cols + (size_t)b * 256 + 32 * j + 4 * q;
                            bb0 = *reinterpret_cast<const uint32_t*>(xc);
                            bb1 = *reinterpret_cast<const uint32_t*>(xc + 16);
                        }
                        int d[4] = {0, 0, 0, 0};
                        mma_k32(d, a, bb0, bb1);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int v = 8 * t + 2 * q + (e & 1);
                            if (v < p.nv) {
                                const int16_t* bs = X.bsum + ((size_t)v * X.nb + b) * 16 + 2 * j;
                                S[t][e] += (e < 2 ? sc0 : sc1) * d[e];
                                Mn[t][e] += (e < 2 ? m0 : m1) * ((int)bs[0] + (int)bs[1]);
                            }
                        }
                    }
                }
            }
            const float dd0 = half_bits_to_float(h0.x & 0xffffu), dm0 = half_bits_to_float(h0.x >> 16);
            const float dd1 = half_bits_to_float(h1.x & 0xffffu), dm1 = half_bits_to_float(h1.x >> 16);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = 8 * t + 2 * q + (e & 1);
                    if (v < p.nv) {
                        const float dx = X.d[v * X.nb + b];
                        acc[t][e] = __fmaf_rn((float)S[t][e], (e < 2 ? dd0 : dd1) * dx, acc[t][e]);
                        acc[t][e] = __fmaf_rn(-(float)Mn[t][e], (e < 2 ? dm0 : dm1) * dx, acc[t][e]);
                    }
                }
        }
    } else {   // Q6_K: sixteen 16-element sub-blocks, element 16s + i
        for (int b = b0; b < b1; ++b) {
            const int bo = (b - c0) * F::BB;
            int S[NT][4];
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[t][e] = 0;
            const uint32_t scw0[4] = {ld_word(s0 + bo + 192), ld_word(s0 + bo + 196), ld_word(s0 + bo + 200),
                                      ld_word(s0 + bo + 204)};
            const uint32_t scw1[4] = {ld_word(s1 + bo + 192), ld_word(s1 + bo + 196), ld_word(s1 + bo + 200),
                                      ld_word(s1 + bo + 204)};
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const int h = s >> 3, gp = (s & 7) >> 1, lh = s & 1;
                const int lo = 64 * h + 32 * (gp & 1) + 16 * lh + 4 * q;
                const int ho = 128 + 32 * h + 16 * lh + 4 * q;
                const int nsh = 4 * (gp >> 1), hsh = 2 * gp;
                const uint32_t a0 = ((ld_word(s0 + bo + lo) >> nsh) & 0x0f0f0f0fu) |
                                    (((ld_word(s0 + bo + ho) >> hsh) & 0x03030303u) << 4);
                const uint32_t a1 = ((ld_word(s1 + bo + lo) >> nsh) & 0x0f0f0f0fu) |
                                    (((ld_word(s1 + bo + ho) >> hsh) & 0x03030303u) << 4);
                const int sc0 = (int)(int8_t)((scw0[s >> 2] >> (8 * (s & 3))) & 0xffu);
                const int sc1 = (int)(int8_t)((scw1[s >> 2] >> (8 * (s & 3))) & 0xffu);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int vb = 8 * t + g;
                    uint32_t bb0 = 0;
                    if (vb < p.nv) bb0 = *reinterpret_cast<const uint32_t*>(X.codes + (size_t)vb * X.cols +
                                                                            (size_t)b * 256 + 16 * s + 4 * q);
                    int d[4] = {0, 0, 0, 0};
                    mma_k16(d, a0, a1, bb0);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int v = 8 * t + 2 * q + (e & 1);
                        if (v < p.nv) {
                            const int isum = d[e] - 32 * (int)X.bsum[((size_t)v * X.nb + b) * 16 + s];
                            S[t][e] += (e < 2 ? sc0 : sc1) * isum;
                        }
                    }
                }
            }
            const float dd0 = half_bits_to_float(ld_u16(s0 + bo + 208)), dd1 = half_bits_to_float(ld_u16(s1 + bo + 208));
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = 8 * t + 2 * q + (e & 1);
                    if (v < p.nv)
                        acc[t][e] = __fmaf_rn((float)S[t][e], (e < 2 ? dd0 : dd1) * X.d[v * X.nb + b], acc[t][e]);
                }
        }
    }
}

template <int T, int NT>
__global__ void __launch_bounds__(kGemvThreads, 1) k_gemv_mma(const GemvParams p)
{
    using F = Fmt<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    float* red = reinterpret_cast<float*>(smem + 256);              // [8 warps][16 rows][16 cols]
    uint8_t* xs = smem + 256 + 8 * 16 * 16 * 4;
    uint8_t* stage0 = xs + ((p.xhat_bytes + 127) & ~127u);
    const int wk = p.wk;                 // K-splits per row group
    const int tr = 16 * (kConsumerWarps / wk);
    const uint32_t stage_bytes = p.stage_bytes;

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
    if (producer) {
        int64_t tile = blockIdx.x;
        int chunk = 0;
        for (int it = 0; it < S && it < n_items; ++it) {
            gemv_produce<F::BB, true>(p, tile, chunk, stage0 + (size_t)it * stage_bytes, &full[it], tr);
            if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
        }
    }
    pdl_wait();
    {
        const size_t xrow = p.quant_x ? (size_t)p.cols * 4 : (size_t)p.nb * (F::BS == 32 ? 34 : 292);
        stage_xhat_a8_natural<T>(xs, p.quant_x != 0, p.x, xrow, p.nv, p.cols, tid, kGemvThreads);
        __syncthreads();
    }
    if (producer) {
        int64_t tile = blockIdx.x + (int64_t)(S / p.n_chunks) * gridDim.x;
        int chunk = S % p.n_chunks;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        int it = S;
        for (; it < n_items; ++it) {
            ok = mbar_wait_bounded(&empty[s], ph, p.status);
            if (!ok) break;
            gemv_produce<F::BB, true>(p, tile, chunk, stage0 + (size_t)s * stage_bytes, &full[s], tr);
            if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
            if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok && lane == 0)
            for (int j = max(0, it - S); j < it; ++j)
                mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1), p.status, 100000000ull);
        return;
    }

    const XView X = carve_xview<T>(xs, true, p.nv, p.cols);
    const int rg = warp / wk, kw = warp % wk, g = lane >> 2, q = lane & 3;
    // A timed-out wait makes the warp skip the rest, but it keeps meeting the
    // consumers' named barrier so that no other warp waits on it forever.
    bool dead = false;
    float acc[NT][4];
    int64_t tile = blockIdx.x;
    int chunk = 0, s = 0;
    uint32_t ph = 0;
    for (int it = 0; it < n_items; ++it) {
        if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], ph, p.status));
        const int c0 = chunk * p.kb;
        const int c1 = min(p.nb, c0 + p.kb);
        const int64_t r0 = tile * tr + 16 * rg;
        if (chunk == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
        }
        if (!dead && r0 < p.rows) {
            const uint8_t* buf = stage0 + (size_t)s * stage_bytes;
            const uint8_t* slot0;
            const uint8_t* slot1;
            if (p.contig) {
                const uint8_t* t0 = buf + (((uint32_t)(tile * tr) * (uint32_t)p.rb) & 15u);
                slot0 = t0 + (size_t)(16 * rg + g) * p.rb;
                slot1 = t0 + (size_t)(16 * rg + g + 8) * p.rb;
            } else {
                const uint32_t base_off = (uint32_t)c0 * (uint32_t)F::BB;
                slot0 = buf + (size_t)(16 * rg + g) * p.seg_cap + (((uint32_t)(r0 + g) * (uint32_t)p.rb + base_off) & 15u);
                slot1 = buf + (size_t)(16 * rg + g + 8) * p.seg_cap +
                        (((uint32_t)(r0 + g + 8) * (uint32_t)p.rb + base_off) & 15u);
            }
            const int n = c1 - c0;
            const int b0 = c0 + (n * kw) / wk, b1 = c0 + (n * (kw + 1)) / wk;
            mma_rows<T, NT>(p, X, slot0, slot1, c0, b0, b1, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (chunk == p.n_chunks - 1) {
            // Combine the K-split partials of each output in K-split order.
            if (wk > 1) {
                float* mine = red + (size_t)warp * 256;
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        mine[(g + 8 * (e >> 1)) * 16 + 8 * t + 2 * q + (e & 1)] = acc[t][e];
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
            }
            if (kw == 0 && !dead) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = g + 8 * (e >> 1), v = 8 * t + 2 * q + (e & 1);
                        float sum = acc[t][e];
                        for (int k2 = 1; k2 < wk; ++k2) sum += red[(size_t)(warp + k2) * 256 + row * 16 + 8 * t + 2 * q + (e & 1)];
                        if (v < p.nv && r0 + row < p.rows) p.y[(int64_t)v * p.rows + r0 + row] = sum;
                    }
            }
            if (wk > 1) asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        }
        if (++chunk == p.n_chunks) { chunk = 0; tile += gridDim.x; }
        if (++s == S) { s = 0; ph ^= 1u; }
    }
}

}  // namespace qmv
