// gemm_deq.cu -- prefill GEMM for the block formats other than Q4_K, with the
// weights dequantised tile by tile into TMEM (tcgen05, sm_103a).
//
// "Architecture" page, "The package map": pkg/tensor MatMul is the prefill
// multiply; "The two phases": prefill is bound by arithmetic.  The pages' own
// prefill workload mixes Q5_0, Q8_0, Q6_K and Q4_K matrices.  Y[m][r] =
// sum_k X[m][k] * bf16(w[r][k]) with w the block's fp32 value (the matvec
// kernels' unit decoders), rounded once to bf16, and bf16 activations,
// accumulating in fp32.  The layout of the kernel is the Q4_K GEMM's
// (gemm_q4k.cu); what differs is the raw weight stream:
//
//   warp 0      TMA producer of activation tiles X[BN tokens][64 k] (bf16,
//               128-byte swizzle)
//   warp 1      TMEM owner and the single-thread MMA issuer (A from TMEM)
//   warp 2      raw weight producer: the 18/22/34/210-byte blocks are rarely
//               16-byte aligned, but with rows of a whole number of 16 bytes
//               a raw stage's bytes start at the same offset in every row, so
//               one TMA box (UINT8 tensor map, 128 rows x up to 256 bytes from
//               that offset rounded down to 16) carries the whole stage
//   warps 4-11  dequantisers: thread t decodes row t % 128, half t / 128 of
//               each 128-k A stage (two 32-element blocks, or one 64-element
//               K-quant unit) and stores the bf16 pairs into TMEM (lane = row,
//               column = k / 2)
//   warps 12-19 epilogue: TMEM -> registers -> Y
// A raw stage is 128 k of the 32-element formats (4 blocks per row) or one
// 256-k super-block (two A stages).  Rows whose byte length is not a multiple
// of 16 are not taken here (the caller converts them in two passes).  Blocks past the end of a row (cols not a
// multiple of 128) decode as zeros.  Rows much shorter than K run as 2 or 4 K
// parts on the CTAs of a thread-block cluster, whose partial tiles are summed
// in part order through distributed shared memory.  Every mbarrier wait is
// bounded; on a timeout the kernel flags the status word, unwinds and frees
// its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "dequant_unit.cuh"
#include "runtime.cuh"
#include "tc.cuh"

namespace qmv {

bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch, uint32_t box_in, uint32_t box_out, CUtensorMapSwizzle sw);

namespace gd {
constexpr int BM = 128, BK = 64, KSUB = 2, SK = 2;
constexpr int X_BYTES_MAX = 256 * BK * 2;   // 32768 per 64-k sub-chunk (BN = 256)
constexpr int OFF_R = SK * KSUB * X_BYTES_MAX;
constexpr int DEQ_WARPS = 8, EPI_WARP0 = 12, EPI_WARPS = 8;
constexpr int THREADS = 640;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_STAGE_COLS = KSUB * BK / 2;   // 64 columns = 128 bf16 k per row
}  // namespace gd

template <int T>
struct DeqCfg {
    using F = Fmt<T>;
    static constexpr int RK = F::BS == 256 ? 256 : 128;   // k per raw stage
    static constexpr int AST = RK / 128;                  // A stages per raw stage
    static constexpr int BPR = RK / F::BS;                // blocks per row per raw stage
    static constexpr int RBYTES = BPR * F::BB;
    // One TMA box per raw stage: the rows' bytes from the stage's first block
    // rounded down to 16 (the same offset in every row, since rows are whole
    // multiples of 16 bytes), an odd number of 16-byte units wide so that eight
    // consecutive rows' 16-byte loads hit distinct banks; 64 bytes of slack
    // after the box take the window loads' over-read, and each stage starts on
    // a 128-byte boundary (the TMA destination's alignment).
    static constexpr int BOXW0 = (RBYTES + 15 + 15) / 16 * 16;
    static constexpr int BOXW = (BOXW0 / 16) % 2 ? BOXW0 : BOXW0 + 16;
    static_assert(BOXW <= 256, "TMA box width");
    static constexpr int PITCH = BOXW;
    static constexpr int R_BYTES = (gd::BM * PITCH + 64 + 127) / 128 * 128;
    static constexpr int SR = gd::OFF_R + 3 * R_BYTES + 2048 <= 227 * 1024 ? 3 : 2;   // raw stages
    static constexpr int OFF_BAR = gd::OFF_R + SR * R_BYTES;
    static constexpr int N_BARS = 2 * gd::SK + 2 * SR + 4;
    static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(gd::OFF_R % 128 == 0 && R_BYTES % 128 == 0, "TMA destination alignment");
};

struct GemmDeqArgs {
    int64_t rows;
    int nb;               // blocks per row
    int cols;             // K
    int m;                // tokens
    float* Y;             // [m][rows]
    unsigned* status;
    int ks;               // K parts: 1, 2 (adding into a zeroed Y) or 4 (a cluster, one tile per CTA)
    int cluster;          // 1: the K parts are the CTAs of a cluster, reduced through its shared memory
    int nrs_all;          // raw stages of a whole row
};

// NC 16-byte chunks of shared memory from p (16-byte aligned) as 4*NC words;
// eight consecutive rows' loads hit distinct banks (odd row pitch in chunks).
template <int NC>
__device__ __forceinline__ void ld_chunks(const uint8_t* p, uint32_t (&u)[4 * NC + 1])
{
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[c];
        u[4 * c] = v.x; u[4 * c + 1] = v.y; u[4 * c + 2] = v.z; u[4 * c + 3] = v.w;
    }
    u[4 * NC] = 0u;
}

// Bytes 4k..4k+3 after byte S (compile-time, < 16) of the loaded chunks.
template <int S>
__device__ __forceinline__ uint32_t word_at(const uint32_t* u, int k)
{
    if constexpr (S % 4 == 0) return u[S / 4 + k];
    else return __funnelshift_r(u[S / 4 + k], u[S / 4 + k + 1], 8 * (S % 4));
}

// The 32-element block (Q4_0 / Q5_0 / Q8_0) at byte O (compile-time) of the
// 16-byte-aligned row -> its 32 weights as 16 bf16x2 words in k order:
// w = d*(q - OFF) as one fused multiply-add of the unsigned code (exact: d has
// 11 significant bits and q at most 8), rounded to bf16.  Codes become floats
// through 0x4B0000qq = 2^23 + q (dq2_bf16).
template <int T, int O>
__device__ __forceinline__ void decode_block32(const uint8_t* row, uint32_t (&o)[16])
{
    using F = Fmt<T>;
    constexpr int S = O % 16, NC = (S + F::BB + 3 + 15) / 16;
    uint32_t u[4 * NC + 1];
    ld_chunks<NC>(row + 16 * (O / 16), u);
    const uint32_t x0 = word_at<S>(u, 0);
    const float d = half_bits_to_float(x0 & 0xffffu);
    uint32_t c[8];   // code bytes of elements 4i..4i+3, unsigned
    if constexpr (T == QMV_Q8_0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            c[i] = __funnelshift_r(word_at<S>(u, i), word_at<S>(u, i + 1), 16) ^ 0x80808080u;   // q + 128
    } else {
        uint32_t n[4], qh = 0;
        constexpr int N0 = T == QMV_Q5_0 ? 1 : 0;   // Q5_0: fp16 d | u32 fifth bits | nibbles
        if constexpr (T == QMV_Q5_0) qh = __funnelshift_r(x0, word_at<S>(u, 1), 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) n[i] = __funnelshift_r(word_at<S>(u, N0 + i), word_at<S>(u, N0 + i + 1), 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c[i] = n[i] & 0x0f0f0f0fu;              // elements 4i..4i+3: low nibbles
            c[4 + i] = (n[i] >> 4) & 0x0f0f0f0fu;   // elements 16+4i..: high nibbles
            if constexpr (T == QMV_Q5_0) {
                // bit e of qh is bit 4 of element e's code
                c[i] |= ((((qh >> (4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
                c[4 + i] |= ((((qh >> (16 + 4 * i)) & 15u) * 0x00204081u) & 0x01010101u) << 4;
            }
        }
    }
    constexpr float OFF = T == QMV_Q8_0 ? 128.f : (float)F::OFF;
    const uint64_t D2 = pk2(d, d), nM2 = pk2(-OFF * d, -OFF * d);   // OFF*d exact
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        o[2 * i] = dq2_bf16(c[i], 0x76517650u, D2, nM2);
        o[2 * i + 1] = dq2_bf16(c[i], 0x76537652u, D2, nM2);
    }
}

// Half h (compile-time) of a 32-element-format A stage: blocks 2h, 2h+1 of the
// stage's four, whose bytes start at byte OFF of the row; k = 64h + 32jj + e.
template <int T, int OFF, int B>
__device__ __forceinline__ void decode_block32_st(const uint8_t* row, int nblk, uint32_t taddr)
{
    uint32_t o[16];
    if (B < nblk) {
        decode_block32<T, OFF + B * Fmt<T>::BB>(row, o);
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = 0u;
    }
    tmem_st16_async(taddr + 16 * B, o);
}

template <int T, int OFF, int H>
__device__ __forceinline__ void decode_half32(const uint8_t* row, int nblk, uint32_t taddr)
{
    decode_block32_st<T, OFF, 2 * H>(row, nblk, taddr);
    decode_block32_st<T, OFF, 2 * H + 1>(row, nblk, taddr);
}

// Q6_K unit (half AS of the super-block, lh = h) whose block starts at byte OFF
// of the row: group g's 16 elements at k = 32g + 16h + e of the A stage, code =
// 4 low bits from ql, 2 high bits from qh; w = d*sc*(q - 32) with d*sc exact,
// one rounding.
template <int OFF, int AS>
__device__ __forceinline__ void decode_q6k(const uint8_t* row, int h, uint32_t taddr)
{
    uint32_t u0[9], u1[9], uh[9], us[9], ud[9];
    // ql[64AS + 16h ..], ql[64AS + 32 + 16h ..], qh[32AS + 16h ..]: 16 bytes each
    ld_chunks<2>(row + 16 * (4 * AS + h), u0);
    ld_chunks<2>(row + 16 * (4 * AS + 2 + h), u1);
    ld_chunks<2>(row + 16 * (8 + 2 * AS + h), uh);
    constexpr int SO = OFF + 192 + 8 * AS;   // this half's 8 scales
    ld_chunks<2>(row + 16 * (SO / 16), us);
    ld_chunks<2>(row + 16 * ((OFF + 208) / 16), ud);
    uint32_t L0[4], L1[4], H[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        L0[k] = word_at<OFF>(u0, k);
        L1[k] = word_at<OFF>(u1, k);
        H[k] = word_at<OFF>(uh, k);
    }
    const uint32_t S[2] = {word_at<SO % 16>(us, 0), word_at<SO % 16>(us, 1)};
    const float d = half_bits_to_float(word_at<(OFF + 208) % 16>(ud, 0) & 0xffffu);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int sc = (int)(int8_t)((S[g >> 1] >> (16 * (g & 1) + 8 * h)) & 0xffu);   // scales[8AS + 2g + h]
        const float D = d * (float)sc;                                                   // exact
        const uint64_t D2 = pk2(D, D), nM2 = pk2(-32.f * D, -32.f * D);
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t c;
            if (g == 0) c = (L0[k] & 0x0f0f0f0fu) | ((H[k] & 0x03030303u) << 4);
            else if (g == 1) c = (L1[k] & 0x0f0f0f0fu) | ((H[k] & 0x0c0c0c0cu) << 2);
            else if (g == 2) c = ((L0[k] >> 4) & 0x0f0f0f0fu) | (H[k] & 0x30303030u);
            else c = ((L1[k] >> 4) & 0x0f0f0f0fu) | ((H[k] & 0xc0c0c0c0u) >> 2);
            o[2 * k] = dq2_bf16(c, 0x76517650u, D2, nM2);
            o[2 * k + 1] = dq2_bf16(c, 0x76537652u, D2, nM2);
        }
        tmem_st8_async(taddr + 16 * g + 8 * h, o);
    }
}

// Decode this thread's half (h, warp-uniform) of A stage AS of a raw stage
// into TMEM columns taddr.. (row = the thread's TMEM lane, column = k / 2 of
// the stage).  row: the row's 16-byte-aligned bytes in the raw tile, whose
// first block starts at byte off (the same in every row); nblk: the raw
// stage's blocks in the row.  The offsets become compile-time constants: off
// is 0 or 8 for the 32-element formats (4 blocks of 18, 22 or 34 bytes per
// stage) and even for Q6_K's 210-byte super-blocks.
template <int T, int AS>
__device__ __forceinline__ void decode_stage(const uint8_t* row, int off, int h, int nblk, uint32_t taddr)
{
    if constexpr (Fmt<T>::BS == 32) {
        if (off == 0) {
            if (h == 0) decode_half32<T, 0, 0>(row, nblk, taddr);
            else decode_half32<T, 0, 1>(row, nblk, taddr);
        } else {
            if (h == 0) decode_half32<T, 8, 0>(row, nblk, taddr);
            else decode_half32<T, 8, 1>(row, nblk, taddr);
        }
    } else {
        switch (off) {
        case 0: decode_q6k<0, AS>(row, h, taddr); break;
        case 2: decode_q6k<2, AS>(row, h, taddr); break;
        case 4: decode_q6k<4, AS>(row, h, taddr); break;
        case 6: decode_q6k<6, AS>(row, h, taddr); break;
        case 8: decode_q6k<8, AS>(row, h, taddr); break;
        case 10: decode_q6k<10, AS>(row, h, taddr); break;
        case 12: decode_q6k<12, AS>(row, h, taddr); break;
        default: decode_q6k<14, AS>(row, h, taddr); break;
        }
    }
}

template <int T, int BN>
__global__ void __launch_bounds__(gd::THREADS, 1)
    k_gemm_deq_bf16(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const GemmDeqArgs a)
{
    using namespace gd;
    using C = DeqCfg<T>;
    using F = Fmt<T>;
    constexpr int SR = C::SR;
    constexpr int X_BYTES = BN * BK * 2;
    // TMEM: NBUF accumulators of BN columns from column 0, then the A stages
    constexpr int NBUF = BN == 256 ? 1 : 2;
    constexpr uint32_t A_COL = NBUF * BN;
    static_assert(A_COL + SK * A_STAGE_COLS <= TMEM_COLS, "TMEM budget");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    // k stage s: X tiles (shared memory) and A tile (TMEM) of 128 k; full[s]
    // completes when the X bytes have landed and the eight dequantising warps
    // have stored A, empty[s] when the MMAs reading both are done.  Raw stage
    // sr: rf[sr] when its bytes have landed, re[sr] when the dequantisers are
    // done with it.
    uint64_t* full = bars;
    uint64_t* empty = full + SK;
    uint64_t* rf = empty + SK;
    uint64_t* re = rf + SR;
    uint64_t* accf = re + SR;
    uint64_t* acce = accf + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_rt = (int)((a.rows + BM - 1) / BM);
    const int n_nt = (a.m + BN - 1) / BN;
    const int n_tiles = n_rt * n_nt * a.ks;
    // work item t: tile t / ks, K part t % ks (with a cluster: the CTA's rank in
    // it, the grid one item per CTA); part p takes raw stages
    // [p * nrs_all / ks, (p + 1) * nrs_all / ks)
    auto rs_begin = [&](int part) { return part * a.nrs_all / a.ks; };

    if (tid == 0) {
        for (int i = 0; i < SK; ++i) { mbar_init(&full[i], DEQ_WARPS + 1); mbar_init(&empty[i], 1); }
        for (int i = 0; i < SR; ++i) { mbar_init(&rf[i], 1); mbar_init(&re[i], DEQ_WARPS); }
        for (int i = 0; i < 2; ++i) { mbar_init(&accf[i], 1); mbar_init(&acce[i], EPI_WARPS); }
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();
    pdl_wait();

    auto fail = [&]() { *abort_flag = 1; };

    if (warp == 0) {
        // ---- activation tiles
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                const int nt = (t / a.ks) % n_nt, part = t % a.ks;
                const int k0 = rs_begin(part) * C::AST, nks = (rs_begin(part + 1) - rs_begin(part)) * C::AST;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_backoff(&empty[s], ph, a.status, 64)) { fail(); break; }
                    mbar_arrive_expect_tx(&full[s], KSUB * X_BYTES);
#pragma unroll
                    for (int j = 0; j < KSUB; ++j)
                        tma_load_2d(smem + (s * KSUB + j) * X_BYTES, &tmX, ((k0 + ks) * KSUB + j) * BK, nt * BN,
                                    &full[s]);
                    if (++s == SK) { s = 0; ph ^= 1; }
                }
            }
        }
    } else if (warp == 2) {
        // ---- raw weight tiles: one box of 128 rows x BOXW bytes per raw stage
        if (lane == 0) {
            int sr = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                const int rt = t / a.ks / n_nt, part = t % a.ks;
                bool bad = false;
                for (int rs = rs_begin(part); rs < rs_begin(part + 1); ++rs) {
                    const int kb = rs * C::BPR;
                    if (!mbar_wait_backoff(&re[sr], ph, a.status, 64)) { bad = true; break; }
                    mbar_arrive_expect_tx(&rf[sr], BM * C::BOXW);
                    tma_load_2d(smem + OFF_R + sr * C::R_BYTES, &tmW, (kb * F::BB) & ~15, rt * BM, &rf[sr]);
                    if (++sr == SR) { sr = 0; ph ^= 1; }
                }
                if (bad) { fail(); break; }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN);
            int s = 0;
            uint32_t pf = 0;
            int local = 0;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++local) {
                const int buf = local % NBUF;
                const uint32_t use = (uint32_t)(local / NBUF);
                if (!mbar_wait_bounded(&acce[buf], (use & 1) ^ 1, a.status)) { fail(); break; }
                tc_fence_after();
                const uint32_t d = tmem + buf * BN;
                const int part = t % a.ks, nks = (rs_begin(part + 1) - rs_begin(part)) * C::AST;
                bool bad = false;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_bounded(&full[s], pf, a.status)) { bad = true; break; }
                    tc_fence_after();
                    const uint32_t at = tmem + A_COL + s * A_STAGE_COLS;
#pragma unroll
                    for (int j = 0; j < KSUB; ++j) {
                        const uint64_t bdesc = smem_desc_sw128(smem + (s * KSUB + j) * X_BYTES);
#pragma unroll
                        for (int k4 = 0; k4 < BK / 16; ++k4)   // A: 8 TMEM columns, B: 32 bytes per K = 16 step
                            mma_f16_ts(d, at + 32 * j + 8 * k4, bdesc + 2 * k4, idesc, (ks | j | k4) != 0);
                    }
                    mma_commit(&empty[s]);
                    if (++s == SK) { s = 0; pf ^= 1; }
                }
                if (bad) { fail(); break; }
                mma_commit(&accf[buf]);
            }
        }
    } else if (warp >= 4 && warp < EPI_WARP0) {
        // ---- dequantisers: thread t -> TMEM lane (row) t % 128 (warp % 4 is the
        // warp's lane quarter), half t / 128 of each A stage
        const int t0 = tid - 128, row = t0 & 127, h = t0 >> 7;
        const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + A_COL;
        int sr = 0, s = 0;
        uint32_t prf = 0, pe = 1;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x) {
            const int part = t % a.ks;
            bool bad = false;
            for (int rs = rs_begin(part); rs < rs_begin(part + 1) && !bad; ++rs) {
                const int kb = rs * C::BPR;
                const int nblk = min(C::BPR, a.nb - kb);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&rf[sr], prf, a.status))) { bad = true; break; }
                // rows past the end of the matrix read the box's zero fill, never stored
                const uint8_t* rowp = smem + OFF_R + sr * C::R_BYTES + row * C::PITCH;
                const int off = (kb * F::BB) & 15;
#pragma unroll
                for (int as = 0; as < C::AST; ++as) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], pe, a.status))) { bad = true; break; }
                    tc_fence_after();
                    if (as == 0) decode_stage<T, 0>(rowp, off, h, nblk, ta + s * A_STAGE_COLS);
                    else decode_stage<T, 1>(rowp, off, h, nblk, ta + s * A_STAGE_COLS);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[s]);
                    if (++s == SK) { s = 0; pe ^= 1; }
                }
                if (bad) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&re[sr]);
                if (++sr == SR) { sr = 0; prf ^= 1; }
            }
            if (bad) { fail(); break; }
        }
    } else if (warp >= EPI_WARP0) {
        // ---- epilogue: lane quarter (warp % 4), column half (warp - 12) / 4
        const int q = warp & 3, ch = (warp - EPI_WARP0) >> 2;
        int local = 0;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x, ++local) {
            const int rt = t / a.ks / n_nt, nt = (t / a.ks) % n_nt;
            const int buf = local % NBUF;
            const uint32_t use = (uint32_t)(local / NBUF);
            // warp-uniform: every lane must take part in the tcgen05.ld below
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&accf[buf], use & 1, a.status))) { fail(); break; }
            tc_fence_after();
            if (a.cluster) break;   // a K part: reduced through the cluster below
            const int64_t row = (int64_t)rt * BM + 32 * q + lane;
            const bool row_ok = row < a.rows;
            const int c0 = ch * BN / 2, nr = BN / 64;
            for (int rd = 0; rd < nr; ++rd) {
                uint32_t v0[16], v1[16];
                const uint32_t tc = tmem + ((uint32_t)(32 * q) << 16) + buf * BN + c0 + rd * 32;
                tmem_ld16_async(tc, v0);
                tmem_ld16_async(tc + 16, v1);
                tmem_wait_ld();
                if (rd == nr - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acce[buf]);
                }
                const int tok0 = nt * BN + c0 + rd * 32;
                if (a.ks == 1) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (row_ok && tok0 + i < a.m) a.Y[(int64_t)(tok0 + i) * a.rows + row] = __uint_as_float(v0[i]);
                        if (row_ok && tok0 + 16 + i < a.m)
                            a.Y[(int64_t)(tok0 + 16 + i) * a.rows + row] = __uint_as_float(v1[i]);
                    }
                } else {
                    // two parts add into the zeroed Y (0 + p0 + p1 = 0 + p1 + p0)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (row_ok && tok0 + i < a.m)
                            atomicAdd(a.Y + (int64_t)(tok0 + i) * a.rows + row, __uint_as_float(v0[i]));
                        if (row_ok && tok0 + 16 + i < a.m)
                            atomicAdd(a.Y + (int64_t)(tok0 + 16 + i) * a.rows + row, __uint_as_float(v1[i]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (a.cluster) {
        // K parts of one tile, one per CTA of the cluster: each lane quarter of
        // the tile (32 rows) has an owner CTA (quarter q -> rank q * ks / 4),
        // which gathers the ks partial sums of its quarters in its X stage area
        // as [quarter][part][column][row] fp32 and adds them in part order:
        // ((p0 + p1) + p2) + p3, the same bits whichever part finishes first.
        // The first cluster barrier orders every CTA's last MMA before the
        // others' stores into its X area; the second, the stores before the sums.
        cluster_sync();
        const int t = blockIdx.x, part = t % a.ks;
        const int rt = t / a.ks / n_nt, nt = (t / a.ks) % n_nt;
        const int qpr = 4 / a.ks;   // lane quarters per owner
        float* red = reinterpret_cast<float*>(smem);
        if (warp >= EPI_WARP0) {
            const int q = warp & 3, ch = (warp - EPI_WARP0) >> 2;
            const uint32_t owner = (uint32_t)(q / qpr), qo = (uint32_t)(q % qpr);
            tc_fence_after();
            const int c0 = ch * BN / 2, nr = BN / 64;
            for (int rd = 0; rd < nr; ++rd) {
                uint32_t v0[16], v1[16];
                const uint32_t tc = tmem + ((uint32_t)(32 * q) << 16) + c0 + rd * 32;
                tmem_ld16_async(tc, v0);
                tmem_ld16_async(tc + 16, v1);
                tmem_wait_ld();
                const int col0 = c0 + rd * 32;
                float* dst = red + ((size_t)(qo * a.ks + part) * BN + col0) * 32 + lane;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    dsmem_st_u32(dsmem_addr(dst + 32 * i, owner), v0[i]);
                    dsmem_st_u32(dsmem_addr(dst + 32 * (16 + i), owner), v1[i]);
                }
            }
        }
        cluster_sync();
        if (warp >= EPI_WARP0) {
            const int rank = part;
            for (int idx = warp - EPI_WARP0; idx < qpr * BN; idx += EPI_WARPS) {
                const int qo = idx / BN, col = idx % BN;
                const int64_t row = (int64_t)rt * BM + 32 * (rank * qpr + qo) + lane;
                const int tok = nt * BN + col;
                const float* src = red + ((size_t)(qo * a.ks) * BN + col) * 32 + lane;
                float sum = src[0];
                for (int p = 1; p < a.ks; ++p) sum += src[(size_t)p * BN * 32];
                if (row < a.rows && tok < a.m) a.Y[(int64_t)tok * a.rows + row] = sum;
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int T>
static int launch_gemm_deq_t(const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m, bool pdl,
                             cudaStream_t st)
{
    using F = Fmt<T>;
    using C = DeqCfg<T>;
    GemmDeqArgs a;
    a.rows = rows;
    a.nb = (int)(cols / F::BS);
    const uint64_t row_bytes = (uint64_t)a.nb * F::BB;
    if (row_bytes % 16) return -3;   // the tensor map needs 16-byte row pitches
    a.cols = (int)cols;
    a.m = (int)m;
    a.Y = Y;
    a.status = status_word();
    // rows much shorter than K: two K halves on different SMs (a whole number
    // of raw stages each), as in the Q4_K GEMM; the split follows the shape
    a.nrs_all = (a.nb + C::BPR - 1) / C::BPR;
    const int64_t n_rt = (rows + gd::BM - 1) / gd::BM;
    // Rows much shorter than K run as K parts; the split follows the weight's
    // shape alone, so a token's summation order does not depend on m.  Few row
    // tiles (four parts stay within half of the SMs) and at least 16 raw stages:
    // four parts on the CTAs of a cluster, one tile each, summed in part order
    // through its shared memory.  Else cols >= 8192 and >= 2 rows: two parts on
    // the persistent grid adding into a zeroed Y (a cluster of two, one tile per
    // CTA, measured slower there: 4096 x 14336 at 2048 tokens 0.208 -> 0.259 ms).
    a.ks = 1;
    a.cluster = 0;
    if (cols >= 2048 && n_rt * 4 <= (int64_t)num_sms() / 2 && a.nrs_all >= 16) {
        a.ks = 4;
        a.cluster = 1;
    } else if (cols >= 8192 && cols >= 2 * rows && a.nrs_all % 2 == 0) {
        a.ks = 2;
    }
    // 256-token tiles unless they cannot give half of the SMs a work item (a
    // tile's cost is mostly dequantising its weight rows: partly empty 256-token
    // tiles beat twice as many 128-token ones)
    const bool narrow = n_rt * ((m + 255) / 256) * a.ks < (int64_t)num_sms() / (a.ks == 1 ? 1 : 2);
    const int BN = narrow ? 128 : 256;
    CUtensorMap tmX, tmW;
    if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)cols, (uint64_t)m, (uint64_t)cols * 2,
                      gd::BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return -8;
    if (!make_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, (uint64_t)rows, row_bytes, C::BOXW, gd::BM,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return -8;
    auto* k = narrow ? &k_gemm_deq_bf16<T, 128> : &k_gemm_deq_bf16<T, 256>;
    prepare_kernel(k, gd::THREADS, C::SMEM);
    const int64_t n_items = n_rt * ((m + BN - 1) / BN) * a.ks;
    if (n_items > INT32_MAX) return -6;
    if (a.ks == 2) {
        // the parts add into Y: zero it first (in stream order, so no programmatic overlap)
        if (cudaMemsetAsync(Y, 0, (size_t)m * (size_t)rows * sizeof(float), st) != cudaSuccess) return -6;
        pdl = false;
    }
    // persistent over the work items, or (a cluster per tile) one item per CTA
    const int grid = a.cluster ? (int)n_items : (int)std::min<int64_t>(n_items, num_sms());
    return launch_ex_cluster(k, dim3(grid), dim3(gd::THREADS), C::SMEM, st, pdl, a.cluster ? a.ks : 1, tmX, tmW, a) ==
                   cudaSuccess
               ? 0
               : -6;
}

}  // namespace qmv

// Block types with a fused tile dequantiser here: Q4_0, Q5_0, Q8_0, Q6_K (Q4_K
// has its own kernel), with rows of a whole number of 16 bytes.  Returns 0, -3
// (type or row length not taken), -6 (launch failure) or -8 (tensor map).
int qmv_launch_gemm_deq_bf16(int t, const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                             bool pdl, cudaStream_t st)
{
    using namespace qmv;
    if (rows == 0 || m == 0) return 0;
    switch (t) {
    case QMV_Q4_0: return launch_gemm_deq_t<QMV_Q4_0>(W, rows, cols, X, Y, m, pdl, st);
    case QMV_Q5_0: return launch_gemm_deq_t<QMV_Q5_0>(W, rows, cols, X, Y, m, pdl, st);
    case QMV_Q8_0: return launch_gemm_deq_t<QMV_Q8_0>(W, rows, cols, X, Y, m, pdl, st);
    case QMV_Q6_K: return launch_gemm_deq_t<QMV_Q6_K>(W, rows, cols, X, Y, m, pdl, st);
    default: return -3;
    }
}
