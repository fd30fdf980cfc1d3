// gemm_w4a8.cu -- the W4A8 prefill GEMM on the 5th-generation tensor cores
// (tcgen05, sm_103a): Q4_K weights against Q8_K activations, exact integer
// block dots.
//
// "Architecture" page, "The package map": pkg/quant carries the fused W4A8
// kernels (4-bit weights, 8-bit activations); "The two phases": prefill is
// bound by arithmetic, so it belongs on the tensor cores.  Per 256-element
// super-block b of weight row r and token t
//   y[t][r] += d_x[t,b] * (d[r,b] * S - dmin[r,b] * Mn),
//   S  = sum_i sc_j(i) * q_i * xq_i          (sc 6-bit, q 4-bit, xq int8)
//   Mn = sum_{g<16} m_{g/2} * bsum_g          (m 6-bit, bsum = sum of 16 xq)
// sm_103a has no tcgen05 integer kind, but every factor above is an integer
// that fp16 holds exactly: sc*q <= 945, |xq| <= 127, m <= 63, |bsum| <= 2032
// (fp16 is exact for integers up to 2048).  So S and Mn come out of
// tcgen05.mma.kind::f16 with fp16 A and B and an fp32 accumulator: every
// product is exact and every partial sum an integer below 2^24 (|Mn| <= 2.1M
// always; |S| <= 30.7M in the worst case, exact in practice, and off by at
// most one unit of 2^-24 relative otherwise).
//
// Pre-pass (k_w4a8_prep): the Q8_K activations to fp16 codes Xh [m][cols],
// fp16 sums Bs [m][cols/16] and scales dxT [cols/256][m] in the workspace.
// Within each 128-element half super-block the codes are stored in the order
// in which the dequantising threads produce weights (any permutation of k
// applied to both operands leaves the sum unchanged): MMA position
// p = 64c + 8w + 2kk + e holds element 32*(2c + kk/2) + 4w + (kk&1) + 2e of
// that half (c = 32-byte code chunk, w = its 4-byte word, kk = which of four
// nibble pairs, e = pair member).
//
// Main kernel, one persistent CTA per SM, 24 warps:
//   warp 0      TMA: Xh tiles [128 tok][64 k] x 2 per 128-k stage (128-byte
//               swizzle), the Bs tile [128 tok][16] once per super-block
//               (32-byte swizzle), d_x of the tile's tokens into the scale ring
//   warp 1      TMEM owner and the single-thread MMA issuer
//   warp 2      TMA: raw Q4_K tiles [128 rows][144 B] per super-block
//   warps 4-7   dequantisers: thread = weight row = TMEM lane; sc*q as fp16
//               (one fp16 fused multiply-add per two weights on the magic
//               number 1024 + q), straight into TMEM (tcgen05.st); the mins
//               into shared memory for the Mn product; d, dmin into the ring
//   warps 8-23  epilogue: per super-block S and Mn out of TMEM, scaled and
//               accumulated in fp32 registers (4 warps per TMEM lane quarter,
//               32 tokens each); Y written once per tile
// TMEM (512 columns): S accumulators 2 x 128 (one super-block each, so one is
// drained while the next accumulates), Mn 128, A stages 2 x 64.  A 128-k stage
// (Xh, A, the mins) has one full and one empty barrier, so the MMA thread
// waits once and commits once per eight MMAs.  With 128-token tiles the MMA
// issue and the per-super-block drain handshake bound the kernel: measured
// with the arithmetic of the dequantisers and of the epilogue removed, it
// reaches ~750 TFLOP/s at 14336 x 4096, 512 tokens (the bf16 kernel's
// 256-token tiles have no room in TMEM here next to the S and Mn buffers).
// Every mbarrier wait is bounded; on a timeout the kernel flags the status
// word, unwinds and frees its TMEM.
#include <cuda.h>

#include "formats.cuh"
#include "q4k_fields.cuh"
#include "runtime.cuh"
#include "tc.cuh"

namespace qmv {

bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch, uint32_t box_in, uint32_t box_out, CUtensorMapSwizzle sw);

namespace w8 {
constexpr int BM = 128, BN = 128;
constexpr int SK = 2;                          // k stages of 128 k: Xh (+ Bs) in shared memory,
                                               // A in TMEM, the mins in shared memory
constexpr int SR = 3;                          // raw weight stages (one super-block each)
constexpr int NSC = 4;                         // scale ring slots (one super-block each)
constexpr int XH_BYTES = BN * 128 * 2;         // 32768: two 64-k boxes of 128-byte rows
constexpr int BS_BYTES = BN * 32;              // 4096: 16 fp16 per token
constexpr int X_STAGE = XH_BYTES + BS_BYTES;   // 36864 (a multiple of 1024)
constexpr int AMIN_BYTES = BM * 32;            // 4096
constexpr int R_BYTES = BM * 144;              // 18432
constexpr int SC_SLOT = 3 * 128 * 4;           // d[128], dmin[128], dx[128] fp32
constexpr int OFF_X = 0;
constexpr int OFF_AMIN = OFF_X + SK * X_STAGE;
constexpr int OFF_R = OFF_AMIN + SK * AMIN_BYTES;
constexpr int OFF_SC = OFF_R + SR * R_BYTES;
constexpr int OFF_BAR = OFF_SC + NSC * SC_SLOT;
constexpr int N_BARS = 2 * SK + 2 * SR + 2 * 2 + 1 + 2 * NSC;
constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + alignment slack
constexpr int THREADS = 768;
constexpr int DEQ_WARP0 = 4, EPI_WARP0 = 8, EPI_WARPS = 16;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_M = 256, COL_A = 384, A_COLS = 64;
static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
static_assert(X_STAGE % 1024 == 0 && OFF_AMIN % 256 == 0 && OFF_R % 16 == 0 && OFF_SC % 128 == 0,
              "swizzle atoms and TMA destinations aligned");
static_assert(COL_A + SK * A_COLS <= TMEM_COLS && COL_M + BN <= COL_A && COL_S + 2 * BN <= COL_M, "TMEM budget");
}  // namespace w8

struct W4a8Args {
    int64_t rows;
    int cols;
    int m;
    float* Y;
    unsigned* status;
};

// ---- pre-pass: Q8_K blocks -> fp16 codes (permuted per half super-block), fp16
// sums of 16, transposed scales.  One warp per block; lane l owns elements
// 8l .. 8l+7 (sub-block l/4).
__global__ void __launch_bounds__(256) k_w4a8_prep(const uint8_t* __restrict__ xq, __half* __restrict__ xh,
                                                   __half* __restrict__ bs, float* __restrict__ dxT, int64_t nblk,
                                                   int nsb, int m, int64_t dx_pitch)
{
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();
    if (blk >= nblk) return;
    const int64_t t = blk / nsb;
    const int sb = (int)(blk % nsb);
    const uint8_t* b = xq + blk * 292;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(b + 4 + 8 * lane);   // blocks are 4-byte aligned
    const uint2 q = make_uint2(qw[0], qw[1]);
    const int sub = lane >> 2, h = sub >> 2, c = (sub & 3) >> 1, hi = sub & 1;
    __half* out = xh + t * (int64_t)nsb * 256 + (int64_t)sb * 256 + 128 * h + 64 * c + 4 * hi;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const uint32_t w = g ? q.y : q.x;            // elements 4wd .. 4wd+3 of the sub-block
        const int wd = 2 * (lane & 3) + g;
        const int8_t e0 = (int8_t)(w & 0xff), e1 = (int8_t)(w >> 8), e2 = (int8_t)(w >> 16), e3 = (int8_t)(w >> 24);
        // positions 4hi + {0, 1, 2, 3} of word wd hold elements {0, 2, 1, 3}
        __half2 lo = __halves2half2(__short2half_rn(e0), __short2half_rn(e2));
        __half2 hi2 = __halves2half2(__short2half_rn(e1), __short2half_rn(e3));
        uint2 v;
        v.x = *reinterpret_cast<uint32_t*>(&lo);
        v.y = *reinterpret_cast<uint32_t*>(&hi2);
        *reinterpret_cast<uint2*>(out + 8 * wd) = v;
    }
    if (lane < 16) {
        const int16_t s = *reinterpret_cast<const int16_t*>(b + 260 + 2 * lane);
        bs[t * (int64_t)nsb * 16 + (int64_t)sb * 16 + lane] = __short2half_rn(s);
    }
    if (lane == 0) dxT[(int64_t)sb * dx_pitch + t] = *reinterpret_cast<const float*>(b);
}

// Four fp16 weights sc*q of one 4-byte word of codes (two nibble pairs of the
// low sub-block, two of the high one), as four fp16x2 words in MMA order.  The
// halves 0x6400 | q are the fp16 values 1024 + q; (1024 + q) * sc - 1024 * sc
// is sc*q <= 945, exact in one fused multiply-add.
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t sc_lo, uint32_t nc_lo, uint32_t sc_hi, uint32_t nc_hi,
                                        uint32_t (&o)[4])
{
    const uint32_t m = 0x000F000Fu, mg = 0x64006400u;
    const uint32_t p0 = (w & m) | mg, p1 = ((w >> 8) & m) | mg, p2 = ((w >> 4) & m) | mg, p3 = ((w >> 12) & m) | mg;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[0]) : "r"(p0), "r"(sc_lo), "r"(nc_lo));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[1]) : "r"(p1), "r"(sc_lo), "r"(nc_lo));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[2]) : "r"(p2), "r"(sc_hi), "r"(nc_hi));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[3]) : "r"(p3), "r"(sc_hi), "r"(nc_hi));
}

// An integer 0..63 as the fp16x2 pair (v, v), and (-1024 v, -1024 v).
__device__ __forceinline__ uint32_t h2_int(int v)
{
    const __half x = __int2half_rn(v);
    const __half2 p = __halves2half2(x, x);
    return *reinterpret_cast<const uint32_t*>(&p);
}

__global__ void __launch_bounds__(w8::THREADS, 1)
    k_gemm_q4k_w4a8(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmW,
                    const W4a8Args a)
{
    using namespace w8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    // k stage s: full[s] completes when its Xh (+ Bs) bytes have landed and the
    // four dequantising warps have written A (TMEM) and the mins; empty[s]
    // when the MMAs reading them are done (one commit per stage).
    uint64_t* full = bars;                  // [SK]
    uint64_t* empty = full + SK;            // [SK]
    uint64_t* rfull = empty + SK;           // [SR]  raw weights landed
    uint64_t* rempty = rfull + SR;          // [SR]  dequantisers done with them
    uint64_t* sfull = rempty + SR;          // [2]   S (and, for the super-block, Mn) ready
    uint64_t* sempty = sfull + 2;           // [2]   S drained
    uint64_t* mempty = sempty + 2;          // [1]   Mn drained
    uint64_t* cfull = mempty + 1;           // [NSC] scale ring slot written (d, dmin, dx)
    uint64_t* cempty = cfull + NSC;         // [NSC]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cempty + NSC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_rt = (int)((a.rows + BM - 1) / BM);
    const int n_nt = (a.m + BN - 1) / BN;
    const int n_tiles = n_rt * n_nt;
    const int nsb = a.cols / 256;

    if (tid == 0) {
        for (int i = 0; i < SK; ++i) { mbar_init(&full[i], 1 + 4); mbar_init(&empty[i], 1); }
        for (int i = 0; i < SR; ++i) { mbar_init(&rfull[i], 1); mbar_init(&rempty[i], 4); }
        for (int i = 0; i < 2; ++i) { mbar_init(&sfull[i], 1); mbar_init(&sempty[i], EPI_WARPS); }
        mbar_init(mempty, EPI_WARPS);
        for (int i = 0; i < NSC; ++i) { mbar_init(&cfull[i], 5); mbar_init(&cempty[i], EPI_WARPS); }
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmD);
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
        // ---- activations: Xh per 128-k stage, Bs per super-block, d_x per super-block
        if (lane == 0) {
            int xs = 0, cs = 0;
            uint32_t xph = 1, cph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                const int nt = t % n_nt;
                bool bad = false;
                for (int sb = 0; sb < nsb && !bad; ++sb) {
                    if (!mbar_wait_backoff(&cempty[cs], cph, a.status, 64)) { bad = true; break; }
                    mbar_arrive_expect_tx(&cfull[cs], BN * 4);
                    tma_load_2d(smem + OFF_SC + cs * SC_SLOT + 2 * 128 * 4, &tmD, nt * BN, sb, &cfull[cs]);
                    if (++cs == NSC) { cs = 0; cph ^= 1; }
                    for (int h = 0; h < 2; ++h) {
                        if (!mbar_wait_backoff(&empty[xs], xph, a.status, 64)) { bad = true; break; }
                        uint8_t* st = smem + OFF_X + xs * X_STAGE;
                        mbar_arrive_expect_tx(&full[xs], XH_BYTES + (h ? BS_BYTES : 0));
                        tma_load_2d(st, &tmX, sb * 256 + h * 128, nt * BN, &full[xs]);
                        tma_load_2d(st + XH_BYTES / 2, &tmX, sb * 256 + h * 128 + 64, nt * BN, &full[xs]);
                        if (h) tma_load_2d(st + XH_BYTES, &tmB, sb * 16, nt * BN, &full[xs]);
                        if (++xs == SK) { xs = 0; xph ^= 1; }
                    }
                }
                if (bad) { fail(); break; }
            }
        }
    } else if (warp == 2) {
        // ---- raw weight super-block tiles
        if (lane == 0) {
            int rs = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                const int rt = t / n_nt;
                bool bad = false;
                for (int sb = 0; sb < nsb; ++sb) {
                    if (!mbar_wait_backoff(&rempty[rs], ph, a.status, 64)) { bad = true; break; }
                    mbar_arrive_expect_tx(&rfull[rs], R_BYTES);
                    tma_load_2d(smem + OFF_R + rs * R_BYTES, &tmW, sb * 144, rt * BM, &rfull[rs]);
                    if (++rs == SR) { rs = 0; ph ^= 1; }
                }
                if (bad) { fail(); break; }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN, true);
            int ks = 0;
            uint32_t kph = 0, mph = 1;
            uint32_t g = 0;   // super-blocks issued so far (S buffer g % 2)
            bool bad = false;
            for (int t = blockIdx.x; t < n_tiles && !bad && !*abort_flag; t += gridDim.x) {
                for (int sb = 0; sb < nsb && !bad; ++sb, ++g) {
                    const int sbuf = (int)(g & 1);
                    if (!mbar_wait_bounded(&sempty[sbuf], ((g >> 1) & 1) ^ 1, a.status)) { bad = true; break; }
                    tc_fence_after();
                    const uint32_t dS = tmem + COL_S + 128 * sbuf;
                    for (int h = 0; h < 2; ++h) {
                        if (!mbar_wait_bounded(&full[ks], kph, a.status)) { bad = true; break; }
                        tc_fence_after();
                        const uint8_t* st = smem + OFF_X + ks * X_STAGE;
                        const uint32_t at = tmem + COL_A + A_COLS * ks;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint64_t bdesc = smem_desc_sw128(st + j * (XH_BYTES / 2));
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)   // A: 8 TMEM columns, B: 32 bytes per K = 16 step
                                mma_f16_ts(dS, at + 32 * j + 8 * k4, bdesc + 2 * k4, idesc, (h | j | k4) != 0);
                        }
                        if (h) {
                            // Mn of the super-block: mins (shared memory) x sums of 16 (the Bs tile)
                            if (!mbar_wait_bounded(mempty, mph, a.status)) { bad = true; break; }
                            mph ^= 1;
                            tc_fence_after();
                            mma_f16(tmem + COL_M, smem_desc_sw32(smem + OFF_AMIN + ks * AMIN_BYTES),
                                    smem_desc_sw32(st + XH_BYTES), idesc, false);
                        }
                        mma_commit(&empty[ks]);
                        if (++ks == SK) { ks = 0; kph ^= 1; }
                    }
                    if (bad) break;
                    mma_commit(&sfull[sbuf]);
                }
            }
            if (bad) fail();
        }
    } else if (warp >= DEQ_WARP0 && warp < EPI_WARP0) {
        // ---- dequantisers: thread r -> weight row r of the tile = TMEM lane r
        // (warp % 4 is the warp's lane quarter)
        const int r = tid - 32 * DEQ_WARP0;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        int rs = 0, as = 0, cs = 0;
        uint32_t rph = 0, aph = 1, cph = 1;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x) {
            bool bad = false;
            for (int sb = 0; sb < nsb && !bad; ++sb) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&rfull[rs], rph, a.status))) { bad = true; break; }
                const uint8_t* rp = smem + OFF_R + rs * R_BYTES + r * 144;
                const uint4 hd = *reinterpret_cast<const uint4*>(rp);
                const Q4kScales ks = q4k_scales(hd.y, hd.z, hd.w);
                // d and dmin of this row for the epilogue
                if (!__all_sync(0xffffffffu, mbar_wait_backoff(&cempty[cs], cph, a.status, 32))) { bad = true; break; }
                float* sc = reinterpret_cast<float*>(smem + OFF_SC + cs * SC_SLOT);
                sc[r] = half_bits_to_float(hd.x & 0xffffu);
                sc[128 + r] = half_bits_to_float(hd.x >> 16);
                __syncwarp();
                if (lane == 0) mbar_arrive(&cfull[cs]);
                if (++cs == NSC) { cs = 0; cph ^= 1; }
                for (int h = 0; h < 2; ++h) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[as], aph, a.status))) { bad = true; break; }
                    tc_fence_after();
                    const uint32_t ta = tmem + lane_base + COL_A + A_COLS * as;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {     // 32-byte code chunk 2h + cc: sub-blocks 4h + 2cc (+1)
                        const int jl = 4 * h + 2 * cc;
                        const uint32_t sl = h2_int(ks.sc(jl)), nl = h2_int(-1024 * ks.sc(jl));
                        const uint32_t sh = h2_int(ks.sc(jl + 1)), nh = h2_int(-1024 * ks.sc(jl + 1));
                        const uint4* qp = reinterpret_cast<const uint4*>(rp + 16 + 32 * (2 * h + cc));
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint4 qv = qp[half];
                            const uint32_t wv[4] = {qv.x, qv.y, qv.z, qv.w};
                            uint32_t o[16];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                uint32_t o4[4];
                                dq_word(wv[k], sl, nl, sh, nh, o4);
                                o[4 * k] = o4[0]; o[4 * k + 1] = o4[1]; o[4 * k + 2] = o4[2]; o[4 * k + 3] = o4[3];
                            }
                            // words 8cc + 4half .. +3 -> columns 4 * word
                            tmem_st16_async(ta + 32 * cc + 16 * half, o);
                        }
                    }
                    if (h) {
                        // the mins, m_{g/2} for g = 0..15, as this row of the Mn operand
                        // (32-byte rows, 8-row groups of 256 bytes, 32-byte swizzle)
                        uint32_t mv[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) mv[j] = h2_int(ks.m(j));
                        uint8_t* am = smem + OFF_AMIN + as * AMIN_BYTES + 256 * (r >> 3) + 32 * (r & 7);
                        const int sw = (r >> 2) & 1;
                        *reinterpret_cast<uint4*>(am + 16 * sw) = make_uint4(mv[0], mv[1], mv[2], mv[3]);
                        *reinterpret_cast<uint4*>(am + 16 * (sw ^ 1)) = make_uint4(mv[4], mv[5], mv[6], mv[7]);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[as]);
                    if (++as == SK) { as = 0; aph ^= 1; }
                }
                if (bad) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&rempty[rs]);
                if (++rs == SR) { rs = 0; rph ^= 1; }
            }
            if (bad) { fail(); break; }
        }
    } else if (warp >= EPI_WARP0) {
        // ---- epilogue: lane quarter warp % 4 (rows), token quarter (warp - 8) / 4
        const int q = warp & 3, cq = (warp - EPI_WARP0) >> 2;
        const int r = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        uint32_t g = 0;
        int cs = 0;
        uint32_t cph = 0;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x) {
            const int rt = t / n_nt, nt = t % n_nt;
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
            bool bad = false;
            for (int sb = 0; sb < nsb; ++sb, ++g) {
                const int sbuf = (int)(g & 1);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&cfull[cs], cph, a.status)) ||
                    !__all_sync(0xffffffffu, mbar_wait_bounded(&sfull[sbuf], (g >> 1) & 1, a.status))) {
                    bad = true;
                    break;
                }
                tc_fence_after();
                const float* sc = reinterpret_cast<const float*>(smem + OFF_SC + cs * SC_SLOT);
                const float dw = sc[r], dmin = sc[128 + r];
                const float4* dx4 = reinterpret_cast<const float4*>(sc + 256 + 32 * cq);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t vs[8], vm[8];
                    tmem_ld8_async(tmem + lane_base + COL_S + 128 * sbuf + 32 * cq + 8 * c8, vs);
                    tmem_ld8_async(tmem + lane_base + COL_M + 32 * cq + 8 * c8, vm);
                    tmem_wait_ld();
                    if (c8 == 3) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&sempty[sbuf]);
                            mbar_arrive(mempty);
                        }
                    }
#pragma unroll
                    for (int i4 = 0; i4 < 2; ++i4) {
                        const float4 dx = dx4[2 * c8 + i4];
                        const float dxv[4] = {dx.x, dx.y, dx.z, dx.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 4 * i4 + e;
                            const float tv = __fmaf_rn(-dmin, __uint_as_float(vm[i]), dw * __uint_as_float(vs[i]));
                            acc[8 * c8 + i] = __fmaf_rn(dxv[e], tv, acc[8 * c8 + i]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&cempty[cs]);
                if (++cs == NSC) { cs = 0; cph ^= 1; }
            }
            if (bad) { fail(); break; }
            const int64_t row = (int64_t)rt * BM + r;
            if (row < a.rows) {
                const int tok0 = nt * BN + 32 * cq;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (tok0 + i < a.m) a.Y[(int64_t)(tok0 + i) * a.rows + row] = acc[i];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace qmv

// Workspace of the W4A8 GEMM for m tokens of `cols` elements: fp16 codes, fp16
// sums of 16, transposed fp32 scales (row pitch a multiple of 16 bytes).
static size_t r256(size_t v) { return (v + 255) & ~size_t(255); }
static int64_t dx_pitch(int64_t m) { return (m + 3) & ~int64_t(3); }

size_t qmv_w4a8_workspace_bytes(int64_t cols, int64_t m)
{
    const int64_t nsb = cols / 256;
    return r256((size_t)m * cols * 2) + r256((size_t)m * nsb * 32) + r256((size_t)nsb * dx_pitch(m) * 4);
}

// Returns 0, -6 (launch failure) or -8 (tensor map could not be built).
int qmv_launch_gemm_q4k_w4a8(const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                             void* ws, bool pdl, cudaStream_t st)
{
    using namespace qmv;
    if (rows == 0 || m == 0) return 0;
    const int64_t nsb = cols / 256;
    uint8_t* w = static_cast<uint8_t*>(ws);
    __half* xh = reinterpret_cast<__half*>(w);
    __half* bs = reinterpret_cast<__half*>(w + r256((size_t)m * cols * 2));
    float* dxT = reinterpret_cast<float*>(w + r256((size_t)m * cols * 2) + r256((size_t)m * nsb * 32));
    const int64_t nblk = m * nsb;
    if (launch_ex(k_w4a8_prep, dim3((unsigned)((nblk + 7) / 8)), dim3(256), 0, st, pdl,
                  static_cast<const uint8_t*>(X), xh, bs, dxT, nblk, (int)nsb, (int)m, dx_pitch(m)) != cudaSuccess)
        return -6;

    const uint64_t rb = (uint64_t)nsb * 144;
    CUtensorMap tmW, tmX, tmB, tmD;
    if (!make_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, rb, (uint64_t)rows, rb, 144, w8::BM,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)cols, (uint64_t)m, (uint64_t)cols * 2, 64,
                      w8::BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bs, (uint64_t)nsb * 16, (uint64_t)m, (uint64_t)nsb * 32,
                      16, w8::BN, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_tmap_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dxT, (uint64_t)dx_pitch(m), (uint64_t)nsb,
                      (uint64_t)dx_pitch(m) * 4, w8::BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return -8;
    W4a8Args a;
    a.rows = rows;
    a.cols = (int)cols;
    a.m = (int)m;
    a.Y = Y;
    a.status = status_word();
    prepare_kernel(&k_gemm_q4k_w4a8, w8::THREADS, w8::SMEM);
    const int64_t n_tiles = ((rows + w8::BM - 1) / w8::BM) * ((m + w8::BN - 1) / w8::BN);
    const int grid = (int)std::min<int64_t>(n_tiles, num_sms());
    // a programmatic dependent of the pre-pass: set-up overlaps it, the
    // activation loads wait for it (griddepcontrol.wait)
    return launch_ex(k_gemm_q4k_w4a8, dim3(grid), dim3(w8::THREADS), w8::SMEM, st, true, tmX, tmB, tmD, tmW, a) ==
                   cudaSuccess
               ? 0
               : -6;
}
