// gemm_q4k.cu -- prefill GEMM with Q4_K weights on the 5th-generation tensor
// cores (tcgen05, sm_103a).
//
// "Architecture" page, "The package map": pkg/tensor MatMul is the prefill
// multiply; "The two phases": prefill is bound by arithmetic, so it runs on
// the tensor cores.  Y[m][r] = sum_k X[m][k] * bf16(w[r][k]): the Q4_K weights
// are dequantised to bf16 (w = d*sc*q - dmin*m in fp32, one rounding, then
// rounded to bf16) and multiplied with bf16 activations, accumulating in fp32.
//
// One persistent CTA per SM, 20 warps, warp-specialised:
//   warp 0      TMA producer of activation tiles X[BN tokens][64 k] (bf16,
//               128-byte swizzle, the UMMA K-major canonical layout)
//   warp 1      TMEM owner (alloc/free) and the single-thread MMA issuer
//   warp 2      TMA producer of raw Q4_K super-block tiles W[128 rows][144 B]
//   warps 4-11  dequantisers: raw super-block -> bf16 A tiles [128 rows][64 k]
//               written straight into TMEM with tcgen05.st (row = TMEM lane,
//               two k per column), packed fp32x2 arithmetic.  A never touches
//               shared memory, which leaves the shared-memory bandwidth to the
//               MMA's reads of X and to the TMA writes.
//   warps 12-19 epilogue: TMEM -> registers -> Y, one 128-byte row segment
//               per column, so every store is coalesced
// MMA: M = 128 weight rows, N = BN tokens (256, or 128 when 256-token tiles
// would leave SMs idle or pad the tokens more), K = 16 per instruction, A from
// TMEM, B from shared memory, fp32 accumulator in TMEM.  TMEM holds 256
// accumulator columns (two 128-column buffers, so that one tile's epilogue
// overlaps the next tile's MMAs, or one 256-column buffer) and two 64-column
// A stages.  X and A of a 128-k stage share one full and one empty barrier, so
// the MMA thread waits once and commits once per eight MMAs.  Every
// mbarrier wait is bounded; on a timeout the kernel flags the status word,
// unwinds and frees its TMEM.
#include <cuda.h>

#include "dequant_unit.cuh"
#include "q4k_fields.cuh"
#include "runtime.cuh"
#include "tc.cuh"

namespace qmv {

namespace gq {
constexpr int BM = 128, BK = 64;           // BK: k of one 128-byte swizzled X row = one TMA box
constexpr int KSUB = 2;                     // 64-k sub-chunks per k stage (8 MMAs per barrier round)
constexpr int SK = 2, SR = 3;               // k stages (X tiles + A tile), raw stages
constexpr int X_BYTES_MAX = 256 * BK * 2;   // 32768 per sub-chunk (BN = 256)
constexpr int R_BYTES = BM * 144;           // 18432
constexpr int OFF_X = 0;
constexpr int OFF_R = OFF_X + SK * KSUB * X_BYTES_MAX;
constexpr int OFF_BAR = OFF_R + SR * R_BYTES;
constexpr int N_BARS = 2 * SK + 2 * SR + 4;
constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + alignment slack
constexpr int DEQ_WARPS = 8;                // warps 4..11
constexpr int EPI_WARP0 = 12;               // warps 12..19
constexpr int EPI_WARPS = 8;                // two per TMEM lane quarter, each half of the columns
constexpr int THREADS = 640;                // 20 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_STAGE_COLS = KSUB * BK / 2;   // 128 bf16 k per row = 64 columns
// accumulators: two of 128 or 192 columns, or one of 256, then the A stages
}  // namespace gq

struct GemmArgs {
    int64_t rows;      // weight rows (outputs per token)
    int cols;          // K
    int m;             // tokens
    float* Y;          // [m][rows]
    unsigned* status;
    int ks;            // K parts: 1, or 2 (each part adds its fp32 sums into a zeroed Y)
};

// Dequantise this thread's part of sub-blocks 2c, 2c+1 of the raw super-block
// tile: w = RN_fp32(d*sc*q - dmin*m) (d*sc and dmin*m are exact products),
// then rounded to bf16.  256 threads: thread t handles row t % 128 and the
// 8-k groups jj = 2*(t / 128) + {0, 1} of both sub-blocks, i.e. k = 16h..16h+15
// (lo, sub-block 2c) and 32+16h..32+16h+15 (hi, sub-block 2c+1) of the 64-k
// chunk, h = t / 128: eight bf16x2 words each, in k order.
__device__ __forceinline__ void dequant_q4k_regs(const uint8_t* raw, int c, int t, uint32_t (&lo)[8],
                                                 uint32_t (&hi)[8])
{
    const int r = t & 127;
    const uint8_t* rp = raw + r * 144;
    const uint4 h = *reinterpret_cast<const uint4*>(rp);
    const uint4 qv = *reinterpret_cast<const uint4*>(rp + 16 + 32 * c + 16 * (t >> 7));
    const Q4kScales ks = q4k_scales(h.y, h.z, h.w);
    const float d = half_bits_to_float(h.x & 0xffffu), dmin = half_bits_to_float(h.x >> 16);
    const float D0 = d * (float)ks.sc(2 * c), M0 = dmin * (float)ks.m(2 * c);       // exact
    const float D1 = d * (float)ks.sc(2 * c + 1), M1 = dmin * (float)ks.m(2 * c + 1);
    const uint64_t D0x2 = pk2(D0, D0), nM0x2 = pk2(-M0, -M0), D1x2 = pk2(D1, D1), nM1x2 = pk2(-M1, -M1);
    const uint32_t q[4] = {qv.x, qv.y, qv.z, qv.w};   // codes of 16 consecutive k
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t l4 = q[k] & 0x0f0f0f0fu, h4 = (q[k] >> 4) & 0x0f0f0f0fu;
        // selectors: byte j of the codes word, then bytes 5, 6, 7 of 0x4B000000
        lo[2 * k] = dq2_bf16(l4, 0x76517650u, D0x2, nM0x2);
        lo[2 * k + 1] = dq2_bf16(l4, 0x76537652u, D0x2, nM0x2);
        hi[2 * k] = dq2_bf16(h4, 0x76517650u, D1x2, nM1x2);
        hi[2 * k + 1] = dq2_bf16(h4, 0x76537652u, D1x2, nM1x2);
    }
}

template <int BN>
__global__ void __launch_bounds__(gq::THREADS, 1)
    k_gemm_q4k_bf16(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const GemmArgs a)
{
    using namespace gq;
    constexpr int X_BYTES = BN * BK * 2;
    // TMEM: NBUF accumulators of BN columns from column 0, then the A stages.
    // 128-token tiles double-buffer the accumulator so one tile's epilogue
    // overlaps the next tile's MMAs; 256-token tiles have room for one only.
    constexpr int NBUF = BN == 256 ? 1 : 2;
    constexpr uint32_t A_COL = NBUF * BN;
    static_assert(A_COL + SK * A_STAGE_COLS <= TMEM_COLS, "TMEM budget");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    // k stage s holds the X tiles (shared memory) and the A tile (TMEM) of 128
    // k: full[s] completes when the X bytes have landed and the eight
    // dequantising warps have stored A; empty[s] when the MMAs reading both
    // are done (one commit).
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
    // work item t: output tile t / ks, K part t % ks (a whole number of
    // 256-k super-blocks each)
    const int n_tiles = n_rt * n_nt * a.ks;
    const int nks = a.cols / (KSUB * BK) / a.ks;   // k stages per item
    const int nsb = a.cols / 256 / a.ks;

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
                const int nt = (t / a.ks) % n_nt, k0 = (t % a.ks) * nks;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_backoff(&empty[s], ph, a.status, 64)) { fail(); break; }
                    mbar_arrive_expect_tx(&full[s], KSUB * X_BYTES);
#pragma unroll
                    for (int j = 0; j < KSUB; ++j)
                        tma_load_2d(smem + OFF_X + (s * KSUB + j) * X_BYTES, &tmX, ((k0 + ks) * KSUB + j) * BK,
                                    nt * BN, &full[s]);
                    if (++s == SK) { s = 0; ph ^= 1; }
                }
            }
        }
    } else if (warp == 2) {
        // ---- raw weight super-block tiles
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                const int rt = t / a.ks / n_nt, sb0 = (t % a.ks) * nsb;
                for (int sb = 0; sb < nsb; ++sb) {
                    if (!mbar_wait_bounded(&re[s], ph, a.status)) { fail(); break; }
                    mbar_arrive_expect_tx(&rf[s], R_BYTES);
                    tma_load_2d(smem + OFF_R + s * R_BYTES, &tmW, (sb0 + sb) * 144, rt * BM, &rf[s]);
                    if (++s == SR) { s = 0; ph ^= 1; }
                }
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
                bool bad = false;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_bounded(&full[s], pf, a.status)) {
                        bad = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t at = tmem + A_COL + s * A_STAGE_COLS;
#pragma unroll
                    for (int j = 0; j < KSUB; ++j) {
                        const uint64_t bdesc = smem_desc_sw128(smem + OFF_X + (s * KSUB + j) * X_BYTES);
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
        // warp's lane quarter), columns 8h.. and 16+8h.. of the A stage
        const int t0 = tid - 128;
        const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + A_COL + 8 * (t0 >> 7);
        int sr = 0, s = 0;
        uint32_t prf = 0, pe = 1;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x) {
            bool bad = false;
            for (int sb = 0; sb < nsb && !bad; ++sb) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&rf[sr], prf, a.status))) { bad = true; break; }
                const uint8_t* raw = smem + OFF_R + sr * R_BYTES;
                for (int cs = 0; cs < 4 / KSUB; ++cs) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], pe, a.status))) { bad = true; break; }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < KSUB; ++j) {
                        uint32_t lo[8], hi[8];
                        dequant_q4k_regs(raw, cs * KSUB + j, t0, lo, hi);
                        tmem_st8_async(ta + s * A_STAGE_COLS + 32 * j, lo);
                        tmem_st8_async(ta + s * A_STAGE_COLS + 32 * j + 16, hi);
                    }
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
        // ---- epilogue: lane quarter (warp % 4) of the 128 TMEM lanes, column
        // half (warp - 12) / 4 of the tile
        const int q = warp & 3, ch = (warp - EPI_WARP0) >> 2;
        int local = 0;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x, ++local) {
            const int rt = t / a.ks / n_nt, nt = (t / a.ks) % n_nt;
            const int buf = local % NBUF;
            const uint32_t use = (uint32_t)(local / NBUF);
            // warp-uniform: every lane must take part in the tcgen05.ld below
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&accf[buf], use & 1, a.status))) { fail(); break; }
            tc_fence_after();
            const int64_t row = (int64_t)rt * BM + 32 * q + lane;
            const bool row_ok = row < a.rows;
            // 32 columns per TMEM round trip; the accumulator is released as
            // soon as the last columns are in registers, before their stores
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
                    // two parts add into the zeroed Y: 0 + p0 + p1 = 0 + p1 + p0 in
                    // IEEE arithmetic, so the result does not depend on which lands first
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
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---- host --------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D tensor map: dims {inner, outer} elements, row pitch in bytes.
bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch, uint32_t box_in, uint32_t box_out, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_in, box_out};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qmv

// Returns 0, -6 (launch failure) or -8 (tensor map could not be built).
int qmv_launch_gemm_q4k_bf16(const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                             bool pdl, cudaStream_t st)
{
    using namespace qmv;
    if (rows == 0 || m == 0) return 0;
    const uint64_t rb = (uint64_t)(cols / 256) * 144;
    CUtensorMap tmW;
    if (!make_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, rb, (uint64_t)rows, rb, 144, gq::BM,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return -8;
    GemmArgs a;
    a.rows = rows;
    a.cols = (int)cols;
    a.m = (int)m;
    a.Y = Y;
    a.status = status_word();
    // Rows much shorter than K (cols >= 2 rows, cols >= 8192, whole 512-k
    // halves): the K range is split in two parts on different SMs, which
    // doubles the work items and lets 256-token tiles fill the GPU; each
    // dequantised weight then serves twice as many tokens.  The split follows
    // the weight's shape alone, so a token's summation order does not depend
    // on m.
    a.ks = (cols >= 8192 && cols >= 2 * rows && cols % 512 == 0) ? 2 : 1;
    // 256-token tiles unless they cannot give half of the SMs a work item.  A
    // tile's cost is mostly dequantising its 128 weight rows, whatever its token
    // count, so a partly empty 256-token tile beats two 128-token tiles (384
    // tokens on 14336 x 4096: 0.066 against 0.084 ms; 1100 tokens: 0.126 against
    // 0.168 ms).
    const int64_t n_rt = (rows + gq::BM - 1) / gq::BM;
    const bool narrow = n_rt * ((m + 255) / 256) * a.ks < (int64_t)num_sms() / (a.ks == 2 ? 2 : 1);
    const int BN = narrow ? 128 : 256;
    CUtensorMap tmX;
    if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)cols, (uint64_t)m, (uint64_t)cols * 2,
                      gq::BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return -8;
    auto* k = narrow ? &k_gemm_q4k_bf16<128> : &k_gemm_q4k_bf16<256>;
    prepare_kernel(k, gq::THREADS, gq::SMEM);
    const int64_t n_tiles = n_rt * ((m + BN - 1) / BN) * a.ks;
    const int grid = (int)std::min<int64_t>(n_tiles, num_sms());
    if (a.ks == 2) {
        // the parts add into Y: zero it first (in stream order, so no programmatic overlap)
        if (cudaMemsetAsync(Y, 0, (size_t)m * (size_t)rows * sizeof(float), st) != cudaSuccess) return -6;
        pdl = false;
    }
    return launch_ex(k, dim3(grid), dim3(gq::THREADS), gq::SMEM, st, pdl, tmX, tmW, a) == cudaSuccess ? 0 : -6;
}
