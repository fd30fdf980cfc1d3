// gemm_bf16.cu -- prefill GEMM for plain weight rows: Y[m][r] = sum_k X[m][k] *
// bf16(w[r][k]) on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// "Architecture" page, "The package map": pkg/tensor MatMul is the prefill
// multiply; "The two phases": prefill is bound by arithmetic.  BF16 weight rows
// are the GEMM's A operand as they are.  F32 and F16 rows, and the block
// formats without a tile dequantiser inside a GEMM (Q4_1, Q5_1, Q8_1, MXFP4,
// Q2_K, Q3_K, Q5_K, and Q4_0 / Q5_0 / Q8_0 / Q6_K rows whose byte length is not
// a multiple of 16), are first converted to bf16 (w's fp32 value rounded to
// nearest even) in the workspace by a streaming pass, then multiplied.  (Q4_K
// and the other Q4_0, Q5_0, Q8_0, Q6_K rows dequantise tile by tile inside
// their GEMMs: gemm_q4k.cu, gemm_deq.cu.)
//
// One persistent CTA per SM, 12 warps:
//   warp 0      TMA producer: per stage one or two 64-k boxes of weight rows
//               W[128 rows][64 k] and as many of tokens X[BN][64 k] (bf16,
//               128-byte swizzle, the UMMA K-major canonical layout)
//   warp 1      TMEM owner (alloc/free) and the single-thread MMA issuer:
//               tcgen05.mma.cta_group::1.kind::f16, A and B from shared
//               memory, M = 128 rows, N = BN tokens, K = 16, fp32 accumulator
//   warps 4-11  epilogue: TMEM -> registers -> Y, two warps per TMEM lane
//               quarter, each half of the columns; the accumulator is released
//               as soon as its last columns are in registers.  Two accumulators
//               (all 512 TMEM columns at 256 tokens): one tile's epilogue
//               overlaps the next tile's MMAs.
// K beyond cols reads zeros (the tensor maps' out-of-bounds fill), so cols need
// only be a multiple of 8 (16-byte rows).  Every mbarrier wait is bounded; on a
// timeout the kernel flags the status word, unwinds and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "dequant_unit.cuh"
#include "runtime.cuh"
#include "tc.cuh"

namespace qmv {

bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch, uint32_t box_in, uint32_t box_out, CUtensorMapSwizzle sw);

namespace gb {
constexpr int BM = 128, BK = 64;           // BK: k of one 128-byte swizzled row = one TMA box
constexpr int A_BOX = BM * BK * 2;         // 16384
constexpr int EPI_WARP0 = 4, EPI_WARPS = 8;
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // 384
constexpr uint32_t TMEM_COLS = 512;   // two accumulators of up to 256 columns (A and B are in shared memory)
// Stages: four of 64 k at 256 tokens, three of 128 k at 128 tokens (192 KB
// either way).  A/B at 256 tokens against two 128-k stages: BF16 14336 x 4096
// x 2048 tokens 1372 -> 1545 TFLOP/s, 4096 x 14336 x 2048 1196 -> 1379; at
// 128 tokens six 64-k stages measured slower than three of 128 k (958 -> 903
// at 14336 x 4096 x 512).
template <int BN>
struct Cfg {
    static constexpr int X_BOX = BN * BK * 2;                     // 16384 / 32768
    static constexpr int KSUB = BN == 256 ? 1 : 2;                // 64-k boxes of each operand per stage
    static constexpr int STAGE = KSUB * (A_BOX + X_BOX);
    static constexpr int SK = BN == 256 ? 4 : 3;                  // stages
    static constexpr int NBUF = 2;   // accumulators: one tile's epilogue overlaps the next tile's MMAs
    static constexpr int OFF_BAR = SK * STAGE;
    static constexpr int SMEM = OFF_BAR + (2 * SK + 4) * 8 + 16 + 1024;   // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(NBUF * BN <= (int)TMEM_COLS, "TMEM budget");
};
}  // namespace gb

struct GemmBf16Args {
    int64_t rows;
    int cols;
    int m;
    float* Y;          // [m][rows]
    unsigned* status;
};

template <int BN>
__global__ void __launch_bounds__(gb::THREADS, 1)
    k_gemm_bf16(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const GemmBf16Args a)
{
    using namespace gb;
    using C = Cfg<BN>;
    constexpr int SK = C::SK, NBUF = C::NBUF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + SK;
    uint64_t* accf = empty + SK;
    uint64_t* acce = accf + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Tile t covers token tile t % n_nt of row tile t / n_nt: the CTAs running
    // at once share few weight row tiles, read from DRAM once and then from L2
    // by each of their token tiles, while the (smaller) activations stay in L2
    // for every row tile.  (Token tiles outermost streamed all the weights
    // once per token tile: 5.4 times the operands' bytes at 14336 x 4096 x
    // 2048.)
    const int n_rt = (int)((a.rows + BM - 1) / BM);
    const int n_nt = (a.m + BN - 1) / BN;
    const int n_tiles = n_rt * n_nt;
    constexpr int KSUB = C::KSUB;
    const int nks = (a.cols + KSUB * BK - 1) / (KSUB * BK);   // stages per tile

    if (tid == 0) {
        for (int i = 0; i < SK; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
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
        // ---- weight rows and token tiles, KSUB 64-k boxes of each per stage
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                const int rt = t / n_nt, nt = t % n_nt;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_backoff(&empty[s], ph, a.status, 64)) { fail(); break; }
                    uint8_t* st = smem + s * C::STAGE;
                    mbar_arrive_expect_tx(&full[s], C::STAGE);
#pragma unroll
                    for (int j = 0; j < KSUB; ++j) {
                        tma_load_2d(st + j * A_BOX, &tmW, (KSUB * ks + j) * BK, rt * BM, &full[s]);
                        tma_load_2d(st + KSUB * A_BOX + j * C::X_BOX, &tmX, (KSUB * ks + j) * BK, nt * BN, &full[s]);
                    }
                    if (++s == SK) { s = 0; ph ^= 1; }
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
                    if (!mbar_wait_bounded(&full[s], pf, a.status)) { bad = true; break; }
                    tc_fence_after();
                    const uint8_t* st = smem + s * C::STAGE;
#pragma unroll
                    for (int j = 0; j < KSUB; ++j) {
                        const uint64_t adesc = smem_desc_sw128(st + j * A_BOX);
                        const uint64_t bdesc = smem_desc_sw128(st + KSUB * A_BOX + j * C::X_BOX);
#pragma unroll
                        for (int k4 = 0; k4 < BK / 16; ++k4)   // 32 bytes per K = 16 step in both operands
                            mma_f16(d, adesc + 2 * k4, bdesc + 2 * k4, idesc, (ks | j | k4) != 0);
                    }
                    mma_commit(&empty[s]);
                    if (++s == SK) { s = 0; pf ^= 1; }
                }
                if (bad) { fail(); break; }
                mma_commit(&accf[buf]);
            }
        }
    } else if (warp >= EPI_WARP0) {
        // ---- epilogue: lane quarter warp % 4, column half (warp - 4) / 4
        const int q = warp & 3, ch = (warp - EPI_WARP0) >> 2;
        int local = 0;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x, ++local) {
            const int rt = t / n_nt, nt = t % n_nt;
            const int buf = local % NBUF;
            const uint32_t use = (uint32_t)(local / NBUF);
            // warp-uniform: every lane must take part in the tcgen05.ld below
            if (!__all_sync(0xffffffffu, mbar_wait_backoff(&accf[buf], use & 1, a.status, 256))) { fail(); break; }
            tc_fence_after();
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
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (row_ok && tok0 + i < a.m) a.Y[(int64_t)(tok0 + i) * a.rows + row] = __uint_as_float(v0[i]);
                    if (row_ok && tok0 + 16 + i < a.m)
                        a.Y[(int64_t)(tok0 + 16 + i) * a.rows + row] = __uint_as_float(v1[i]);
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

// ---------------------------------------------------------------------------
// The dequantising pass: bf16(w) tiles, w = the block's fp32 value (the same
// unit decoders as the matvec kernels), rounded to nearest even.  A stream over
// the weights: each CTA stages a chunk of 256 units' blocks (contiguous bytes,
// 16-byte loads) in shared memory, then each thread decodes one unit (32
// elements of a 32-element block, 64 of a super-block, 8 plain values) and
// writes it with 16-byte stores.  Blocks are row-major and rows have whole
// blocks, so block i's elements land at i*BS in the [rows][cols] bf16 tiles.

// Eight values -> eight bf16 (round to nearest even) in one 16-byte store.
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* p, const float* v)
{
    uint4 o;
    uint32_t* u = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        u[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = o;
}

template <int T>
__global__ void __launch_bounds__(256) k_dequant_bf16(const uint8_t* __restrict__ W, int64_t n_blocks,
                                                      __nv_bfloat16* __restrict__ out)
{
    using F = Fmt<T>;
    constexpr int NB = 256 / F::UPB;       // blocks per chunk (one unit per thread)
    constexpr int CHUNK = NB * F::BB;      // a multiple of 16 bytes for every format
    static_assert(CHUNK % 16 == 0, "chunk alignment");
    __shared__ __align__(16) uint8_t raw[CHUNK + 16];   // + the decoders' word over-read
    const int64_t b0 = (int64_t)blockIdx.x * NB;
    const int nbk = n_blocks - b0 < NB ? (int)(n_blocks - b0) : NB;
    const uint8_t* src = W + b0 * F::BB;
    const int bytes = nbk * F::BB, n16 = bytes >> 4;
    for (int i = threadIdx.x; i < n16; i += 256)
        reinterpret_cast<uint4*>(raw)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
    for (int i = 16 * n16 + threadIdx.x; i < bytes; i += 256) raw[i] = src[i];
    __syncthreads();
    pdl_trigger();   // the GEMM after this pass may start its prologue
    const int j = threadIdx.x / F::UPB, s = threadIdx.x % F::UPB;
    if (j >= nbk) return;
    float v[F::UE];
    unit_values<T>(raw + j * F::BB, s, v);
    __nv_bfloat16* o = out + (b0 + j) * F::BS;
    if constexpr (T == QMV_Q6_K) {
        const int h = s >> 1, lh = s & 1;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            store_bf16x8(o + 128 * h + 32 * g + 16 * lh, v + 16 * g);
            store_bf16x8(o + 128 * h + 32 * g + 16 * lh + 8, v + 16 * g + 8);
        }
    } else {
#pragma unroll
        for (int e = 0; e < F::UE; e += 8) store_bf16x8(o + s * F::UE + e, v + e);
    }
}

template <int T>
static int launch_dequant_bf16_t(const void* W, int64_t rows, int64_t cols, void* out, cudaStream_t st)
{
    using F = Fmt<T>;
    const int64_t n_blocks = rows * (cols / F::BS);
    if (n_blocks == 0) return 0;
    constexpr int NB = 256 / F::UPB;
    k_dequant_bf16<T><<<(unsigned)((n_blocks + NB - 1) / NB), 256, 0, st>>>(static_cast<const uint8_t*>(W), n_blocks,
                                                                            static_cast<__nv_bfloat16*>(out));
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}

static int launch_dequant_bf16(int t, const void* W, int64_t rows, int64_t cols, void* out, cudaStream_t st)
{
    switch (t) {
    case QMV_Q4_0: return launch_dequant_bf16_t<QMV_Q4_0>(W, rows, cols, out, st);
    case QMV_Q5_0: return launch_dequant_bf16_t<QMV_Q5_0>(W, rows, cols, out, st);
    case QMV_Q8_0: return launch_dequant_bf16_t<QMV_Q8_0>(W, rows, cols, out, st);
    case QMV_Q6_K: return launch_dequant_bf16_t<QMV_Q6_K>(W, rows, cols, out, st);
    case QMV_MXFP4: return launch_dequant_bf16_t<QMV_MXFP4>(W, rows, cols, out, st);
    case QMV_Q4_1: return launch_dequant_bf16_t<QMV_Q4_1>(W, rows, cols, out, st);
    case QMV_Q5_1: return launch_dequant_bf16_t<QMV_Q5_1>(W, rows, cols, out, st);
    case QMV_Q8_1: return launch_dequant_bf16_t<QMV_Q8_1>(W, rows, cols, out, st);
    case QMV_Q2_K: return launch_dequant_bf16_t<QMV_Q2_K>(W, rows, cols, out, st);
    case QMV_Q3_K: return launch_dequant_bf16_t<QMV_Q3_K>(W, rows, cols, out, st);
    case QMV_Q5_K: return launch_dequant_bf16_t<QMV_Q5_K>(W, rows, cols, out, st);
    case QMV_F32: return launch_dequant_bf16_t<QMV_F32>(W, rows, cols, out, st);
    case QMV_F16: return launch_dequant_bf16_t<QMV_F16>(W, rows, cols, out, st);
    default: return -3;
    }
}

}  // namespace qmv

// Bytes of workspace the two-pass product needs: the bf16 weight tiles.
size_t qmv_bf16_gemm_workspace_bytes(int64_t rows, int64_t cols)
{
    return ((size_t)rows * (size_t)cols * 2 + 255) & ~size_t(255);
}

namespace qmv {

// Y = X * Wb^T with Wb bf16 [rows][cols] (16-byte rows).  as_dependent: launch
// as a programmatic dependent of the kernel before it on the stream (the GEMM
// waits for it before its first copy).
static int launch_gemm_bf16(const void* Wb, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                            bool as_dependent, cudaStream_t st)
{
    CUtensorMap tmW, tmX;
    if (!make_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Wb, (uint64_t)cols, (uint64_t)rows, (uint64_t)cols * 2,
                      gb::BK, gb::BM, CU_TENSOR_MAP_SWIZZLE_128B))
        return -8;
    GemmBf16Args a;
    a.rows = rows;
    a.cols = (int)cols;
    a.m = (int)m;
    a.Y = Y;
    a.status = status_word();
    // 128- or 256-token tiles by the wave model of gemm_bf16_narrow
    const int64_t n_rt = (rows + gb::BM - 1) / gb::BM;
    const bool narrow = gemm_bf16_narrow(rows, m, num_sms());
    const int BN = narrow ? 128 : 256;
    if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)cols, (uint64_t)m, (uint64_t)cols * 2,
                      gb::BK, (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return -8;
    const int64_t n_tiles = n_rt * ((m + BN - 1) / BN);
    const int grid = (int)std::min<int64_t>(n_tiles, num_sms());
    if (narrow) {
        prepare_kernel(&k_gemm_bf16<128>, gb::THREADS, gb::Cfg<128>::SMEM);
        return launch_ex(&k_gemm_bf16<128>, dim3(grid), dim3(gb::THREADS), gb::Cfg<128>::SMEM, st, as_dependent, tmX,
                         tmW, a) == cudaSuccess
                   ? 0
                   : -6;
    }
    prepare_kernel(&k_gemm_bf16<256>, gb::THREADS, gb::Cfg<256>::SMEM);
    return launch_ex(&k_gemm_bf16<256>, dim3(grid), dim3(gb::THREADS), gb::Cfg<256>::SMEM, st, as_dependent, tmX, tmW,
                     a) == cudaSuccess
               ? 0
               : -6;
}

}  // namespace qmv

// BF16 weights multiply as they are; the other types here are first converted
// to bf16 tiles in ws (qmv_bf16_gemm_workspace_bytes).  Returns 0, -3 (type), -6
// (launch failure) or -8 (tensor map).
int qmv_launch_gemm_two_pass_bf16(int t, const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                               void* ws, bool pdl, cudaStream_t st)
{
    using namespace qmv;
    if (rows == 0 || m == 0) return 0;
    if (t == QMV_BF16) return launch_gemm_bf16(W, rows, cols, X, Y, m, pdl, st);
    const int rc = launch_dequant_bf16(t, W, rows, cols, ws, st);
    if (rc) return rc;
    return launch_gemm_bf16(ws, rows, cols, X, Y, m, true, st);
}
