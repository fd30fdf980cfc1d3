// moe_gemm.cu -- grouped tensor-core GEMM for the mixture of experts with
// bf16 activations.
//
// "Models and formats" page, "Architectures": experts are stacked 3-D tensors,
// a router sends each token to k of n experts, and gpt-oss adds a bias to
// every expert projection; "Tensor formats": the experts are MXFP4.  Every
// MXFP4 weight 2^(e-127) * E2M1 is exact in bf16 (E2M1 values have at most two
// significant bits), so the bf16 tensor-core product is the plain definition
// up to the fp32 accumulation order.
//
//   k_moe_tiles   one warp: the list of (expert, token tile) slots of the
//                 experts that received pairs, from the grouping offsets.
//   k_moe_gather  the routed activation rows, packed per expert in grouped
//                 order (bf16 [n_valid][cols]) so one TMA tensor map covers
//                 every expert's token tiles.
//   k_moe_gemm_mxfp4   persistent, one CTA per SM, warp-specialised (bf16 form;
//                 the MXFP8 form's differences follow the list):
//     warp 0      TMA producer of packed token tiles X[128 tokens][128 k]
//                 (bf16, two 64-k boxes with 128-byte swizzle)
//     warp 1      TMEM owner and the single-thread MMA issuer
//     raw weight producers:
//       GGUF rows (warps 2, 3, 24-27): per weight row, the 16-byte pieces of
//                 its next 8 MXFP4 blocks (256 k) as cp.async copies (the
//                 1530-byte row pitch of the gpt-oss experts is not a legal
//                 TMA tensor stride, and one bulk copy per 136-byte row
//                 segment is bound by the copy engine's per-request cost)
//       MXFP4_R rows (warp 2, one thread): per 512-k stage of 128 rows, two
//                 128-byte-swizzled code boxes and one exponent box, as TMA
//                 tensor copies
//     warps 4-19  dequantisers, two groups of eight taking alternate 128-k
//                 stages: MXFP4 -> bf16 A tiles [128 rows][128 k] stored
//                 straight into TMEM (tcgen05.st; row = TMEM lane), through a
//                 per-block table of the eight E2M1 magnitudes already scaled
//                 by 2^(e-127).  Keeping A out of shared memory leaves the
//                 shared-memory bandwidth to the token tiles and raw blocks.
//     warps 20-23 epilogue: TMEM -> registers -> the (token, slot) output rows,
//                 plus the expert bias
//   MMA M = 128 weight rows, N = 128 tokens, K = 16, A from TMEM, B (tokens)
//   from shared memory, fp32 accumulator in TMEM, double-buffered so one
//   tile's epilogue overlaps the next tile's MMAs.  The X and A tiles of a
//   128-k stage share one full and one empty barrier: one wait and one commit
//   per eight MMAs.
//   Every mbarrier wait is bounded; on a timeout the kernel flags the status
//   word, unwinds and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include "formats.cuh"
#include "runtime.cuh"
#include "tc.cuh"

namespace qmv {

bool make_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t pitch, uint32_t box_in, uint32_t box_out, CUtensorMapSwizzle sw);

namespace mg {
constexpr int BM = 128, BN = 128, BK = 64;   // BK: k of one 128-byte swizzled X row = one TMA box
constexpr int KSUB = 2;                  // 64-k sub-chunks per k stage (8 MMAs per barrier round)
constexpr int SK = 4;                    // k stages (X tiles + A tile)
constexpr int X_BYTES = BN * BK * 2;     // 16384 per sub-chunk (bf16: 64 k; MXFP8: 128 k)
constexpr int OFF_X = 0;
constexpr int DEQ_WARPS = 16;            // warps 4..19: two groups of eight, alternate 128-k stages
constexpr int EPI_WARP0 = 20;            // warps 20..23

// Raw weight staging per layout.
// GGUF MXFP4 rows: per raw stage, each row's next 8 blocks (256 k) as the
// 16-byte-aligned span holding them, cp.async pieces from warps 2, 3 and 16..19.
constexpr int PIECES = 10;               // 16-byte pieces per row per raw stage: 136 bytes + up to 15 of alignment
constexpr int SLOT = 176;                // bytes per row per raw stage (>= 16 * PIECES; 11 x 16 bytes, odd)
// Repacked MXFP4_R rows: per raw stage, 16 blocks (512 k) of 128 rows as TMA
// tensor copies: two 128-byte-swizzled code boxes [128 rows][128 B] and one
// exponent box [128 rows][16 B].
constexpr int RC_BYTES = BM * 128;       // one code box
// MX (MXFP8 activations): the scale bytes of a token tile's rows, staged whole
// per tile (double-buffered): rows of at most this many bytes (cols <= 4096).
constexpr int MX_SPITCH_MAX = 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_STAGE_COLS = KSUB * BK / 2;   // bf16 A stage: 128 rows x 128 k, two per column
constexpr uint32_t A_STAGE_COLS_MX = 32;           // E2M1 A stage: four byte-container codes per column
// Per variant: TBN tokens per tile (128 or, when experts average more than 96
// routed tokens, 192 so that one tile covers them), SKV k stages.  TMEM columns: two TBN-column fp32 accumulators, then SKV A
// stages; MX adds per stage four columns of weight scales and TBN/32 of token
// scales.  Weight row m's scale for K step j of a stage sits in lane m, column
// SFA + m/32, byte j; token n's in lane 32q + n % 32, column SFB + n/32, byte j,
// for every lane quarter q (the MMA reads the quarter of the output row).
template <bool PLANAR, bool MX = false, int TBN = 128>
struct RawCfg {
    static constexpr int BLOCKS = PLANAR ? 16 : 8;                        // blocks per row per raw stage
    static constexpr int SR = PLANAR ? 2 : 4;                             // raw stages
    static constexpr int R_BYTES = PLANAR ? 2 * RC_BYTES + BM * 16 : BM * SLOT;   // 34816 / 22528
    static constexpr int ARRIVALS = PLANAR ? 1 : 192;                     // arrivals that fill a raw stage
    // + warps 24..27 (GGUF producers); MX: + four warps that place the token
    // scales in every TMEM lane quarter (the last four)
    static constexpr int THREADS = (PLANAR ? 768 : 896) + (MX ? 128 : 0);
    static constexpr int SF_WARP0 = THREADS / 32 - 4;
    // 192-token tiles: three k stages (MX) or two (bf16, whose 64-column A
    // stages leave room for two next to two 192-column accumulators)
    static constexpr int SKV = TBN > 128 ? (MX ? 3 : 2) : SK;
    static constexpr int XBF = TBN * BK * 2;                              // bf16: bytes of one 64-k X box
    static constexpr int XB = MX ? TBN * 128 : XBF;                       // bytes of one X box
    static constexpr int XS = MX ? XB : KSUB * XBF;                       // X bytes per 128-k stage
    static constexpr int SFBUF = TBN * MX_SPITCH_MAX;
    static constexpr int OFF_R = OFF_X + SKV * XS;
    static constexpr int OFF_SF = OFF_R + SR * R_BYTES;
    static constexpr int OFF_BAR = OFF_SF + (MX ? 2 * SFBUF : 0);
    static constexpr int N_BARS = 2 * SKV + 2 * SR + 4 + (MX ? 4 : 0);
    static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + alignment slack
    static constexpr uint32_t A_COL = 2 * TBN;
    static constexpr uint32_t SFA_COL = A_COL + SKV * A_STAGE_COLS_MX;
    static constexpr uint32_t SFB_COL = SFA_COL + SKV * 4;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(A_COL + SKV * (MX ? A_STAGE_COLS_MX : A_STAGE_COLS) + (MX ? SKV * (4 + TBN / 32) : 0) <= TMEM_COLS,
                  "TMEM budget");
};
}  // namespace mg

// 16-byte asynchronous copy global -> shared (dst, src 16-byte aligned);
// bytes beyond src_bytes (< 16 only at the end of the tensor) are zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// bf16 bit patterns of the eight E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}
// times 2^(e-127), as two byte tables (high bytes, low bytes) that prmt.b32
// indexes with a 3-bit magnitude.  For magnitude 2^j * (1 + m/2) the bf16
// pattern is ((e + j) << 7) | (m << 6); this holds while every exponent field
// e + j (j = -1..2) stays in the normal range 1..254, i.e. 2 <= e <= 252.
struct E2m1Tab {
    uint32_t hi0, hi1, lo0, lo1;
};

__device__ __forceinline__ bool e2m1_table(uint32_t e, E2m1Tab& t)
{
    // pairs of 16-bit patterns (low half = even magnitude): with b = e << 7,
    // [0, b - 128], [b, b + 64], [b + 128, b + 192], [b + 256, b + 320];
    // written as multiply-adds of e
    const uint32_t p01 = e * 0x00800000u - 0x00800000u;
    const uint32_t p23 = e * 0x00800080u + 0x00400000u;
    const uint32_t p45 = e * 0x00800080u + 0x00C00080u;
    const uint32_t p67 = e * 0x00800080u + 0x01400100u;
    t.hi0 = prmt(p01, p23, 0x7531u);
    t.hi1 = prmt(p45, p67, 0x7531u);
    t.lo0 = prmt(p01, p23, 0x6420u);
    t.lo1 = prmt(p45, p67, 0x6420u);
    return e - 2u <= 250u;
}

// Eight E2M1 codes, the nibbles of code word w (bytes i..i+3 of a block:
// element i+j in the low nibble of byte j, element i+16+j in the high one),
// -> bf16 pairs o_lo[0] = (i, i+1), o_lo[1] = (i+2, i+3), o_hi[0] =
// (i+16, i+17), o_hi[1] = (i+18, i+19).
__device__ __forceinline__ void e2m1_word(uint32_t w, const E2m1Tab& t, uint32_t (&o_lo)[2], uint32_t (&o_hi)[2])
{
    // prmt.b32 reads a selector's low 16 bits; bit 3 of a selector nibble
    // switches to replicating bit 7 of the selected byte, so magnitudes are
    // masked to 3 bits, and the sign masks come from that replication:
    // byte k of (w << 4) has the sign of the even nibbles in bit 7, byte k of
    // w that of the odd ones.
    const uint32_t mag = w & 0x77777777u, mag_h = mag >> 16, w4 = w << 4;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t m = q ? mag_h : mag;
        uint32_t H = prmt(t.hi0, t.hi1, m);
        const uint32_t L = prmt(t.lo0, t.lo1, m);
        const uint32_t neg = prmt(w4, w, q ? 0xfbeau : 0xd9c8u);   // 0xff where the code is negative
        H |= neg & 0x80808080u;
        o_lo[q] = prmt(L, H, 0x6240u);
        o_hi[q] = prmt(L, H, 0x7351u);
    }
}

// Exact bf16 of one block whose exponent leaves the table's range (zero or
// subnormal scales, overflow, NaN): code * 2^(e-127) in fp32, then rounded to
// bf16 (exact unless it overflows).
__device__ __forceinline__ void mxfp4_block_bf16_slow(uint32_t e, const uint32_t (&w)[4], uint32_t (&o)[16])
{
    using M = Fmt<QMV_MXFP4>;
    const float sc = M::e8m0_half(e);   // 2^(e-128); the codes below are doubled
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t nib = h ? (w[k] >> 4) & 0x0f0f0f0fu : w[k] & 0x0f0f0f0fu;
            const uint32_t v = M::lut4(__byte_perm(nib | (nib >> 4), 0u, 0x0020u) & 0xffffu);
            float f[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) f[j] = (float)(int)(int8_t)((v >> (8 * j)) & 0xffu) * sc;
            const __nv_bfloat162 p = __floats2bfloat162_rn(f[0], f[1]), q = __floats2bfloat162_rn(f[2], f[3]);
            o[8 * h + 2 * k] = *reinterpret_cast<const uint32_t*>(&p);
            o[8 * h + 2 * k + 1] = *reinterpret_cast<const uint32_t*>(&q);
        }
    }
}

// One 32-element MXFP4 block (17 bytes at byte offset o of a shared-memory
// row slot, any alignment) -> 16 bf16x2 words in element order (word i =
// elements 2i, 2i+1).
__device__ __forceinline__ void mxfp4_codes_bf16(uint32_t e, const uint32_t (&w)[4], uint32_t (&out)[16]);

__device__ __forceinline__ void mxfp4_block_bf16(const uint8_t* slot, int o, uint32_t (&out)[16])
{
    const uint8_t* p = slot + o;
    uint32_t w[4];
    load_words<4>(p + 1, w);   // the 16 code bytes
    mxfp4_codes_bf16(p[0], w, out);
}

// One block given as its exponent and its four code words.
__device__ __forceinline__ void mxfp4_codes_bf16(uint32_t e, const uint32_t (&w)[4], uint32_t (&out)[16])
{
    E2m1Tab t;
    if (e2m1_table(e, t)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t lo[2], hi[2];
            e2m1_word(w[k], t, lo, hi);
            out[2 * k] = lo[0];
            out[2 * k + 1] = lo[1];
            out[8 + 2 * k] = hi[0];
            out[8 + 2 * k + 1] = hi[1];
        }
    } else {
        mxfp4_block_bf16_slow(e, w, out);
    }
}

// The 16 code bytes of one MXFP4 block (as four words) -> its 32 E2M1 codes in
// the MMA's byte containers (the code in bits 5..2 of its byte), in element
// order: o[i] = elements 4i..4i+3.  Byte j of word k holds element 4k + j in
// its low nibble and element 16 + 4k + j in its high one.  The block's
// 2^(e-127) becomes the MMA's weight scale.
__device__ __forceinline__ void mxfp4_codes_e2m1x8(const uint32_t (&w)[4], uint32_t (&o)[8])
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        o[k] = (w[k] & 0x0f0f0f0fu) << 2;
        o[4 + k] = (w[k] >> 2) & 0x3c3c3c3cu;
    }
}

// tiles[0] = number of (expert, token tile) slots; slot i = (tiles[1+2i] =
// expert, tiles[2+2i] = token tile within the expert's group).
__global__ void k_moe_tiles(const int* __restrict__ offsets, const int* __restrict__ active, int bn,
                            int* __restrict__ tiles)
{
    const int lane = threadIdx.x;
    pdl_wait();
    const int na = active[0];
    int base = 0;
    for (int i0 = 0; i0 < na; i0 += 32) {
        const int i = i0 + lane;
        const int e = i < na ? active[1 + i] : 0;
        const int nt = i < na ? (offsets[e + 1] - offsets[e] + bn - 1) / bn : 0;
        int pre = nt;   // inclusive prefix sum over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, pre, o);
            if (lane >= o) pre += v;
        }
        const int start = base + pre - nt;
        for (int j = 0; j < nt; ++j) {
            tiles[1 + 2 * (start + j)] = e;
            tiles[2 + 2 * (start + j)] = j;
        }
        base += __shfl_sync(0xffffffffu, pre, 31);
    }
    if (lane == 0) tiles[0] = base;
}

// Xs[j] = x row perm[j] / kdiv for the n_valid grouped pairs (bf16, 16 bytes
// per thread).
__global__ void k_moe_gather(const uint16_t* __restrict__ x, const int* __restrict__ perm,
                             const int* __restrict__ offsets, int n_expert, int kdiv, int cols,
                             uint16_t* __restrict__ Xs)
{
    const int n_valid = offsets[n_expert];
    const int per_row = cols / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n_valid * per_row) return;
    const int j = (int)(i / per_row), c = (int)(i % per_row);
    const int src = perm[j] / kdiv;
    reinterpret_cast<uint4*>(Xs + (size_t)j * cols)[c] = reinterpret_cast<const uint4*>(x + (size_t)src * cols)[c];
}

// MXFP8 operands of the grouped pairs: row j = x row perm[j] / kdiv (fp32),
// codes to Xc[j][cols] and E8M0 scales to Sf[j][spitch] (bytes past the
// blocks: 127, a scale of one).  Eight threads per 32-element block.
__global__ void k_moe_gather_mxfp8(const float* __restrict__ x, const int* __restrict__ perm,
                                   const int* __restrict__ offsets, int n_expert, int kdiv, int cols, int spitch,
                                   uint8_t* __restrict__ Xc, uint8_t* __restrict__ Sf)
{
    const int n_valid = offsets[n_expert];
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t slot = g >> 3;
    const int sub = (int)(g & 7);
    const int j = (int)(slot / spitch), b = (int)(slot % spitch);
    if (j >= n_valid) return;   // whole groups of eight leave together
    const int nblk = cols / 32;
    if (b >= nblk) {
        if (sub == 0) Sf[(size_t)j * spitch + b] = 127;
        return;
    }
    const float* xr = x + (size_t)(perm[j] / kdiv) * cols + 32 * b;
    const float4 v = reinterpret_cast<const float4*>(xr)[sub];
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    const unsigned group = 0xffu << (threadIdx.x & 24);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(group, m, o, 8));
    const int E = mx_scale_exp(m);
    const uint32_t w = mx_e4m3(v.x, E) | (mx_e4m3(v.y, E) << 8) | (mx_e4m3(v.z, E) << 16) | (mx_e4m3(v.w, E) << 24);
    reinterpret_cast<uint32_t*>(Xc + (size_t)j * cols + 32 * b)[sub] = w;
    if (sub == 0) Sf[(size_t)j * spitch + b] = (uint8_t)(E + 127);
}

struct MoeGemmArgs {
    const uint8_t* W3d;   // 16-byte aligned
    int64_t rows;         // rows per expert
    int64_t rb;           // bytes per row
    int64_t total;        // bytes of all experts
    int nblk;             // MXFP4 blocks per row
    const int* offsets;
    const int* perm;
    const int* tiles;
    const float* bias;    // [n_expert][rows] or NULL
    float* out;           // row of pair p at out + p*rows
    unsigned* status;
    const uint8_t* sf;    // MX: E8M0 scales of the grouped pairs [sf_rows][spitch]
    int spitch, sf_rows;
};

// PLANAR: the experts are MXFP4_R rows (tmC, tmE: code and exponent tensor
// maps over all experts' rows); otherwise GGUF MXFP4 rows (tmC, tmE unused).
// MX: MXFP8 activations on kind::mxf8f6f4.block_scale -- the weights' E2M1
// codes in TMEM byte containers with their E8M0 exponents as the weight
// scales, the tokens' E4M3 codes in shared memory with their scales --
// instead of bf16 on kind::f16.
template <bool PLANAR, bool MX, int TBN>
__global__ void __launch_bounds__(mg::RawCfg<PLANAR, MX, TBN>::THREADS, 1)
    k_moe_gemm_mxfp4(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmE, const MoeGemmArgs a)
{
    using namespace mg;
    using RC = RawCfg<PLANAR, MX, TBN>;
    constexpr int SR = RC::SR, R_BYTES = RC::R_BYTES, OFF_BAR = RC::OFF_BAR, SC_BLOCKS = RC::BLOCKS;
    constexpr int OFF_R = RC::OFF_R, XS = RC::XS, SK = RC::SKV, BN = TBN;
    constexpr uint32_t A_COL = RC::A_COL, SFA_COL = RC::SFA_COL, SFB_COL = RC::SFB_COL;
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
    uint64_t* sff = acce + 2;   // MX: the scale rows of a token tile have landed (two buffers)
    uint64_t* sfe = sff + 2;    // MX: the scale warps are done with a buffer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2 + (MX ? 4 : 0));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    const int n_rt = (int)((a.rows + BM - 1) / BM);
    const int n_tiles = n_rt * a.tiles[0];
    const int nks = (a.nblk + 3) / 4;                      // 128-k stages (the last may be partly empty)
    const int nsc = (a.nblk + SC_BLOCKS - 1) / SC_BLOCKS;  // raw stages per row

    if (tid == 0) {
        // full: eight dequantising warps and the X copy (MX: and the four scale warps)
        for (int i = 0; i < SK; ++i) { mbar_init(&full[i], DEQ_WARPS / 2 + (MX ? 5 : 1)); mbar_init(&empty[i], 1); }
        for (int i = 0; i < SR; ++i) { mbar_init(&rf[i], RC::ARRIVALS); mbar_init(&re[i], DEQ_WARPS); }
        for (int i = 0; i < 2; ++i) { mbar_init(&accf[i], 1); mbar_init(&acce[i], 4); }
        if (MX) for (int i = 0; i < 2; ++i) { mbar_init(&sff[i], 1); mbar_init(&sfe[i], 4); }
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmX);
        if (PLANAR) {
            prefetch_tmap(&tmC);
            prefetch_tmap(&tmE);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() { *abort_flag = 1; };
    auto tile_of = [&](int t, int& e, int& nt, int& rt) {
        const int slot = t / n_rt;
        rt = t - slot * n_rt;
        e = a.tiles[1 + 2 * slot];
        nt = a.tiles[2 + 2 * slot];
    };

    if (MX && warp == 0) {
        // ---- token tiles: E4M3 codes, one 128-k box per stage; and once per
        // tile the tile's scale rows (double-buffered, refilled once the
        // scale warps are done with the buffer)
        if (lane == 0) {
            int s = 0, local = 0, pend = -1;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++local) {
                int e, nt, rt;
                tile_of(t, e, nt, rt);
                const int row0 = a.offsets[e] + nt * BN;
                const int nsf = min(BN, a.sf_rows - row0);
                const int sb = local & 1;
                if (!mbar_wait_backoff(&sfe[sb], (uint32_t)(((local >> 1) & 1) ^ 1), a.status, 128)) { fail(); break; }
                mbar_arrive_expect_tx(&sff[sb], (uint32_t)(nsf * a.spitch));
                bulk_g2s(smem + RC::OFF_SF + sb * RC::SFBUF, a.sf + (size_t)row0 * a.spitch, (uint32_t)(nsf * a.spitch),
                         &sff[sb]);
                pend = local;
                bool bad = false;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_backoff(&empty[s], ph, a.status, 128)) { bad = true; break; }
                    mbar_arrive_expect_tx(&full[s], RC::XB);
                    tma_load_2d(smem + OFF_X + s * XS, &tmX, ks * 128, row0, &full[s]);
                    if (++s == SK) { s = 0; ph ^= 1; }
                }
                if (bad) { fail(); break; }
            }
            // the last scale copy lands before the block can leave (bounded)
            if (pend >= 0)
                mbar_wait_bounded(&sff[pend & 1], (uint32_t)((pend >> 1) & 1), a.status, 100000000ull);
        }
    } else if (MX && warp >= RC::SF_WARP0) {
        // ---- token scales: each of the four warps writes its lane quarter;
        // lane l holds the words of tokens l, l + 32, l + 64, l + 96 (columns
        // SFB + 0..3 of the stage)
        const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        int s = 0, local = 0;
        uint32_t ph = 1;
        bool bad = false;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x, ++local) {
            int e, nt, rt;
            tile_of(t, e, nt, rt);
            const int row0 = a.offsets[e] + nt * BN;
            const int nsf = min(BN, a.sf_rows - row0);
            const int sb = local & 1;
            const uint8_t* sfb = smem + RC::OFF_SF + sb * RC::SFBUF;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sff[sb], (uint32_t)((local >> 1) & 1), a.status))) {
                bad = true;
            }
            for (int ks = 0; ks < nks && !bad; ++ks) {
                if (!__all_sync(0xffffffffu, mbar_wait_backoff(&empty[s], ph, a.status, 128))) { bad = true; break; }
#pragma unroll
                for (int c = 0; c < TBN / 32; ++c) {
                    const int j = lane + 32 * c;
                    tmem_st1_async(tq + SFB_COL + (TBN / 32) * s + c,
                                   j < nsf ? *reinterpret_cast<const uint32_t*>(sfb + j * a.spitch + 4 * ks)
                                           : 0x7f7f7f7fu);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[s]);
                if (++s == SK) { s = 0; ph ^= 1; }
            }
            if (bad) { fail(); break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfe[sb]);   // done with this tile's scale rows
        }
    } else if (warp == 0) {
        // ---- packed token tiles
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                int e, nt, rt;
                tile_of(t, e, nt, rt);
                const int row0 = a.offsets[e] + nt * BN;
                for (int ks = 0; ks < nks; ++ks) {
                    if (!mbar_wait_backoff(&empty[s], ph, a.status, 128)) { fail(); break; }
                    mbar_arrive_expect_tx(&full[s], KSUB * RC::XBF);
#pragma unroll
                    for (int j = 0; j < KSUB; ++j)
                        tma_load_2d(smem + OFF_X + s * XS + j * RC::XBF, &tmX, (ks * KSUB + j) * BK, row0, &full[s]);
                    if (++s == SK) { s = 0; ph ^= 1; }
                }
            }
        }
    } else if (PLANAR && warp == 2) {
        // ---- raw weights, repacked rows: three TMA tensor copies per stage
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 1;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
                int e, nt, rt;
                tile_of(t, e, nt, rt);
                const int y = (int)((int64_t)e * a.rows + (int64_t)rt * BM);   // first row of the tile
                for (int sc = 0; sc < nsc; ++sc) {
                    if (!mbar_wait_backoff(&re[s], ph, a.status, 128)) { fail(); break; }
                    uint8_t* buf = smem + OFF_R + s * R_BYTES;
                    mbar_arrive_expect_tx(&rf[s], R_BYTES);
                    tma_load_2d(buf, &tmC, sc * 256, y, &rf[s]);
                    tma_load_2d(buf + RC_BYTES, &tmC, sc * 256 + 128, y, &rf[s]);
                    tma_load_2d(buf + 2 * RC_BYTES, &tmE, sc * 16, y, &rf[s]);
                    if (++s == SR) { s = 0; ph ^= 1; }
                }
            }
        }
    } else if (!PLANAR && (warp == 2 || warp == 3 || (warp >= EPI_WARP0 + 4 && warp < EPI_WARP0 + 8))) {   // 2, 3, 24..27
        // ---- raw weights: for each row of the tile, the 16-byte-aligned span
        // holding its next (up to) 8 blocks, as 16-byte cp.async pieces spread
        // over the 192 threads of warps 2, 3 and 16..19 (consecutive threads take
        // consecutive pieces of a row).  The last piece of the tensor reads
        // only the bytes that exist and zero-fills the rest.  Each thread then
        // arrives on the stage's barrier once its own copies have landed.
        const int pt = warp < 4 ? tid - 64 : tid - 32 * (EPI_WARP0 + 4) + 64;
        int s = 0;
        uint32_t ph = 1;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x) {
            int e, nt, rt;
            tile_of(t, e, nt, rt);
            const int64_t tile0 = ((int64_t)e * a.rows + (int64_t)rt * BM) * a.rb;   // byte offset of row 0
            const int nrows = (int)min((int64_t)BM, a.rows - (int64_t)rt * BM);
            bool bad = false;
            for (int sc = 0; sc < nsc; ++sc) {
                if (!__all_sync(0xffffffffu, mbar_wait_backoff(&re[s], ph, a.status, 128))) { bad = true; break; }
                uint8_t* buf = smem + OFF_R + s * R_BYTES;
                const int nb = min(SC_BLOCKS, a.nblk - sc * SC_BLOCKS);
                for (int p = pt; p < nrows * PIECES; p += RC::ARRIVALS) {
                    const int i = p / PIECES, j = p - i * PIECES;
                    const int64_t b0 = tile0 + (int64_t)i * a.rb + (int64_t)sc * SC_BLOCKS * 17;
                    const int64_t src = (b0 & ~int64_t(15)) + 16 * j;
                    if (src < b0 + nb * 17)
                        cp_async16(buf + i * SLOT + 16 * j, a.W3d + src, (uint32_t)min((int64_t)16, a.total - src));
                }
                cp_async_arrive_noinc(&rf[s]);
                if (++s == SR) { s = 0; ph ^= 1; }
            }
            if (bad) { fail(); break; }
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN);
            // MX: E2M1 A x E4M3 B, E8M0 scales, M = 128, N = 128; K step j reads
            // byte j of the scale words
            auto idesc_mx = [](uint32_t j) {
                return (j << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
                       ((uint32_t)(BM >> 7) << 27) | (j << 29);
            };
            int s = 0;
            uint32_t pf = 0;
            int local = 0;
            for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
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
                    if constexpr (MX) {
                        const uint32_t at = tmem + A_COL + s * A_STAGE_COLS_MX;
                        const uint64_t bdesc = smem_desc_sw128(smem + OFF_X + s * XS);
#pragma unroll
                        for (int j = 0; j < 4; ++j)   // A: 8 TMEM columns, B: 32 bytes per K = 32 step
                            mma_mx_ts(d, at + 8 * j, bdesc + 2 * j, idesc_mx((uint32_t)j), tmem + SFA_COL + 4 * s,
                                      tmem + SFB_COL + (TBN / 32) * s, (ks | j) != 0);
                    } else {
                        const uint32_t at = tmem + A_COL + s * A_STAGE_COLS;
#pragma unroll
                        for (int j = 0; j < KSUB; ++j) {
                            const uint64_t bdesc = smem_desc_sw128(smem + OFF_X + s * XS + j * RC::XBF);
#pragma unroll
                            for (int k4 = 0; k4 < BK / 16; ++k4)   // A: 8 TMEM columns, B: 32 bytes per K = 16 step
                                mma_f16_ts(d, at + 32 * j + 8 * k4, bdesc + 2 * k4, idesc, (ks | j | k4) != 0);
                        }
                    }
                    mma_commit(&empty[s]);
                    if (++s == SK) { s = 0; pf ^= 1; }
                }
                if (bad) { fail(); break; }
                mma_commit(&accf[buf]);
            }
        }
    } else if (warp >= 4 && warp < 4 + DEQ_WARPS) {
        // ---- dequantisers, two groups of eight warps taking alternate 128-k
        // stages (group g the stages of even / odd global index; with four
        // stages each group cycles through two of them).  Within a group,
        // thread t -> weight row t % 128 (its TMEM lane: warp % 4 is the warp's
        // lane quarter) and block 2c + t / 128 of each 64-k chunk c, i.e. A
        // tile columns 16 * (t / 128) .. +15
        const int t0 = (tid - 128) & 255, grp = (tid - 128) >> 8, r = t0 & 127, half = t0 >> 7;
        const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's lane quarter
        const uint32_t ta = tq + A_COL + 16 * half;
        int sr = 0;
        uint32_t prf = 0;
        uint32_t gk = 0;   // global index of the next 128-k stage
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x) {
            int e, nt, rt;
            tile_of(t, e, nt, rt);
            const int64_t row = (int64_t)rt * BM + r;
            const int64_t row_start = ((int64_t)e * a.rows + row) * a.rb;   // byte offset of the row
            bool bad = false;
            for (int sc = 0; sc < nsc && !bad; ++sc) {
                if (!__all_sync(0xffffffffu, mbar_wait_backoff(&rf[sr], prf, a.status, 32))) { bad = true; break; }
                const uint8_t* rbuf = smem + OFF_R + sr * R_BYTES;
                const uint8_t* slot = rbuf + r * SLOT;
                const int off = (int)((row_start + (int64_t)sc * SC_BLOCKS * 17) & 15);
                const int nb = min(SC_BLOCKS, a.nblk - sc * SC_BLOCKS);
                const int nc = (nb + 1) / 2;
                // one 128-k stage (chunks 2cs, 2cs+1) per pass: two independent
                // blocks per thread in flight, one wait for both TMEM stores
                for (int cs = 0; 2 * cs < nc; ++cs, ++gk) {
                    if ((int)(gk & 1) != grp) continue;
                    const int s = (int)(gk % SK);
                    const uint32_t pe = ((gk / SK) & 1) ^ 1;
                    if (!__all_sync(0xffffffffu, mbar_wait_backoff(&empty[s], pe, a.status, 32))) { bad = true; break; }
                    tc_fence_after();
                    if constexpr (MX) {
                        // E2M1 codes: block 2j + half of the stage at columns 8 (2j + half)
#pragma unroll
                        for (int j = 0; j < KSUB; ++j) {
                            const int blk = 2 * (KSUB * cs + j) + half;
                            uint32_t o[8];
                            if (row < a.rows && blk < nb) {
                                uint32_t w[4];
                                if constexpr (PLANAR) {
                                    const uint4 u = *reinterpret_cast<const uint4*>(
                                        rbuf + (blk >> 3) * RC_BYTES + r * 128 + (((blk & 7) ^ (r & 7)) << 4));
                                    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
                                } else {
                                    load_words<4>(slot + off + 17 * blk + 1, w);
                                }
                                mxfp4_codes_e2m1x8(w, o);
                            } else {
#pragma unroll
                                for (int i = 0; i < 8; ++i) o[i] = 0u;
                            }
                            tmem_st8_async(tq + A_COL + s * A_STAGE_COLS_MX + 16 * j + 8 * half, o);
                        }
                        if (half == 0) {
                            // the row's four block exponents: its scale word (column m / 32)
                            uint32_t sw = 0;
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                const int blk = 4 * cs + b;
                                uint32_t ev = 127u;
                                if (row < a.rows && blk < nb)
                                    ev = PLANAR ? rbuf[2 * RC_BYTES + r * 16 + blk] : slot[off + 17 * blk];
                                sw |= ev << (8 * b);
                            }
                            tmem_st1_async(tq + SFA_COL + 4 * s + (uint32_t)(warp & 3), sw);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < KSUB; ++j) {
                            const int blk = 2 * (KSUB * cs + j) + half;
                            uint32_t o[16];
                            if (row < a.rows && blk < nb) {
                                if constexpr (PLANAR) {
                                    // code box blk / 8, 16-byte chunk (blk % 8) swizzled by the row
                                    const uint4 u = *reinterpret_cast<const uint4*>(
                                        rbuf + (blk >> 3) * RC_BYTES + r * 128 + (((blk & 7) ^ (r & 7)) << 4));
                                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                                    mxfp4_codes_bf16(rbuf[2 * RC_BYTES + r * 16 + blk], w, o);
                                } else {
                                    mxfp4_block_bf16(slot, off + 17 * blk, o);
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] = 0u;
                            }
                            tmem_st16_async(ta + s * A_STAGE_COLS + 32 * j, o);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[s]);
                }
                if (bad) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&re[sr]);
                if (++sr == SR) { sr = 0; prf ^= 1; }
            }
            if (bad) { fail(); break; }
        }
    } else if (warp >= EPI_WARP0) {
        // ---- epilogue: lane quarter (warp % 4) of the 128 TMEM lanes; column
        // j of the accumulator is the expert's grouped pair offsets[e] + nt*128 + j
        const int q = warp & 3;
        int local = 0;
        for (int t = blockIdx.x; t < n_tiles && !__any_sync(0xffffffffu, *abort_flag); t += gridDim.x, ++local) {
            int e, nt, rt;
            tile_of(t, e, nt, rt);
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            // warp-uniform: every lane must take part in the tcgen05.ld below
            if (!__all_sync(0xffffffffu, mbar_wait_backoff(&accf[buf], use & 1, a.status, 512))) { fail(); break; }
            tc_fence_after();
            const int64_t row = (int64_t)rt * BM + 32 * q + lane;
            const bool row_ok = row < a.rows;
            const float bv = (a.bias && row_ok) ? a.bias[(int64_t)e * a.rows + row] : 0.f;
            const int g0 = a.offsets[e] + nt * BN, cnt = a.offsets[e + 1] - g0;
            for (int c16 = 0; c16 < BN / 16; ++c16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + buf * BN + c16 * 16, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int j = c16 * 16 + i;
                    if (j < cnt && row_ok) a.out[(int64_t)a.perm[g0 + j] * a.rows + row] = v[i] + bv;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[buf]);
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

inline size_t tiles_bytes(int64_t n_pairs)
{
    const size_t slots = (size_t)n_pairs + (size_t)n_pairs / mg::BN + 1;   // >= sum over experts of ceil(count/128) (and /192)
    return ((1 + 2 * slots) * 4 + 255) & ~size_t(255);
}

}  // namespace qmv

namespace qmv {
inline int mx_spitch(int64_t cols)   // scale bytes per token row: 4 per 128-k stage, 16-byte multiple
{
    const int64_t nks = (cols / 32 + 3) / 4;
    return (int)((4 * nks + 15) & ~int64_t(15));
}
inline size_t r256g(size_t v) { return (v + 255) & ~size_t(255); }
}  // namespace qmv

// Bytes of workspace beyond the grouping that the grouped GEMM needs: the slot
// list and the packed activations (bf16, or MXFP8 codes and scales).
size_t qmv_moe_gemm_extra_bytes(int64_t cols, int64_t n_pairs, bool mx)
{
    using namespace qmv;
    if (mx)
        return tiles_bytes(n_pairs) + r256g((size_t)n_pairs * (size_t)cols) +
               r256g((size_t)n_pairs * (size_t)mx_spitch(cols));
    return tiles_bytes(n_pairs) + (size_t)n_pairs * (size_t)cols * 2;
}

// Enqueues the slot list, the gather and the grouped GEMM.  ws points at the
// GEMM's part of the workspace (qmv_moe_gemm_extra_bytes bytes, 256-aligned).
// planar: W3d holds MXFP4_R rows.  mx: x is fp32, quantised to MXFP8 by the
// gather, and the GEMM runs on kind::mxf8f6f4 (cols <= 4096); otherwise x is
// bf16.  Returns 0, -2 (shape beyond the plan), -6 (launch failure) or -8
// (tensor map).
int qmv_launch_moe_gemm_mxfp4(const void* W3d, bool planar, bool mx, int n_expert, int64_t rows, int64_t cols,
                              const void* x, int kdiv, int64_t n_pairs, const int* offsets, const int* active,
                              const int* perm, void* ws, float* out, const float* bias, cudaStream_t st)
{
    using namespace qmv;
    const int spitch = mx_spitch(cols);
    if (mx && spitch > mg::MX_SPITCH_MAX) return -2;
    int* tiles = static_cast<int*>(ws);
    uint8_t* act = static_cast<uint8_t*>(ws) + tiles_bytes(n_pairs);
    uint8_t* sf = act + r256g((size_t)n_pairs * (size_t)cols);
    // 192-token tiles when the experts average more than 96 routed pairs, so
    // that one tile pass over an expert's rows (one dequantisation of them)
    // covers its tokens
    // MX with at most 32 routed pairs per expert on average: 64-token tiles
    // (the E2M1 operands cost little to form, so the MMA's padded columns are
    // what a mostly empty 128-token tile wastes)
    const int tbn = n_pairs > (int64_t)96 * n_expert ? 192 : (mx && n_pairs <= (int64_t)32 * n_expert) ? 64 : 128;
    k_moe_tiles<<<1, 32, 0, st>>>(offsets, active, tbn, tiles);
    CUtensorMap tmX, tmC, tmE;
    if (mx) {
        const int64_t threads = n_pairs * spitch * 8;
        k_moe_gather_mxfp8<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
            static_cast<const float*>(x), perm, offsets, n_expert, kdiv, (int)cols, spitch, act, sf);
        if (cudaGetLastError() != cudaSuccess) return -6;
        if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, act, (uint64_t)cols, (uint64_t)n_pairs,
                          (uint64_t)cols, 128, (uint32_t)tbn, CU_TENSOR_MAP_SWIZZLE_128B))
            return -8;
    } else {
        uint16_t* Xs = reinterpret_cast<uint16_t*>(act);
        const int64_t per = n_pairs * (cols / 8);
        k_moe_gather<<<(unsigned)((per + 255) / 256), 256, 0, st>>>(static_cast<const uint16_t*>(x), perm, offsets,
                                                                      n_expert, kdiv, (int)cols, Xs);
        if (cudaGetLastError() != cudaSuccess) return -6;
        if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xs, (uint64_t)cols, (uint64_t)n_pairs,
                          (uint64_t)cols * 2, mg::BK, (uint32_t)tbn, CU_TENSOR_MAP_SWIZZLE_128B))
            return -8;
    }
    MoeGemmArgs a;
    a.W3d = static_cast<const uint8_t*>(W3d);
    a.rows = rows;
    a.nblk = (int)(cols / 32);
    a.rb = planar ? (((int64_t)a.nblk * 17 + 15) & ~int64_t(15)) : (int64_t)a.nblk * 17;
    a.total = (int64_t)n_expert * rows * a.rb;
    a.offsets = offsets;
    a.perm = perm;
    a.tiles = tiles;
    a.bias = bias;
    a.out = out;
    a.status = status_word();
    a.sf = sf;
    a.spitch = spitch;
    a.sf_rows = (int)n_pairs;
    if (planar) {
        // codes: [all rows][16 * nblk bytes], exponents: [all rows][nblk bytes] at +16*nblk; row pitch rb
        const uint64_t all_rows = (uint64_t)n_expert * (uint64_t)rows;
        if (!make_tmap_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, W3d, (uint64_t)a.nblk * 16, all_rows, (uint64_t)a.rb,
                          128, mg::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tmap_2d(&tmE, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<const uint8_t*>(W3d) + (size_t)a.nblk * 16,
                          (uint64_t)a.nblk, all_rows, (uint64_t)a.rb, 16, mg::BM, CU_TENSOR_MAP_SWIZZLE_NONE))
            return -8;
    } else {
        tmC = tmX;   // unused by the GGUF-layout kernel
        tmE = tmX;
    }
    auto launch = [&](auto* k, int threads, int smem) {
        prepare_kernel(k, threads, smem);
        return launch_ex(k, dim3(num_sms()), dim3(threads), smem, st, false, tmX, tmC, tmE, a) == cudaSuccess ? 0 : -6;
    };
    using mg::RawCfg;
    if (planar) {
        if (!mx)
            return tbn == 192 ? launch(&k_moe_gemm_mxfp4<true, false, 192>, RawCfg<true, false, 192>::THREADS,
                                       RawCfg<true, false, 192>::SMEM)
                              : launch(&k_moe_gemm_mxfp4<true, false, 128>, RawCfg<true>::THREADS, RawCfg<true>::SMEM);
        if (tbn == 64)
            return launch(&k_moe_gemm_mxfp4<true, true, 64>, RawCfg<true, true, 64>::THREADS,
                          RawCfg<true, true, 64>::SMEM);
        return tbn == 192
                   ? launch(&k_moe_gemm_mxfp4<true, true, 192>, RawCfg<true, true, 192>::THREADS,
                            RawCfg<true, true, 192>::SMEM)
                   : launch(&k_moe_gemm_mxfp4<true, true, 128>, RawCfg<true, true>::THREADS, RawCfg<true, true>::SMEM);
    }
    if (!mx)
        return tbn == 192 ? launch(&k_moe_gemm_mxfp4<false, false, 192>, RawCfg<false, false, 192>::THREADS,
                                   RawCfg<false, false, 192>::SMEM)
                          : launch(&k_moe_gemm_mxfp4<false, false, 128>, RawCfg<false>::THREADS, RawCfg<false>::SMEM);
    if (tbn == 64)
        return launch(&k_moe_gemm_mxfp4<false, true, 64>, RawCfg<false, true, 64>::THREADS,
                      RawCfg<false, true, 64>::SMEM);
    return tbn == 192 ? launch(&k_moe_gemm_mxfp4<false, true, 192>, RawCfg<false, true, 192>::THREADS,
                               RawCfg<false, true, 192>::SMEM)
                      : launch(&k_moe_gemm_mxfp4<false, true, 128>, RawCfg<false, true>::THREADS,
                               RawCfg<false, true>::SMEM);
}

// ---- repack: GGUF MXFP4 rows -> MXFP4_R rows --------------------------------------
// One thread per block: its 16 code bytes to 16-byte-aligned position 16*b of
// the row, its exponent to 16*nblk + b; the first thread of a row zeroes the
// row's padding.
__global__ void k_repack_mxfp4(const uint8_t* __restrict__ W, int64_t rows, int nblk, int64_t rb_out,
                               uint8_t* __restrict__ out)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * nblk) return;
    const int64_t r = i / nblk;
    const int b = (int)(i - r * nblk);
    const uint8_t* src = W + i * 17;
    uint8_t* row = out + r * rb_out;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = (uint32_t)src[1 + 4 * k] | ((uint32_t)src[2 + 4 * k] << 8) | ((uint32_t)src[3 + 4 * k] << 16) |
               ((uint32_t)src[4 + 4 * k] << 24);
    *reinterpret_cast<uint4*>(row + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    row[16 * nblk + b] = src[0];
    if (b == 0)
        for (int64_t k = (int64_t)17 * nblk; k < rb_out; ++k) row[k] = 0;
}

int qmv_launch_repack_mxfp4(const void* W, int64_t rows, int64_t cols, void* Wout, cudaStream_t st)
{
    const int nblk = (int)(cols / 32);
    const int64_t rb_out = ((int64_t)nblk * 17 + 15) & ~int64_t(15);
    const int64_t n = rows * nblk;
    k_repack_mxfp4<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(static_cast<const uint8_t*>(W), rows, nblk, rb_out,
                                                                static_cast<uint8_t*>(Wout));
    return cudaGetLastError() == cudaSuccess ? 0 : -6;
}
