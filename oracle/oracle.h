/*
 * oracle.h -- plain, slow CPU oracle for block-quantised weight multiplies.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no source with the CUDA library.
 *
 * Subject: the llamay documentation pages --
 *   "Models and formats" (llamay.com/docs/models), section "Tensor formats":
 *       the block formats that are read (Q4_0, Q5_0, Q8_0, the K-quants, MXFP4).
 *   "Architecture" (llamay.com/docs/architecture), section "The package map":
 *       pkg/quant (block layouts, dequantisation, fused W4A8 kernels) and
 *       pkg/tensor (MatVec for decode, MatMul for prefill).
 *   "Architecture", section "The forward pass": batched prefill is an
 *       optimisation of sequential decode and must agree with it.
 *   "Models and formats", section "Architectures": mixture-of-experts models
 *       store experts as stacked 3-D tensors, a router picks k of n per token;
 *       gpt-oss puts a bias on every expert projection.
 *
 * The byte layouts follow the GGUF block conventions (the pages name the
 * formats but print no layouts); see blocks.c for each one.
 *
 * Arithmetic: integer codes are exact; scales and sums are carried in fp64.
 * Compile with -ffp-contract=off and without fast-math so that every fp32
 * operation in the activation quantiser is a single IEEE rounding.
 */
#ifndef QMV_ORACLE_H
#define QMV_ORACLE_H

#include <stdint.h>
#include <stddef.h>

/* Type numbers (the oracle's own table). */
enum {
    ORC_Q4_0 = 1, ORC_Q5_0 = 2, ORC_Q8_0 = 3, ORC_Q4_K = 4, ORC_Q6_K = 5,
    ORC_MXFP4 = 6, ORC_Q8_K = 7, ORC_F32 = 8, ORC_BF16 = 9,
    ORC_Q4_1 = 10, ORC_Q5_1 = 11, ORC_Q5_K = 12, ORC_Q2_K = 13, ORC_Q3_K = 14,
    ORC_Q8_1 = 15, ORC_F16 = 16,
    ORC_MXFP8 = 17   /* activations: E8M0 scale | 32 E4M3 codes, 33 bytes (mx.c) */
};

/* Return codes. */
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ESHAPE = -2, ORC_EUNSUP = -3, ORC_ERANGE = -4 };

/* ---- fp.c : IEEE-754 binary16 / bfloat16 written out from the encodings ---- */
double   orc_f16_to_f64(uint16_t h);
uint16_t orc_f32_to_f16_rn(float f);
double   orc_bf16_to_f64(uint16_t b);
uint16_t orc_f32_to_bf16_rn(float f);

/* ---- blocks.c : one block -> exact integer codes and scales ---- */
/* A decoded block.  Every element i satisfies
 *     w_i = d * sub_scale[i] * code[i] - dmin * sub_min[i]
 * exactly (in real arithmetic).  For the 32-element formats sub_scale = 1 and
 * sub_min = 0 (Q4_1 and Q5_1: sub_min = 1 and dmin = -m, their offset;
 * Q8_1 is Q8_0's codes and scale, its second field unused);
 * Q4_K and Q5_K carry their 6-bit sub-block scale/min, Q2_K its 4-bit
 * scale/min, Q3_K its 6-bit scale minus 32, Q6_K its int8 sub-block scale.  MXFP4 stores twice the E2M1 value (an integer) in code[]
 * and 2^(e-128) in d. */
typedef struct {
    int     n;              /* elements in the block: 32 or 256 */
    int32_t code[256];
    int32_t sub_scale[256];
    int32_t sub_min[256];
    double  d;
    double  dmin;
} orc_block;

int64_t orc_block_elems(int type);           /* 32 / 256, or 0 if not a block type */
/* Plain (unblocked) weight types: F32, F16, BF16 -- one value per element,
 * little-endian, row-major.  Their bytes per element, or 0 for block types. */
int64_t orc_plain_bytes(int type);
int64_t orc_block_bytes(int type);           /* bytes per block, or 0 */
int     orc_decode_block(int type, const uint8_t* blk, orc_block* out);
/* Element i of a row of a plain weight type (F32, F16, BF16), exactly. */
double  orc_plain_weight(int type, const uint8_t* row, int64_t i);
/* Decoded weight of element i as an exact fp64 value. */
double  orc_block_weight(const orc_block* b, int i);
/* rows x cols weights -> fp32.  Every format's weight is exactly representable
 * in fp32 except Q4_K's, which is the single rounding RN_fp32(d*sc*q - dmin*m),
 * and Q4_1's and Q5_1's, the single rounding RN_fp32(d*q + m).  Plain F16,
 * BF16 and F32 weights convert exactly. */
int     orc_dequant(int type, const uint8_t* W, int64_t rows, int64_t cols, float* out);

/* ---- quant.c : the 8-bit activation quantisers ---- */
/* x holds n values (n a multiple of the block size, vectors laid end to end);
 * out receives n/bs blocks of ORC_Q8_0 (fp16 d, int8[32]) or ORC_Q8_K
 * (fp32 d, int8[256], int16 bsums[16]). */
int     orc_quantize_act(int atype, const float* x, int64_t n, uint8_t* out);
/* fp32 weights to Q4_0, Q4_1, Q5_0, Q5_1, Q8_0 (n a multiple of 32) or Q4_K,
 * Q5_K, Q6_K blocks (n a multiple of 256) (wquant.c). */
int     orc_quantize_weights(int wtype, const float* w, int64_t n, uint8_t* out);
/* Decode one activation block to its integer codes and fp64 scale. */
int     orc_decode_act_block(int atype, const uint8_t* blk, int32_t* q, double* d, int32_t* bsums);

/* ---- mm.c : integer block dots, matvec, matmul, mixture of experts ---- */
/* Per-block integers of one weight row against one quantised activation
 * vector: for block b, out[2b] = S_b = sum_i sub_scale_i*code_i*xq_i and
 * out[2b+1] = Mn_b = sum_i sub_min_i*xq_i (zero except Q4_K).
 * W is rows x (cols/bs) blocks, xq is n_vec x (cols/bs) activation blocks,
 * out is [n_vec][rows][cols/bs][2]. */
int     orc_block_dots(int wtype, const uint8_t* W, int64_t rows, int64_t cols,
                       const uint8_t* xq, int64_t n_vec, int64_t* out);

/* y[v][j] = sum_c w[r_j][c] * xhat[v][c] for the selected rows r_j
 * (row_ids == NULL selects all rows in order).  atype:
 *   ORC_F32  : x is fp32 [n_vec][cols], xhat = x, w exact;
 *   ORC_BF16 : x is bf16 [n_vec][cols], xhat = x, w rounded to bf16 first;
 *   ORC_MXFP8: x is [n_vec][cols/32] MXFP8 blocks (32-element weight types),
 *              xhat = E4M3 * 2^(e-127) exactly, products in fp64;
 *   ORC_Q8_0 / ORC_Q8_K : x is [n_vec][cols/bs] blocks, the per-block integer
 *              dots are scaled by the weight and activation scales in fp64.
 * yabs (nullable) receives sum_c |w*xhat| per output, in the same layout. */
int     orc_matvec(int wtype, int atype, const uint8_t* W, int64_t rows, int64_t cols,
                   const void* x, int64_t n_vec, const int64_t* row_ids, int64_t n_rows,
                   double* y, double* yabs);

/* Mixture of experts over a stacked weight tensor W3d[n_expert][rows][cols].
 * ids, gates: [n_tok][k].  bias: [n_expert][rows] or NULL.
 *   gates == NULL : x is [n_tok][cols] (shared by the k slots);
 *                   y[t][s][r] = W[ids[t][s]] x_t + bias[ids[t][s]]
 *   gates != NULL : x is [n_tok][k][cols] (one input per slot);
 *                   y[t][r] = sum_s gates[t][s] * (W[ids[t][s]] x_{t,s} + bias[ids[t][s]])
 * yabs is sum |w*xhat| (+|b|), gate-weighted in the second form. */
int     orc_moe(int wtype, int atype, const uint8_t* W3d, int64_t n_expert,
                int64_t rows, int64_t cols, const int32_t* ids, const float* gates,
                int64_t k, const void* x, int64_t n_tok, const float* bias,
                double* y, double* yabs);

/* ---- mx.c : MXFP8 activations ---- */
double  orc_e4m3_to_f64(uint8_t b);
/* Round to the nearest E4M3 value (ties to even), magnitudes clamped to 448. */
uint8_t orc_f64_to_e4m3_rn_sat(double v);
/* n fp32 values (n a multiple of 32, all finite) -> n/32 MXFP8 blocks. */
int     orc_quantize_mxfp8(const float* x, int64_t n, uint8_t* out);
/* Element i of an MXFP8 block, exactly. */
double  orc_mxfp8_value(const uint8_t* blk, int i);

/* ---- moeblock.c : the router and the gated activation of an expert block ---- */
/* logits[t][e] = x[t] . Wr[e] (+ br[e]) in fp32, in the 32-partial order the
 * top-k decision is taken in (see moeblock.c). */
int     orc_router(const float* x, const float* Wr, const float* br, int64_t n_tok, int64_t hidden,
                   int64_t n_expert, float* logits);
/* ids[t][s]: the k largest logits (ties to the lower id), descending; gates:
 * softmax over them in fp64. */
int     orc_topk_softmax(const float* logits, int64_t n_tok, int64_t n_expert, int64_t k, int32_t* ids,
                         double* gates);
/* min(g, limit) * sigmoid(alpha * min(g, limit)) * (clamp(u, -limit, limit) + 1), fp64 */
double  orc_swiglu(double g, double u, double alpha, double limit);

#endif