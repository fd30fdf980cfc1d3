/*
 * qmv.h -- C ABI of the GB300 block-quantised matrix multiply library (libqmv).
 *
 * The library multiplies by weights stored in GGUF quantised blocks, unpacking
 * and scaling them inside the dot product.  The operations are those named on
 * the llamay documentation pages:
 *   "Architecture" page, "The package map": pkg/quant owns the block layouts,
 *     dequantisation and the fused W4A8 kernels (4-bit weights, 8-bit
 *     activations); pkg/tensor owns MatVec (decode) and MatMul (prefill).
 *   "Architecture" page, "The two phases": decode is bound by memory, prefill
 *     by arithmetic, so the two get different kernels.
 *   "Architecture" page, "A request, end to end": decode is batched across
 *     sequences so that the weights are read once for N of them.
 *   "Models and formats" page, "Tensor formats": the block formats.
 *   "Models and formats" page, "Architectures": mixture-of-experts models keep
 *     experts as stacked 3-D tensors, a router picks k of n per token, and
 *     gpt-oss carries a bias on every expert projection.
 *
 * Conventions shared by every call
 * ---------------------------------
 *  - A weight matrix W has `rows` outputs and `cols` inputs.  Each row is
 *    cols/bs consecutive blocks, rows are consecutive (the GGUF layout).  W must
 *    start on a 16-byte boundary.
 *  - Every pointer argument named W, x, xq, X, y, Y, ids, gates, bias, out is a
 *    DEVICE pointer owned by the caller; the library never frees or keeps it.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call only enqueues work on that stream and returns; none
 *    synchronises.  Inputs must stay valid, and outputs must not be read, until
 *    the stream reaches the call.  Outputs must not alias inputs.
 *  - Calls allocate no device memory.  The mixture-of-experts call and the
 *    W4A8 prefill need scratch, given once through qmv_set_workspace().
 *  - Errors: every call validates its arguments on the host before launching
 *    and returns a negative qmv_status without launching anything on failure;
 *    qmv_last_error() then names what is supported (the pages' convention of
 *    refusing with a message that names what does work).  A launch failure
 *    returns QMV_ERR_CUDA.  Faults found on the device (an expert id out of
 *    range, a pipeline wait that gave up) set a device status word that
 *    qmv_get_status() reads; kernels never trap.
 *  - Results are deterministic: the same inputs give bit-identical outputs,
 *    and output row r of vector v does not depend on the other vectors of the
 *    batch (decode is batch-invariant, as the pages' determinism claim asks).
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMV_VERSION 10000   /* 1.0.0 */

/* Block and element types. */
typedef enum {
    QMV_Q4_0 = 1,   /* 32 w, 18 B: fp16 d | 16 B nibbles;                 w = d*(q-8)            */
    QMV_Q5_0 = 2,   /* 32 w, 22 B: fp16 d | u32 5th bits | 16 B nibbles;  w = d*(q-16)           */
    QMV_Q8_0 = 3,   /* 32 w, 34 B: fp16 d | int8[32];                     w = d*q                */
    QMV_Q4_K = 4,   /* 256 w, 144 B: fp16 d | fp16 dmin | 12 B 6-bit sc/m | 128 B nibbles;
                                                                         w = d*sc*q - dmin*m    */
    QMV_Q6_K = 5,   /* 256 w, 210 B: 128 B low 4 bits | 64 B high 2 bits | int8 sc[16] | fp16 d;
                                                                         w = d*sc*(q-32)        */
    QMV_MXFP4 = 6,  /* 32 w, 17 B: E8M0 e | 16 B E2M1 codes;             w = 2^(e-127)*E2M1(q)  */
    QMV_Q8_K = 7,   /* activations only, 256 w, 292 B: fp32 d | int8[256] | int16 bsums[16]      */
    QMV_F32 = 8,    /* plain fp32 */
    QMV_BF16 = 9,   /* plain bfloat16 */
    QMV_MXFP4_R = 10, /* MXFP4 rows repacked by qmv_repack: the 16 code bytes of each 32-element
                        block in block order, then the row's E8M0 bytes, zero-padded to a
                        multiple of 16 bytes (row bytes = 16*ceil(17*cols/32/16)).  Weights of
                        qmv_moe_matvec with BF16 activations only. */
    QMV_Q4_1 = 11,  /* 32 w, 20 B: fp16 d | fp16 m | 16 B nibbles;      w = d*q + m            */
    QMV_Q5_1 = 12,  /* 32 w, 24 B: fp16 d | fp16 m | u32 5th bits | 16 B nibbles; w = d*q + m  */
    QMV_Q8_1 = 13,  /* 32 w, 36 B: fp16 d | fp16 s (block sum, unused by weights) | int8[32];
                                                                         w = d*q                */
    QMV_Q2_K = 14,  /* 256 w, 84 B: 16 B 4-bit sc|m per 16 | 64 B 2-bit codes | fp16 d | fp16 dmin;
                                                                         w = d*sc*q - dmin*m    */
    QMV_Q3_K = 15,  /* 256 w, 110 B: 32 B high bits | 64 B 2-bit codes | 12 B 6-bit scales | fp16 d;
                                                                         w = d*(s-32)*(q-4)     */
    QMV_Q5_K = 16,  /* 256 w, 176 B: Q4_K's d, dmin, 12 B sc/m | 32 B fifth bits | 128 B nibbles;
                                                                         w = d*sc*q - dmin*m    */
    QMV_F16 = 17,   /* plain IEEE half (weights) */
    QMV_MXFP8 = 18  /* activations only, 32 w, 33 B: E8M0 e | E4M3[32];  x = 2^(e-127)*E4M3(q)
                       (OCP Microscaling v1.0 MXFP8; see qmv_quantize_act) */
    /* QMV_F32 and QMV_BF16 are also accepted as plain weight types. */
} qmv_type;

/* A multiply's format is the weight type plus the activation type. */
#define QMV_FMT(wtype, atype) ((int)(wtype) | ((int)(atype) << 8))

/* Flags OR-ed into fmt.
 * QMV_FLAG_QUANTIZE_X: qmv_matvec with an 8-bit activation type (Q8_0/Q8_K)
 *   takes x as fp32 [n_vec][cols] (16-byte aligned) and quantises it inside the
 *   kernel, with results bit-identical to qmv_quantize_act followed by
 *   qmv_matvec (one launch instead of two).
 * QMV_FLAG_PDL: launch as a programmatic dependent of the kernel before it on
 *   the stream.  The kernel may start streaming W before that kernel has
 *   finished; it still waits for it before reading x or writing y (X, Y).
 *   Only for weights that the immediately preceding kernels do not write.
 *   Accepted by qmv_quantize_act, qmv_matvec and qmv_matmul. */
#define QMV_FLAG_QUANTIZE_X (1 << 16)
#define QMV_FLAG_PDL (1 << 17)

typedef enum {
    QMV_OK = 0,
    QMV_ERR_INVALID_ARG = -1,   /* null pointer, negative size                              */
    QMV_ERR_SHAPE = -2,         /* cols not a multiple of the block length, or over a limit */
    QMV_ERR_UNSUPPORTED = -3,   /* format / activation pair not provided                    */
    QMV_ERR_ALIGN = -4,         /* a pointer is not aligned as the call requires            */
    QMV_ERR_WORKSPACE = -5,     /* workspace missing or too small                           */
    QMV_ERR_CUDA = -6,          /* a CUDA call failed (the message has the CUDA string)     */
    QMV_ERR_DEVICE_STATUS = -7  /* a kernel reported a fault through the status word        */
} qmv_status;

/* Library version, QMV_VERSION of the build. */
int qmv_version(void);
/* Static text for a qmv_status code. */
const char* qmv_strerror(int err);
/* Detail of the last failed call on this host thread ("" if none). */
const char* qmv_last_error(void);

/* Block geometry: elements per block (32 or 256; 1 for F32/BF16; 0 if unknown),
 * bytes per block (17 for QMV_MXFP4_R, whose rows are padded), bytes of one row
 * of `cols` elements (0 if cols is not a multiple of the block length). */
int    qmv_block_elems(int type);
size_t qmv_block_bytes(int type);
size_t qmv_row_bytes(int type, int64_t cols);

/* ---------------------------------------------------------------------------
 * qmv_quantize_act -- fp32 activations to 8-bit blocks (the "A8" of W4A8;
 * "Architecture" page, "The package map", pkg/quant).
 *   fmt : QMV_Q8_0 (32-element blocks, fp16 scale, 34 B) or
 *         QMV_Q8_K (256-element blocks, fp32 scale, int16 sums of each run of
 *         16 codes, 292 B), optionally | QMV_FLAG_PDL.
 *   x   : n fp32 values, 4-byte aligned; several vectors may be laid end to end
 *         as long as each vector's length is a multiple of the block length.
 *   xq  : n/bs blocks out.
 *   n   : multiple of 32 (Q8_0) or 256 (Q8_K); 0 is a no-op.
 * Per block: amax = max|x|, d = amax/127, q = round-half-away(x * (1/d))
 * clamped to +-127 (q = 0 when amax = 0; when d is below 2^-128 and 1/d
 * overflows, q = round-half-away(x / d)); fp32 arithmetic, one rounding per
 * operation.  Q8_0 stores d rounded to fp16, Q8_K the fp32 d.
 *   fmt QMV_MXFP8 (x 16-byte aligned, n a multiple of 32, finite values):
 * the OCP Microscaling v1.0 conversion -- E = floor(log2 amax) - 8 (at least
 * -127; -127 for a block of zeros), stored as the E8M0 byte E + 127, and
 * q = E4M3(x / 2^E) rounded to nearest even, magnitudes clamped to 448.  The
 * MXFP8 mixture-of-experts path quantises its activations the same way.
 * ------------------------------------------------------------------------- */
int qmv_quantize_act(int fmt, const float* x, void* xq, int64_t n, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_quantize_weights -- fp32 or bf16 weights to the block formats the pages'
 * quantiser writes ("Models and formats", "Tensor formats": Q4_0/1, Q5_0/1,
 * Q8_0 and the K-quants).  The pages do not print the procedure; each format
 * takes one pass of min/max rules per run, no search:
 *   Q4_0 / Q5_0: m = the signed value of largest magnitude (the first on
 *     ties), d = m / -8 (Q4_0) or m / -16 (Q5_0), code = trunc(clamp(w / d +
 *     8.5, 0, 15)) (Q5_0: + 16.5, 0, 31).  The largest-magnitude weight
 *     decodes exactly to -8 fp16(d) (-16 for Q5_0).
 *   Q8_0: the symmetric 8-bit form, byte for byte qmv_quantize_act(QMV_Q8_0).
 *   Q4_1 / Q5_1: m = min, d = (max - m) / 15 (31), code = trunc(clamp((w -
 *     m) / d + 0.5, 0, 15 (31))).
 *   Q4_K / Q5_K: per 32-weight sub-block lo = min(0, min w), s = (max w - lo)
 *     / 15 (31), z = -lo; d = max s / 63, dmin = max z / 63; six-bit scales
 *     and mins round(s / d), round(z / dmin); codes round((w + dmin*m) /
 *     (d*sc)) on the stored fp16 scales.
 *   Q6_K: per 16-weight run the signed extreme e, s = e / -32; the s of
 *     largest magnitude s_e, d = s_e / -128; int8 scales round(s / d); codes
 *     round(w / (d*sc)) + 32.
 *   Each step is one fp32 rounding, divisions are multiplications by the
 *   fp32 reciprocal (the quotient when it overflows), ties round away from
 *   zero; fp16 values are stored rounded to nearest even.
 *   type : the block type, or QMV_FMT(block type, QMV_BF16) for bf16 weights
 *          (QMV_FMT(block type, QMV_F32) or the bare type: fp32).
 *   W    : rows x cols weights, 16-byte aligned; cols a multiple of 32 (256
 *          for the K-quants).
 *   out  : rows * qmv_row_bytes(block type, cols) bytes, 2-byte aligned, not
 *          overlapping W.
 * Returns QMV_ERR_UNSUPPORTED for other types, QMV_ERR_SHAPE, QMV_ERR_ALIGN,
 * QMV_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
int qmv_quantize_weights(int type, const void* W, int64_t rows, int64_t cols, void* out, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_repack -- weights to a layout for the tensor-core kernels, once at load
 * time (the "Architecture" page's bench transcript runs its engine with
 * "repack on").  The GGUF layout stays the canonical input; the repacked copy
 * holds the same bits.
 *   type : QMV_MXFP4 -> Wout in QMV_MXFP4_R rows: every 17-byte block's 16
 *          code bytes land 16-byte aligned and the row pitch becomes a
 *          multiple of 16, so TMA tensor copies can move the codes and the
 *          exponents of many rows at once.
 *   W    : rows x cols GGUF blocks (16-byte aligned; for stacked experts rows
 *          counts all of them, n_expert*rows).  Wout: rows x
 *          qmv_row_bytes(QMV_MXFP4_R, cols) bytes, 16-byte aligned, not
 *          overlapping W.  Asynchronous on `stream`; allocates nothing.
 * Returns QMV_OK, or QMV_ERR_UNSUPPORTED for other types, QMV_ERR_SHAPE,
 * QMV_ERR_ALIGN, QMV_ERR_INVALID_ARG, QMV_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int qmv_repack(int type, const void* W, int64_t rows, int64_t cols, void* Wout, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_dequantize -- weights to fp32 ("The package map", pkg/quant:
 * dequantisation).  out is rows x cols fp32, row-major.  Bit-exact: every
 * format's weight is an fp32 value, except Q4_K whose weight is the single
 * rounding of d*sc*q - dmin*m.
 * ------------------------------------------------------------------------- */
int qmv_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_block_dots -- the integers of the fused W4A8 dot product, exposed for
 * verification.  For weight block b of row r against activation block b of
 * vector v:
 *   out[((v*rows + r)*nb + b)*2 + 0] = S  = sum_i sub_scale_i * code_i * xq_i
 *   out[((v*rows + r)*nb + b)*2 + 1] = Mn = sum_i sub_min_i * xq_i  (Q4_K; else 0)
 * with code = q-8 (Q4_0), q-16 (Q5_0), q (Q8_0, Q4_K), q-32 (Q6_K), twice the
 * E2M1 value (MXFP4); sub_scale = the 6-bit (Q4_K) or int8 (Q6_K) sub-block
 * scale, else 1; sub_min = the Q4_K 6-bit min.  xq is Q8_0 for the 32-element
 * formats and Q8_K for Q4_K/Q6_K, [n_vec][cols/bs] blocks.  out is int32,
 * [n_vec][rows][cols/bs][2].  These are the same device routines the matvec
 * kernels use.
 * ------------------------------------------------------------------------- */
int qmv_block_dots(int type, const void* W, int64_t rows, int64_t cols,
                   const void* xq, int n_vec, int32_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_matvec -- decode: y[v][r] = sum_c w[r][c] * xhat[v][c] for n_vec
 * vectors sharing one pass over the weights ("The package map", pkg/tensor
 * MatVec; "A request, end to end": N sequences read the weights once).
 *   fmt : QMV_FMT(wtype, atype): the 32-element formats {Q4_0, Q4_1, Q5_0,
 *         Q5_1, Q8_0, Q8_1, MXFP4} with atype in {F32, Q8_0}; the K-quants
 *         {Q2_K, Q3_K, Q4_K, Q5_K, Q6_K} with atype in {F32, Q8_K}; the plain
 *         weights {F32, F16, BF16} with atype F32 (cols a multiple of 8);
 *         optionally | QMV_FLAG_QUANTIZE_X (8-bit atype only) | QMV_FLAG_PDL.
 *   x   : F32: fp32 [n_vec][cols], 16-byte aligned, xhat = x.
 *         Q8_0/Q8_K: [n_vec][cols/bs] blocks from qmv_quantize_act,
 *         4-byte aligned, xhat = d_x*q (the W4A8 product: integer dot per
 *         block, then the two scales, fp32 accumulation).
 *   y   : fp32 [n_vec][rows], overwritten.
 *   n_vec : 0..64 (0 is a no-op).
 * Accuracy: |y - exact| <= 1e-4 * sum_c |w*xhat| per output (in practice
 * ~1e-6).  Batch-invariant: row r of vector v is bit-identical whatever
 * n_vec is and whatever the other vectors hold.
 * ------------------------------------------------------------------------- */
int qmv_matvec(int fmt, const void* W, int64_t rows, int64_t cols,
               const void* x, float* y, int n_vec, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_matmul -- prefill: Y[m][r] = sum_c w[r][c] * xhat[m][c]
 * ("The package map", pkg/tensor MatMul; "The two phases": prefill is
 * arithmetic-bound).  Batched prefill must agree with sequential decode
 * ("The forward pass").
 *   fmt : QMV_FMT(QMV_Q4_K, QMV_BF16): X bf16 [m][cols]; the weights are
 *         dequantised to bf16 tiles (w rounded once from its fp32 value) and
 *         multiplied on the tensor cores with fp32 accumulation.  Rows much
 *         shorter than K (cols >= 8192, cols >= 2*rows, cols a multiple of
 *         512) run as two K halves on different SMs whose fp32 sums are added
 *         into Y after zeroing it (cudaMemsetAsync on the stream; two addends
 *         commute, so Y does not depend on which half lands first; the split
 *         follows the weight's shape, so a token's result does not depend
 *         on m).
 *         QMV_FMT(QMV_Q4_K, QMV_Q8_K): X Q8_K blocks [m][cols/256] (W4A8):
 *         per super-block the integers S = sum sc*q*xq and Mn = sum m*bsum
 *         come out of the tensor cores exactly (sm_103a has no tcgen05
 *         integer kind; sc*q, xq, m and the sums of 16 are integers that fp16
 *         holds exactly, so they run as fp16 operands with an fp32
 *         accumulator), then d_x*(d*S - dmin*Mn) is accumulated in fp32.
 *         Needs qmv_workspace_size(QMV_OP_MATMUL, fmt, rows, cols, m) bytes
 *         of workspace (qmv_set_workspace): the activation codes laid out as
 *         fp16, about m*cols*2.1 bytes; calls that share it must be ordered on
 *         one stream.  Agrees with the W4A8 decode of each token within the
 *         accuracy bar above.
 *         QMV_FMT(t, QMV_BF16) for every other weight type t (Q4_0, Q5_0,
 *         Q8_0, Q6_K, MXFP4, Q4_1, Q5_1, Q8_1, Q2_K, Q3_K, Q5_K and plain
 *         F32/F16/BF16 rows; not QMV_MXFP4_R): the same product, bf16(w)
 *         rounded once from w's fp32 value.  Q4_0, Q5_0, Q8_0 and Q6_K rows
 *         of a whole number of 16 bytes (cols a multiple of 256, or of 2048
 *         for Q6_K) are dequantised tile by tile into the tensor cores'
 *         operand memory inside the GEMM (with the same two-K-halves rule as
 *         Q4_K); BF16 rows are the operand as they are; the other types and
 *         row lengths (Q4_1, Q5_1, Q8_1, MXFP4, Q2_K, Q3_K, Q5_K, F32, F16,
 *         and e.g. Q8_0 with cols = 896) are converted to bf16 in the
 *         workspace first, which needs qmv_workspace_size(QMV_OP_MATMUL, fmt,
 *         rows, cols, m) bytes (rows*cols*2 rounded up to 256;
 *         QMV_ERR_WORKSPACE otherwise; calls that share it must be ordered on
 *         one stream).
 *         Any of these may be | QMV_FLAG_PDL (the W these kernels read must
 *         not be written by the kernels just before them on the stream).
 *   X   : 16-byte aligned.   Y : fp32 [m][rows], overwritten.
 *   m   : >= 0.
 * ------------------------------------------------------------------------- */
int qmv_matmul(int fmt, const void* W, int64_t rows, int64_t cols,
               const void* X, float* Y, int64_t m, void* stream);

/* ---------------------------------------------------------------------------
 * qmv_moe_matvec -- mixture of experts over a stacked 3-D weight tensor
 * W3d[n_expert][rows][cols] ("Models and formats", "Architectures": k of n
 * experts per token, stacked 3-D expert tensors, a bias on every expert
 * projection).  (token, slot) pairs are grouped by expert with a stable
 * counting sort so that each expert's weights are read once per call.
 *   ids   : int32 [n_tok][k], expert of each slot (0 <= id < n_expert; an id
 *           out of range sets the device status word and its slot is skipped).
 *   gates : NULL -> the up/gate form: x is [n_tok][cols], shared by the k
 *                   slots, and y[t][s][r] = (W[ids[t][s]] x_t)[r] + bias.
 *           non-NULL fp32 [n_tok][k] -> the down form: x is [n_tok][k][cols],
 *                   one input per slot, and
 *                   y[t][r] = sum_s gates[t][s] * ((W[ids[t][s]] x_{t,s})[r] + bias),
 *                   summed in slot order.
 *   bias  : fp32 [n_expert][rows], or NULL for none.
 *   fmt   : QMV_FMT(wtype, atype) with the pairs of qmv_matvec: activations
 *           F32 (fp32 rows, 16-byte aligned) or the paired 8-bit blocks (one
 *           block row per input vector, 4-byte aligned), optionally
 *           | QMV_FLAG_QUANTIZE_X (fp32 rows quantised inside the kernel);
 *           or, for MXFP4 experts only, BF16 (bf16 rows, 16-byte aligned):
 *           the grouped tensor-core GEMM, whose weights 2^(e-127)*E2M1 are
 *           exact in bf16 (fp32 accumulation; rows < 2^30); or MXFP8 (x fp32
 *           rows, 16-byte aligned, cols <= 4096): the activations are
 *           quantised to MXFP8 as qmv_quantize_act does, and the grouped GEMM
 *           runs on the block-scaled MMA (kind::mxf8f6f4): each MXFP4 code as
 *           E4M3 with its block's E8M0 exponent as the scale, against the
 *           tokens' E4M3 codes and scales, products exact, fp32 accumulation.
 *           The experts may also be given as QMV_MXFP4_R (qmv_repack output,
 *           same results), which the GEMM moves with TMA tensor copies.
 *   n_expert in 1..1024, k in 1..64, n_tok*k <= 2^24.
 *   Results per (token, slot) are, for F32 and 8-bit activations, those of
 *   qmv_matvec on that expert's matrix (same arithmetic and reduction
 *   order), plus the bias; with BF16 activations a token's result does not
 *   depend on the other tokens routed with it.  The down form's
 *   gate-weighted sum runs in fp32 in slot order.
 *   Workspace: qmv_workspace_size(QMV_OP_MOE, ...) bytes set by
 *           qmv_set_workspace(); calls that share the workspace must be
 *           ordered on one stream.
 * ------------------------------------------------------------------------- */
int qmv_moe_matvec(int fmt, const void* W3d, int n_expert, int64_t rows, int64_t cols,
                   const int32_t* ids, const float* gates, int k,
                   const void* x, float* y, int64_t n_tok, const float* bias,
                   void* stream);

/* ---------------------------------------------------------------------------
 * qmv_moe_matvec_noalloc -- qmv_moe_matvec for callers that cannot allocate
 * device memory.  (This entry point has no counterpart on the llamay pages;
 * it is a property of this library's interface.)
 *
 * Some callers can't call cudaMalloc or hand the library a buffer: a plugin
 * inside a host program that owns all device memory through its own pool, a
 * latency-critical loop where an allocation (which may synchronise the
 * device) is not allowed, or code that runs before the host's allocator
 * exists.  This call takes exactly the arguments of qmv_moe_matvec and gives
 * the same results, but its scratch (the expert grouping and the per-slot
 * outputs) lives in a fixed array inside the library's device image instead
 * of a registered workspace.  It allocates nothing and needs no
 * qmv_set_workspace().
 *   Limit: the scratch holds QMV_MOE_NOALLOC_MAX_BYTES (4 MiB); a call needs
 *   qmv_workspace_size(QMV_OP_MOE, fmt, rows, cols, n_tok*k) bytes (about
 *   n_tok*k*rows*4), and a larger one is refused with QMV_ERR_SHAPE.  Every
 *   GPU that loads the library holds these 4 MiB until the process exits.
 *   Set-up: the first call on each device looks up the array's device address
 *   (with that device current); make that first call before any stream
 *   capture.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents (each call overwrites what it reads, so nothing needs clearing).
 *   Calls that can overlap on the GPU -- on different streams, or from
 *   different host threads -- race on the array; order them on one stream.
 * ------------------------------------------------------------------------- */
#define QMV_MOE_NOALLOC_MAX_BYTES ((size_t)4 << 20)
int qmv_moe_matvec_noalloc(int fmt, const void* W3d, int n_expert, int64_t rows, int64_t cols,
                           const int32_t* ids, const float* gates, int k,
                           const void* x, float* y, int64_t n_tok, const float* bias,
                           void* stream);

/* ---------------------------------------------------------------------------
 * qmv_moe_block -- a whole mixture-of-experts block for fp32 hidden states:
 * router -> top k -> gate_up -> clipped SwiGLU -> down, gate-weighted
 * ("Models and formats", "Architectures": a router picks k of n experts per
 * token; stacked 3-D expert tensors; gpt-oss gates with a clipped SwiGLU
 * whose linear half is offset by one and has a bias on every expert
 * projection).  The pages print neither the router's arithmetic nor the
 * clipping constants; this call fixes them as follows.
 *   Router : logit[t][e] = x_t . Wr[e] + br[e] in fp32, summed as 32 partial
 *            sums (partial l takes the elements l, l+32, ... by fused
 *            multiply-add from 0) combined by a butterfly (l + (l xor o),
 *            o = 16, 8, 4, 2, 1), then the bias: the top-k choice depends on
 *            this order only, not on the GPU.
 *   Top k  : the k largest logits, ties to the lower expert id; ids[t][0]
 *            is the largest.  Gates: softmax over the k kept logits in fp32
 *            (exp(l_s - l_0), summed in slot order).  If a logit is NaN the
 *            chosen ids are unspecified (but distinct and in range).
 *   gate_up: W_gu [n_expert][2*inter][hidden]; rows [0, inter) are the gate
 *            half g, rows [inter, 2*inter) the linear half u; b_gu
 *            [n_expert][2*inter] or NULL.
 *   Gate   : h = min(g, limit) * sigmoid(alpha * min(g, limit))
 *                * (clamp(u, -limit, limit) + 1), fp32.
 *   down   : W_down [n_expert][hidden][inter], b_down [n_expert][hidden] or
 *            NULL; y[t] = sum over slots, in slot order, of
 *            gates[t][s] * (W_down[ids[t][s]] h_{t,s} + b_down[ids[t][s]]).
 *   fmt    : QMV_FMT(wtype, atype): atype F32 (fp32 activations), the paired
 *            8-bit type (x and h are quantised to it inside the expert
 *            kernels, as QMV_FLAG_QUANTIZE_X does), or, for MXFP4 / MXFP4_R
 *            experts, BF16 (x and h rounded to bf16, the grouped tensor-core
 *            GEMM) or MXFP8 (x and h quantised to MXFP8, the block-scaled
 *            GEMM; hidden, inter <= 4096).  No flags.  Each projection gives
 *            the results of qmv_moe_matvec with the same format.
 *   Wr     : fp32 [n_expert][hidden]; br fp32 [n_expert] or NULL.
 *   x      : fp32 [n_tok][hidden], 16-byte aligned.  y : fp32 [n_tok][hidden].
 *   ids    : int32 [n_tok][k] out.   gates : fp32 [n_tok][k] out.
 *   n_expert in 1..1024, k in 1..min(64, n_expert), n_tok*k <= 2^24; hidden
 *   and inter multiples of the weight block length.
 *   Workspace: qmv_moe_block_workspace_size(...) bytes set by
 *   qmv_set_workspace(); calls that share it must be ordered on one stream.
 * ------------------------------------------------------------------------- */
int qmv_moe_block(int fmt, int n_expert, int k, int64_t hidden, int64_t inter,
                  const float* Wr, const float* br,
                  const void* W_gu, const float* b_gu,
                  const void* W_down, const float* b_down,
                  float alpha, float limit,
                  const float* x, int64_t n_tok, float* y,
                  int32_t* ids, float* gates, void* stream);
/* Bytes of workspace qmv_moe_block needs (about n_tok*(n_expert + 3*k*inter)*4
 * plus the expert calls' grouping and slot outputs); 0 for empty sizes. */
size_t qmv_moe_block_workspace_size(int fmt, int n_expert, int k, int64_t hidden, int64_t inter,
                                    int64_t n_tok);

/* Workspace for the calls that need scratch. */
enum { QMV_OP_MATVEC = 1, QMV_OP_MATMUL = 2, QMV_OP_MOE = 3 };
/* Bytes of workspace `op` needs for these sizes.  QMV_OP_MOE, n = n_tok*k:
 * the grouping, 2050 + n ints, and n*rows fp32 slot outputs; with BF16
 * activations also the GEMM's slot list, about 2n ints, and the n packed
 * bf16 activation rows, n*cols*2 bytes.  QMV_OP_MATMUL with
 * QMV_FMT(QMV_Q4_K, QMV_Q8_K), n = m tokens: the fp16 activation codes
 * (m*cols*2), sums of 16 (m*cols/8) and scales (about m*cols/64 bytes).
 * QMV_OP_MATMUL with QMV_FMT(t, QMV_BF16) converted in two passes (see
 * qmv_matmul): the bf16 weights, rows*cols*2 bytes rounded up to 256.  0 if
 * the call needs none. */
size_t qmv_workspace_size(int op, int fmt, int64_t rows, int64_t cols, int64_t n);
/* Register a caller-owned device buffer (256-byte aligned) as the workspace of
 * the current device; NULL/0 clears it.  The library keeps the pointer only. */
int qmv_set_workspace(void* ptr, size_t bytes);

/* Diagnostics: limit the bounded pipeline waits of the decode and expert
 * matvec kernels (qmv_matvec, qmv_moe_matvec and the block's projections with
 * F32 or 8-bit activations) launched afterwards on the current device to `ns`
 * nanoseconds; 0 restores the default of 2 s.  A limit under 1 ms polls without
 * blocking, so a wait that has to wait at all gives up: it sets the status
 * word's wait-timeout bit and its kernel stops early -- its outputs are then
 * incomplete -- after letting its own copies in flight land.  For exercising
 * that path in tests; calls launched while a short limit is set fail on
 * purpose.  Host-side setting, read when a call launches its kernels. */
int qmv_set_wait_limit(unsigned ns);

/* Synchronise `stream`, read and clear the device status word of the current
 * device.  Returns QMV_OK, or QMV_ERR_DEVICE_STATUS with qmv_last_error()
 * describing the fault, or QMV_ERR_CUDA. */
int qmv_get_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
