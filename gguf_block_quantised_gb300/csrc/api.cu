// api.cu -- the extern "C" boundary of libqmv (declared in include/qmv.h).
//
// Every entry point validates its arguments on the host, returns a negative
// qmv_status without launching anything when they are wrong, and otherwise
// only enqueues kernels on the caller's stream.  Unsupported input is refused
// with a message naming what is supported ("Models and formats" page: anything
// outside the supported set "is refused at load with a message naming what
// does work"; "Tensor formats": rows that are not a multiple of 256 cannot be
// K-quants).  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "runtime.cuh"

// Launchers defined in the kernel translation units.
int qmv_launch_quantize(int atype, const float* x, void* xq, int64_t n, bool pdl, cudaStream_t st);
int qmv_launch_dequant(int t, const void* W, int64_t rows, int64_t cols, float* out, cudaStream_t st);
int qmv_launch_quantize_weights(int wtype, bool bf16, const void* W, int64_t n, void* out, cudaStream_t st);
int qmv_launch_block_dots(int t, const void* W, int64_t rows, int64_t cols, const void* xq, int n_vec,
                          int32_t* out, cudaStream_t st);
#define QMV_GEMV_DECL(NAME) \
    int NAME(bool a8, bool quant_x, bool pdl, const void*, int64_t, int64_t, const void*, float*, int, cudaStream_t);
QMV_GEMV_DECL(qmv_gemv_q4_0)
QMV_GEMV_DECL(qmv_gemv_q5_0)
QMV_GEMV_DECL(qmv_gemv_q8_0)
QMV_GEMV_DECL(qmv_gemv_mxfp4)
QMV_GEMV_DECL(qmv_gemv_q4_k)
QMV_GEMV_DECL(qmv_gemv_q6_k)
QMV_GEMV_DECL(qmv_gemv_q4_1)
QMV_GEMV_DECL(qmv_gemv_q5_1)
QMV_GEMV_DECL(qmv_gemv_q8_1)
QMV_GEMV_DECL(qmv_gemv_q2_k)
QMV_GEMV_DECL(qmv_gemv_q3_k)
QMV_GEMV_DECL(qmv_gemv_q5_k)
QMV_GEMV_DECL(qmv_gemv_f32)
QMV_GEMV_DECL(qmv_gemv_f16)
QMV_GEMV_DECL(qmv_gemv_bf16)
size_t qmv_w4a8_workspace_bytes(int64_t cols, int64_t m);
size_t qmv_bf16_gemm_workspace_bytes(int64_t rows, int64_t cols);
int qmv_launch_gemm_two_pass_bf16(int t, const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                               void* ws, bool pdl, cudaStream_t st);
int qmv_launch_gemm_deq_bf16(int t, const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                             bool pdl, cudaStream_t st);
int qmv_launch_gemm_q4k_w4a8(const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m,
                             void* ws, bool pdl, cudaStream_t st);
size_t qmv_moe_workspace_bytes(bool bf16, int64_t rows, int64_t cols, int64_t n_pairs, bool mx);
size_t qmv_moe_block_workspace_bytes(bool bf16, bool mx, int n_expert, int64_t hidden, int64_t inter, int64_t n_tok,
                                     int k);
int qmv_launch_moe_block(int wtype, bool a8, bool bf16, bool mx, size_t act_block_bytes, int n_expert, int k,
                         int64_t hidden, int64_t inter, const float* Wr, const float* br, const void* Wgu,
                         const float* bgu, const void* Wd, const float* bd, float alpha, float limit, const float* x,
                         int64_t n_tok, float* y, int32_t* ids, float* gates, void* ws, cudaStream_t st);
int qmv_launch_repack_mxfp4(const void* W, int64_t rows, int64_t cols, void* Wout, cudaStream_t st);
int qmv_launch_moe_ex(int wtype, bool a8, bool quant_x, bool bf16, bool mx, size_t act_block_bytes,
                      const void* W3d, int n_expert, int64_t rows, int64_t cols, const int32_t* ids,
                      const float* gates, int k, const void* x, float* y, int64_t n_tok, const float* bias, void* ws,
                      bool grouped, cudaStream_t st);
int qmv_launch_gemm_q4k_bf16(const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m, bool pdl,
                             cudaStream_t st);

// The device status word: kernels OR fault bits into it (QMV_DEV_*).
__device__ unsigned g_qmv_status;

// Built-in scratch of qmv_moe_matvec_noalloc: a fixed array in the library's
// device image, present on every GPU that loads the library until the process
// exits.  Host code must not use this name as an address; see
// moe_noalloc_scratch() below.
static __device__ __align__(256) uint8_t g_moe_noalloc_scratch[QMV_MOE_NOALLOC_MAX_BYTES];

namespace qmv {

unsigned* status_word()
{
    static std::atomic<unsigned*> cache[kMaxDevices];
    const int d = current_device();
    unsigned* p = (d >= 0 && d < kMaxDevices) ? cache[d].load(std::memory_order_acquire) : nullptr;
    if (!p) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_qmv_status) != cudaSuccess) return nullptr;
        p = static_cast<unsigned*>(a);
        if (d >= 0 && d < kMaxDevices) cache[d].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace qmv

namespace {

thread_local std::string t_err;

int fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return code;
}

int ok()
{
    t_err.clear();
    return QMV_OK;
}

// Weight types whose rows the bf16 dequantising pass reads (the GGUF block
// types and the plain F32/F16/BF16 rows; not the repacked QMV_MXFP4_R rows).
bool dequant_type(int t)
{
    switch (t) {
    case QMV_Q4_0: case QMV_Q5_0: case QMV_Q8_0: case QMV_MXFP4: case QMV_Q4_K: case QMV_Q6_K:
    case QMV_Q4_1: case QMV_Q5_1: case QMV_Q8_1: case QMV_Q2_K: case QMV_Q3_K: case QMV_Q5_K:
    case QMV_F32: case QMV_F16: case QMV_BF16:
        return true;
    default: return false;
    }
}

// Block types and row lengths whose prefill GEMM dequantises tiles into TMEM
// itself (besides Q4_K's own kernel): the raw tiles are TMA boxes, which need
// rows of a whole number of 16 bytes.
bool fused_tile(int t, int64_t cols)
{
    if (t != QMV_Q4_0 && t != QMV_Q5_0 && t != QMV_Q8_0 && t != QMV_Q6_K) return false;
    const int64_t bs = qmv_block_elems(t);
    return cols > 0 && cols % bs == 0 && (cols / bs) * (int64_t)qmv_block_bytes(t) % 16 == 0;
}

const char* type_name(int t)
{
    switch (t) {
    case QMV_Q4_0: return "Q4_0";
    case QMV_Q5_0: return "Q5_0";
    case QMV_Q8_0: return "Q8_0";
    case QMV_Q4_K: return "Q4_K";
    case QMV_Q6_K: return "Q6_K";
    case QMV_MXFP4: return "MXFP4";
    case QMV_Q8_K: return "Q8_K";
    case QMV_F32: return "F32";
    case QMV_BF16: return "BF16";
    case QMV_MXFP4_R: return "MXFP4_R";
    case QMV_Q4_1: return "Q4_1";
    case QMV_Q5_1: return "Q5_1";
    case QMV_Q8_1: return "Q8_1";
    case QMV_Q2_K: return "Q2_K";
    case QMV_Q3_K: return "Q3_K";
    case QMV_Q5_K: return "Q5_K";
    case QMV_F16: return "F16";
    case QMV_MXFP8: return "MXFP8";
    default: return "unknown";
    }
}

bool is_plain(int t) { return t == QMV_F32 || t == QMV_F16 || t == QMV_BF16; }

bool is_weight_type(int t)
{
    return t == QMV_Q4_0 || t == QMV_Q5_0 || t == QMV_Q8_0 || t == QMV_MXFP4 || t == QMV_Q4_K || t == QMV_Q6_K ||
           t == QMV_Q4_1 || t == QMV_Q5_1 || t == QMV_Q8_1 || t == QMV_Q2_K || t == QMV_Q3_K || t == QMV_Q5_K ||
           is_plain(t);
}

bool is_kquant(int t) { return qmv::kq_rt(t); }

// The 8-bit activation type a block format pairs with (plain weights: none, F32 only).
int paired_act(int wtype) { return is_plain(wtype) ? QMV_F32 : is_kquant(wtype) ? QMV_Q8_K : QMV_Q8_0; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

const char* kWeightList =
    "Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q8_1, MXFP4 (32-element blocks), Q2_K, Q3_K, Q4_K, Q5_K, Q6_K (256-element "
    "blocks) and plain F32, F16, BF16";

int check_weights(int wtype, const void* W, int64_t rows, int64_t cols)
{
    if (!is_weight_type(wtype))
        return fail(QMV_ERR_UNSUPPORTED, "weight type %d (%s) is not supported; supported: %s", wtype,
                    type_name(wtype), kWeightList);
    if (rows < 0 || cols <= 0) return fail(QMV_ERR_INVALID_ARG, "rows must be >= 0 and cols > 0 (got %lld x %lld)",
                                           (long long)rows, (long long)cols);
    const int bs = is_plain(wtype) ? 8 : qmv_block_elems(wtype);
    if (cols % bs)
        return fail(QMV_ERR_SHAPE,
                    "%s rows hold %d-element %s; cols = %lld is not a multiple of %d%s", type_name(wtype), bs,
                    is_plain(wtype) ? "units" : "blocks", (long long)cols, bs,
                    is_kquant(wtype) ? " (rows whose length is not a multiple of 256 are stored as Q4_0/Q5_0/Q8_0)"
                                     : "");
    if (cols > (int64_t)1 << 24) return fail(QMV_ERR_SHAPE, "cols = %lld is over the limit of 16777216", (long long)cols);
    if (rows > 0 && !W) return fail(QMV_ERR_INVALID_ARG, "W is NULL");
    if (W && !aligned(W, 16)) return fail(QMV_ERR_ALIGN, "W must start on a 16-byte boundary");
    return QMV_OK;
}

int cuda_fail(const char* where)
{
    const cudaError_t e = cudaGetLastError();
    return fail(QMV_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
Workspace g_ws[qmv::kMaxDevices];

// What the argument checks of the MoE calls settle.
struct MoeCall {
    int wtype = 0;
    bool a8 = false, quant_x = false, bf16 = false, mx = false;
    bool empty = false;   // nothing to compute: return QMV_OK
    size_t need = 0;      // bytes of scratch
};

// The checks both MoE entry points share.  Activations: F32, the paired 8-bit
// blocks (optionally quantised in-kernel), or -- MXFP4 experts only -- BF16
// rows for the grouped tensor-core GEMM.
int moe_check(const char* name, int fmt, const void* W3d, int n_expert, int64_t rows, int64_t cols,
              const int32_t* ids, const float* gates, int k, const void* x, float* y, int64_t n_tok,
              const float* bias, MoeCall& c)
{
    if (fmt & ~(0xffff | QMV_FLAG_QUANTIZE_X)) return fail(QMV_ERR_INVALID_ARG, "unknown flags 0x%x", fmt & ~0xffff);
    c.quant_x = (fmt & QMV_FLAG_QUANTIZE_X) != 0;
    c.wtype = fmt & 0xff;
    const int atype = (fmt >> 8) & 0xff;
    c.bf16 = atype == QMV_BF16 && (c.wtype == QMV_MXFP4 || c.wtype == QMV_MXFP4_R);
    c.mx = atype == QMV_MXFP8 && (c.wtype == QMV_MXFP4 || c.wtype == QMV_MXFP4_R);
    if (c.wtype == QMV_MXFP4_R && !c.bf16 && !c.mx)
        return fail(QMV_ERR_UNSUPPORTED, "%s: repacked MXFP4_R experts take BF16 or MXFP8 activations (got %s)", name,
                    type_name(atype));
    if (is_weight_type(c.wtype) && atype != QMV_F32 && atype != paired_act(c.wtype) && !c.bf16 && !c.mx)
        return fail(QMV_ERR_UNSUPPORTED, "%s: %s experts take F32 or %s activations%s (got %s)", name,
                    type_name(c.wtype), type_name(paired_act(c.wtype)),
                    c.wtype == QMV_MXFP4 ? ", BF16 or MXFP8" : "", type_name(atype));
    // MXFP4_R has the MXFP4 block geometry (padded rows)
    int rc = check_weights(c.wtype == QMV_MXFP4_R ? QMV_MXFP4 : c.wtype, W3d, rows, cols);
    if (rc) return rc;
    if (c.quant_x && (atype == QMV_F32 || c.bf16 || c.mx))
        return fail(QMV_ERR_INVALID_ARG, "QMV_FLAG_QUANTIZE_X needs an 8-bit activation type (Q8_0 or Q8_K)");
    if (n_expert < 1 || n_expert > 1024) return fail(QMV_ERR_INVALID_ARG, "n_expert must be in 1..1024 (got %d)", n_expert);
    if (k < 1 || k > 64) return fail(QMV_ERR_INVALID_ARG, "k must be in 1..64 (got %d)", k);
    if (n_tok < 0 || n_tok > ((int64_t)1 << 24) / k)   // range first: n_tok * k must not overflow
        return fail(QMV_ERR_INVALID_ARG, "n_tok must be >= 0 with n_tok*k <= 16777216");
    if ((c.bf16 || c.mx) && rows > (int64_t)1 << 30) return fail(QMV_ERR_SHAPE, "rows must be below 2^30");
    if (c.mx && cols > 4096)
        return fail(QMV_ERR_SHAPE, "%s: MXFP8 activations take cols <= 4096 (got %lld)", name, (long long)cols);
    c.empty = n_tok == 0 || rows == 0;
    if (c.empty) return QMV_OK;
    if (!ids || !x || !y) return fail(QMV_ERR_INVALID_ARG, "ids, x and y must not be NULL");
    c.a8 = atype != QMV_F32 && !c.bf16 && !c.mx;
    const int xal = (c.a8 && !c.quant_x) ? 4 : 16;
    if (!aligned(x, xal)) return fail(QMV_ERR_ALIGN, "x must be %d-byte aligned", xal);
    if (!aligned(ids, 4) || !aligned(y, 4) || (gates && !aligned(gates, 4)) || (bias && !aligned(bias, 4)))
        return fail(QMV_ERR_ALIGN, "ids, gates, bias and y must be 4-byte aligned");
    c.need = qmv_moe_workspace_bytes(c.bf16, rows, cols, n_tok * k, c.mx);
    return QMV_OK;
}

int moe_run(const char* name, const MoeCall& c, const void* W3d, int n_expert, int64_t rows, int64_t cols,
            const int32_t* ids, const float* gates, int k, const void* x, float* y, int64_t n_tok, const float* bias,
            void* ws, void* stream)
{
    if (!qmv::status_word()) return cuda_fail(name);
    const int rc = qmv_launch_moe_ex(c.wtype, c.a8, c.quant_x, c.bf16, c.mx, qmv_block_bytes(paired_act(c.wtype)),
                                     W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias, ws, false,
                                     static_cast<cudaStream_t>(stream));
    if (rc == -2) return fail(QMV_ERR_SHAPE, "cols = %lld needs more shared memory than one SM has", (long long)cols);
    if (rc == -8) return fail(QMV_ERR_CUDA, "%s: could not build a TMA tensor map", name);
    if (rc) return cuda_fail(name);
    return ok();
}

}  // namespace

extern "C" {

int qmv_version(void) { return QMV_VERSION; }

const char* qmv_strerror(int err)
{
    switch (err) {
    case QMV_OK: return "ok";
    case QMV_ERR_INVALID_ARG: return "invalid argument";
    case QMV_ERR_SHAPE: return "unsupported shape";
    case QMV_ERR_UNSUPPORTED: return "unsupported format";
    case QMV_ERR_ALIGN: return "misaligned pointer";
    case QMV_ERR_WORKSPACE: return "workspace missing or too small";
    case QMV_ERR_CUDA: return "CUDA error";
    case QMV_ERR_DEVICE_STATUS: return "fault reported by a kernel";
    default: return "unknown error";
    }
}

const char* qmv_last_error(void) { return t_err.c_str(); }

int qmv_block_elems(int type)
{
    switch (type) {
    case QMV_Q4_0: case QMV_Q5_0: case QMV_Q8_0: case QMV_MXFP4: case QMV_MXFP4_R: case QMV_Q4_1: case QMV_Q5_1:
    case QMV_Q8_1: case QMV_MXFP8: return 32;
    case QMV_Q4_K: case QMV_Q6_K: case QMV_Q8_K: case QMV_Q2_K: case QMV_Q3_K: case QMV_Q5_K: return 256;
    case QMV_F32: case QMV_BF16: case QMV_F16: return 1;
    default: return 0;
    }
}

size_t qmv_block_bytes(int type)
{
    switch (type) {
    case QMV_Q4_0: return 18;
    case QMV_Q5_0: return 22;
    case QMV_Q8_0: return 34;
    case QMV_MXFP4: case QMV_MXFP4_R: return 17;
    case QMV_MXFP8: return 33;
    case QMV_Q4_K: return 144;
    case QMV_Q6_K: return 210;
    case QMV_Q8_K: return 292;
    case QMV_Q4_1: return 20;
    case QMV_Q5_1: return 24;
    case QMV_Q8_1: return 36;
    case QMV_Q2_K: return 84;
    case QMV_Q3_K: return 110;
    case QMV_Q5_K: return 176;
    case QMV_F32: return 4;
    case QMV_BF16: case QMV_F16: return 2;
    default: return 0;
    }
}

size_t qmv_row_bytes(int type, int64_t cols)
{
    const int bs = qmv_block_elems(type);
    if (bs == 0 || cols < 0 || cols % bs) return 0;
    if (type == QMV_MXFP4_R) return ((size_t)(cols / 32) * 17 + 15) & ~size_t(15);   // padded rows
    return (size_t)(cols / bs) * qmv_block_bytes(type);
}

int qmv_quantize_act(int fmt, const float* x, void* xq, int64_t n, void* stream)
{
    const bool pdl = (fmt & QMV_FLAG_PDL) != 0;
    if (fmt & ~(0xffff | QMV_FLAG_PDL)) return fail(QMV_ERR_INVALID_ARG, "unknown flags 0x%x", fmt & ~0xffff);
    fmt &= 0xffff;
    if (fmt != QMV_Q8_0 && fmt != QMV_Q8_K && fmt != QMV_MXFP8)
        return fail(QMV_ERR_UNSUPPORTED, "activation format %d (%s) is not supported; supported: Q8_0, Q8_K, MXFP8",
                    fmt, type_name(fmt));
    const int bs = qmv_block_elems(fmt);
    if (n < 0) return fail(QMV_ERR_INVALID_ARG, "n must be >= 0");
    if (n % bs) return fail(QMV_ERR_SHAPE, "%s quantises %d-element blocks; n = %lld is not a multiple of %d",
                            type_name(fmt), bs, (long long)n, bs);
    if (n == 0) return ok();
    if (!x || !xq) return fail(QMV_ERR_INVALID_ARG, "x and xq must not be NULL");
    const int xal = fmt == QMV_Q8_0 ? 4 : 16, qal = fmt == QMV_Q8_K ? 4 : fmt == QMV_Q8_0 ? 2 : 1;
    if (!aligned(x, xal)) return fail(QMV_ERR_ALIGN, "x must be %d-byte aligned", xal);
    if (!aligned(xq, qal)) return fail(QMV_ERR_ALIGN, "xq must be %d-byte aligned", qal);
    if (qmv_launch_quantize(fmt, x, xq, n, pdl, static_cast<cudaStream_t>(stream))) return cuda_fail("qmv_quantize_act");
    return ok();
}

int qmv_quantize_weights(int type, const void* W, int64_t rows, int64_t cols, void* out, void* stream)
{
    const int wtype = type & 0xff, in = (type >> 8) & 0xff;
    if (type & ~0xffff) return fail(QMV_ERR_INVALID_ARG, "unknown flags 0x%x", type & ~0xffff);
    if (in != 0 && in != QMV_F32 && in != QMV_BF16)
        return fail(QMV_ERR_UNSUPPORTED, "qmv_quantize_weights reads F32 or BF16 weights (got %s)", type_name(in));
    const bool bf16 = in == QMV_BF16;
    if (wtype != QMV_Q4_0 && wtype != QMV_Q4_1 && wtype != QMV_Q5_0 && wtype != QMV_Q5_1 && wtype != QMV_Q8_0 &&
        wtype != QMV_Q4_K && wtype != QMV_Q5_K && wtype != QMV_Q6_K)
        return fail(QMV_ERR_UNSUPPORTED,
                    "qmv_quantize_weights writes Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K and Q6_K (got %s)",
                    type_name(wtype));
    if (rows < 0 || cols <= 0) return fail(QMV_ERR_INVALID_ARG, "rows must be >= 0 and cols > 0 (got %lld x %lld)",
                                           (long long)rows, (long long)cols);
    const int bs = qmv_block_elems(wtype);
    if (cols % bs)
        return fail(QMV_ERR_SHAPE, "%s rows hold %d-element blocks; cols = %lld is not a multiple of %d",
                    type_name(wtype), bs, (long long)cols, bs);
    if (rows == 0) return ok();
    if (rows > ((int64_t)1 << 40) / cols) return fail(QMV_ERR_SHAPE, "rows * cols must be below 2^40");
    if (!W || !out) return fail(QMV_ERR_INVALID_ARG, "W and out must not be NULL");
    if (!aligned(W, 16)) return fail(QMV_ERR_ALIGN, "W must be 16-byte aligned");
    if (!aligned(out, 2)) return fail(QMV_ERR_ALIGN, "out must be 2-byte aligned");
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(W), a1 = a0 + (uintptr_t)(rows * cols) * (bf16 ? 2 : 4);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(out), b1 = b0 + (uintptr_t)rows * qmv_row_bytes(wtype, cols);
    if (a0 < b1 && b0 < a1) return fail(QMV_ERR_INVALID_ARG, "qmv_quantize_weights: out overlaps W");
    if (qmv_launch_quantize_weights(wtype, bf16, W, rows * cols, out, static_cast<cudaStream_t>(stream)))
        return cuda_fail("qmv_quantize_weights");
    return ok();
}

int qmv_repack(int type, const void* W, int64_t rows, int64_t cols, void* Wout, void* stream)
{
    if (type != QMV_MXFP4)
        return fail(QMV_ERR_UNSUPPORTED, "qmv_repack: %s weights have no repacked layout; supported: MXFP4 (-> MXFP4_R)",
                    type_name(type));
    int rc = check_weights(type, W, rows, cols);
    if (rc) return rc;
    if (rows == 0) return ok();
    if (!Wout) return fail(QMV_ERR_INVALID_ARG, "Wout must not be NULL");
    if (!aligned(Wout, 16)) return fail(QMV_ERR_ALIGN, "Wout must start on a 16-byte boundary");
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(W), a1 = a0 + (uintptr_t)rows * qmv_row_bytes(type, cols);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(Wout), b1 = b0 + (uintptr_t)rows * qmv_row_bytes(QMV_MXFP4_R, cols);
    if (a0 < b1 && b0 < a1) return fail(QMV_ERR_INVALID_ARG, "qmv_repack: Wout overlaps W");
    if (qmv_launch_repack_mxfp4(W, rows, cols, Wout, static_cast<cudaStream_t>(stream))) return cuda_fail("qmv_repack");
    return ok();
}

int qmv_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out, void* stream)
{
    int rc = check_weights(type, W, rows, cols);
    if (rc) return rc;
    if (rows == 0) return ok();
    if (!out) return fail(QMV_ERR_INVALID_ARG, "out is NULL");
    if (qmv_launch_dequant(type, W, rows, cols, out, static_cast<cudaStream_t>(stream))) return cuda_fail("qmv_dequantize");
    return ok();
}

int qmv_block_dots(int type, const void* W, int64_t rows, int64_t cols, const void* xq, int n_vec, int32_t* out,
                   void* stream)
{
    int rc = check_weights(type, W, rows, cols);
    if (rc) return rc;
    if (is_plain(type))
        return fail(QMV_ERR_UNSUPPORTED, "qmv_block_dots: %s weights have no integer block dots (block formats only)",
                    type_name(type));
    if (n_vec < 0) return fail(QMV_ERR_INVALID_ARG, "n_vec must be >= 0");
    if (rows == 0 || n_vec == 0) return ok();
    if (!xq || !out) return fail(QMV_ERR_INVALID_ARG, "xq and out must not be NULL");
    if (qmv_launch_block_dots(type, W, rows, cols, xq, n_vec, out, static_cast<cudaStream_t>(stream)))
        return cuda_fail("qmv_block_dots");
    return ok();
}

int qmv_matvec(int fmt, const void* W, int64_t rows, int64_t cols, const void* x, float* y, int n_vec, void* stream)
{
    if (fmt & ~(0xffff | QMV_FLAG_QUANTIZE_X | QMV_FLAG_PDL))
        return fail(QMV_ERR_INVALID_ARG, "unknown flags 0x%x", fmt & ~0xffff);
    const bool quant_x = (fmt & QMV_FLAG_QUANTIZE_X) != 0, pdl = (fmt & QMV_FLAG_PDL) != 0;
    const int wtype = fmt & 0xff, atype = (fmt >> 8) & 0xff;
    if (atype != QMV_F32 && atype != paired_act(wtype) && is_weight_type(wtype))
        return fail(QMV_ERR_UNSUPPORTED,
                    "%s weights take F32 or %s activations in qmv_matvec (got %s); 32-element formats pair with "
                    "Q8_0, K-quants with Q8_K",
                    type_name(wtype), type_name(paired_act(wtype)), type_name(atype));
    int rc = check_weights(wtype, W, rows, cols);
    if (rc) return rc;
    if (quant_x && atype == QMV_F32)
        return fail(QMV_ERR_INVALID_ARG, "QMV_FLAG_QUANTIZE_X needs an 8-bit activation type (Q8_0 or Q8_K)");
    if (n_vec < 0 || n_vec > 64) return fail(QMV_ERR_INVALID_ARG, "n_vec must be in 0..64 (got %d)", n_vec);
    if (rows == 0 || n_vec == 0) return ok();
    if (!x || !y) return fail(QMV_ERR_INVALID_ARG, "x and y must not be NULL");
    const bool a8 = atype != QMV_F32;
    const int xal = (a8 && !quant_x) ? 4 : 16;
    if (!aligned(x, xal)) return fail(QMV_ERR_ALIGN, "x must be %d-byte aligned", xal);
    if (!aligned(y, 4)) return fail(QMV_ERR_ALIGN, "y must be 4-byte aligned");
    if (!qmv::status_word()) return cuda_fail("qmv_matvec (status word)");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (wtype) {
    case QMV_Q4_0: rc = qmv_gemv_q4_0(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q5_0: rc = qmv_gemv_q5_0(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q8_0: rc = qmv_gemv_q8_0(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_MXFP4: rc = qmv_gemv_mxfp4(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q4_K: rc = qmv_gemv_q4_k(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q6_K: rc = qmv_gemv_q6_k(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q4_1: rc = qmv_gemv_q4_1(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q5_1: rc = qmv_gemv_q5_1(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q8_1: rc = qmv_gemv_q8_1(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q2_K: rc = qmv_gemv_q2_k(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q3_K: rc = qmv_gemv_q3_k(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_Q5_K: rc = qmv_gemv_q5_k(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_F32: rc = qmv_gemv_f32(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_F16: rc = qmv_gemv_f16(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    case QMV_BF16: rc = qmv_gemv_bf16(a8, quant_x, pdl, W, rows, cols, x, y, n_vec, st); break;
    }
    if (rc == -2) return fail(QMV_ERR_SHAPE, "cols = %lld needs more shared memory than one SM has", (long long)cols);
    if (rc) return cuda_fail("qmv_matvec");
    return ok();
}

int qmv_matmul(int fmt, const void* W, int64_t rows, int64_t cols, const void* X, float* Y, int64_t m, void* stream)
{
    if (fmt & ~(0xffff | QMV_FLAG_PDL)) return fail(QMV_ERR_INVALID_ARG, "unknown flags 0x%x", fmt & ~0xffff);
    const bool pdl = (fmt & QMV_FLAG_PDL) != 0;
    const int wtype = fmt & 0xff, atype = (fmt >> 8) & 0xff;
    const bool two_pass = atype == QMV_BF16 && wtype != QMV_Q4_K && dequant_type(wtype);
    if (!two_pass && (wtype != QMV_Q4_K || (atype != QMV_BF16 && atype != QMV_Q8_K)))
        return fail(QMV_ERR_UNSUPPORTED,
                    "qmv_matmul: %s weights with %s activations are not provided; supported: QMV_FMT(Q4_K, Q8_K) "
                    "and QMV_FMT(t, BF16) for every GGUF block type and F32/F16/BF16 rows t",
                    type_name(wtype), type_name(atype));
    int rc = check_weights(wtype, W, rows, cols);
    if (rc) return rc;
    if (m < 0) return fail(QMV_ERR_INVALID_ARG, "m must be >= 0");
    if (m > (int64_t)1 << 30 || rows > (int64_t)1 << 30) return fail(QMV_ERR_SHAPE, "m and rows must be below 2^30");
    if (rows == 0 || m == 0) return ok();
    if (!X || !Y) return fail(QMV_ERR_INVALID_ARG, "X and Y must not be NULL");
    if (!aligned(X, 16)) return fail(QMV_ERR_ALIGN, "X must be 16-byte aligned");
    if (!aligned(Y, 4)) return fail(QMV_ERR_ALIGN, "Y must be 4-byte aligned");
    if (!qmv::status_word()) return cuda_fail("qmv_matmul (status word)");
    if (atype == QMV_Q8_K) {
        // W4A8: exact integer block dots on the tensor cores (fp16 operands that
        // hold the integer codes exactly), after a pre-pass that lays the
        // activation codes out as fp16 in the workspace.
        const size_t need = qmv_w4a8_workspace_bytes(cols, m);
        void* ws = nullptr;
        size_t have = 0;
        const int d = qmv::current_device();
        if (d >= 0 && d < qmv::kMaxDevices) {
            std::lock_guard<std::mutex> lock(g_ws_mu);
            ws = g_ws[d].ptr;
            have = g_ws[d].bytes;
        }
        if (!ws || have < need)
            return fail(QMV_ERR_WORKSPACE,
                        "qmv_matmul (W4A8) needs %zu bytes of workspace (qmv_workspace_size(QMV_OP_MATMUL, ...)); "
                        "%zu set", need, have);
        rc = qmv_launch_gemm_q4k_w4a8(W, rows, cols, X, Y, m, ws, pdl, static_cast<cudaStream_t>(stream));
        if (rc == -8) return fail(QMV_ERR_CUDA, "qmv_matmul: could not build a TMA tensor map");
        if (rc) return cuda_fail("qmv_matmul");
        return ok();
    }
    if (two_pass && fused_tile(wtype, cols)) {
        // tiles dequantised into TMEM inside the GEMM
        rc = qmv_launch_gemm_deq_bf16(wtype, W, rows, cols, X, Y, m, pdl, static_cast<cudaStream_t>(stream));
        if (rc == -8) return fail(QMV_ERR_CUDA, "qmv_matmul: could not build a TMA tensor map");
        if (rc) return cuda_fail("qmv_matmul");
        return ok();
    }
    if (two_pass) {
        // BF16 rows as they are; the other types converted to bf16 tiles in
        // the workspace first
        void* ws = nullptr;
        if (wtype != QMV_BF16) {
            const size_t need = qmv_bf16_gemm_workspace_bytes(rows, cols);
            size_t have = 0;
            const int d = qmv::current_device();
            if (d >= 0 && d < qmv::kMaxDevices) {
                std::lock_guard<std::mutex> lock(g_ws_mu);
                ws = g_ws[d].ptr;
                have = g_ws[d].bytes;
            }
            if (!ws || have < need)
                return fail(QMV_ERR_WORKSPACE,
                            "qmv_matmul (%s weights) needs %zu bytes of workspace (qmv_workspace_size(QMV_OP_MATMUL, "
                            "...)); %zu set",
                            type_name(wtype), need, have);
        }
        rc = qmv_launch_gemm_two_pass_bf16(wtype, W, rows, cols, X, Y, m, ws, pdl, static_cast<cudaStream_t>(stream));
        if (rc == -8) return fail(QMV_ERR_CUDA, "qmv_matmul: could not build a TMA tensor map");
        if (rc) return cuda_fail("qmv_matmul");
        return ok();
    }
    rc = qmv_launch_gemm_q4k_bf16(W, rows, cols, X, Y, m, pdl, static_cast<cudaStream_t>(stream));
    if (rc == -8) return fail(QMV_ERR_CUDA, "qmv_matmul: could not build a TMA tensor map");
    if (rc) return cuda_fail("qmv_matmul");
    return ok();
}

int qmv_moe_matvec(int fmt, const void* W3d, int n_expert, int64_t rows, int64_t cols, const int32_t* ids,
                   const float* gates, int k, const void* x, float* y, int64_t n_tok, const float* bias, void* stream)
{
    MoeCall c;
    int rc = moe_check("qmv_moe_matvec", fmt, W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias, c);
    if (rc || c.empty) return rc;
    const int d = qmv::current_device();
    void* ws = nullptr;
    size_t have = 0;
    if (d >= 0 && d < qmv::kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_ws_mu);
        ws = g_ws[d].ptr;
        have = g_ws[d].bytes;
    }
    if (!ws || have < c.need)
        return fail(QMV_ERR_WORKSPACE,
                    "qmv_moe_matvec needs %zu bytes of workspace (qmv_workspace_size(QMV_OP_MOE, ...)); %zu set",
                    c.need, have);
    return moe_run("qmv_moe_matvec", c, W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias, ws, stream);
}

int qmv_moe_block(int fmt, int n_expert, int k, int64_t hidden, int64_t inter, const float* Wr, const float* br,
                  const void* W_gu, const float* b_gu, const void* W_down, const float* b_down, float alpha,
                  float limit, const float* x, int64_t n_tok, float* y, int32_t* ids, float* gates, void* stream)
{
    static const char* name = "qmv_moe_block";
    if (fmt & ~0xffff) return fail(QMV_ERR_INVALID_ARG, "unknown flags 0x%x (8-bit activations are always "
                                   "quantised inside the block)", fmt & ~0xffff);
    const int wtype = fmt & 0xff, atype = (fmt >> 8) & 0xff;
    const bool bf16 = atype == QMV_BF16 && (wtype == QMV_MXFP4 || wtype == QMV_MXFP4_R);
    const bool mx = atype == QMV_MXFP8 && (wtype == QMV_MXFP4 || wtype == QMV_MXFP4_R);
    if (wtype == QMV_MXFP4_R && !bf16 && !mx)
        return fail(QMV_ERR_UNSUPPORTED, "%s: repacked MXFP4_R experts take BF16 or MXFP8 activations (got %s)", name,
                    type_name(atype));
    if (!is_weight_type(wtype) && wtype != QMV_MXFP4_R)
        return fail(QMV_ERR_UNSUPPORTED, "%s: %s is not a weight type", name, type_name(wtype));
    if (atype != QMV_F32 && atype != paired_act(wtype) && !bf16 && !mx)
        return fail(QMV_ERR_UNSUPPORTED, "%s: %s experts take F32 or %s activations%s (got %s)", name,
                    type_name(wtype), type_name(paired_act(wtype)), wtype == QMV_MXFP4 ? ", BF16 or MXFP8" : "",
                    type_name(atype));
    if (mx && (hidden > 4096 || inter > 4096))
        return fail(QMV_ERR_SHAPE, "%s: MXFP8 activations take hidden and inter <= 4096", name);
    if (n_expert < 1 || n_expert > 1024) return fail(QMV_ERR_INVALID_ARG, "n_expert must be in 1..1024 (got %d)", n_expert);
    if (k < 1 || k > 64 || k > n_expert)
        return fail(QMV_ERR_INVALID_ARG, "k must be in 1..min(64, n_expert) (got %d)", k);
    if (hidden <= 0 || inter <= 0) return fail(QMV_ERR_INVALID_ARG, "hidden and inter must be > 0");
    if (n_tok < 0 || n_tok > ((int64_t)1 << 24) / k)
        return fail(QMV_ERR_INVALID_ARG, "n_tok must be >= 0 with n_tok*k <= 16777216");
    const int geo = wtype == QMV_MXFP4_R ? QMV_MXFP4 : wtype;
    int rc = check_weights(geo, W_gu, 2 * inter, hidden);
    if (rc) return rc;
    rc = check_weights(geo, W_down, hidden, inter);
    if (rc) return rc;
    if ((bf16 || mx) && (2 * inter > (int64_t)1 << 30 || hidden > (int64_t)1 << 30))
        return fail(QMV_ERR_SHAPE, "rows must be below 2^30");
    if (n_tok == 0) return ok();
    if (!Wr || !x || !y || !ids || !gates)
        return fail(QMV_ERR_INVALID_ARG, "Wr, x, y, ids and gates must not be NULL");
    if (!aligned(x, 16)) return fail(QMV_ERR_ALIGN, "x must be 16-byte aligned");
    if (!aligned(Wr, 4) || !aligned(y, 4) || !aligned(ids, 4) || !aligned(gates, 4) || (br && !aligned(br, 4)) ||
        (b_gu && !aligned(b_gu, 4)) || (b_down && !aligned(b_down, 4)))
        return fail(QMV_ERR_ALIGN, "Wr, br, biases, y, ids and gates must be 4-byte aligned");
    const size_t need = qmv_moe_block_workspace_bytes(bf16, mx, n_expert, hidden, inter, n_tok, k);
    const int d = qmv::current_device();
    void* ws = nullptr;
    size_t have = 0;
    if (d >= 0 && d < qmv::kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_ws_mu);
        ws = g_ws[d].ptr;
        have = g_ws[d].bytes;
    }
    if (!ws || have < need)
        return fail(QMV_ERR_WORKSPACE, "%s needs %zu bytes of workspace (qmv_moe_block_workspace_size); %zu set",
                    name, need, have);
    if (!qmv::status_word()) return cuda_fail(name);
    rc = qmv_launch_moe_block(wtype, atype != QMV_F32 && !bf16 && !mx, bf16, mx, qmv_block_bytes(paired_act(wtype)), n_expert,
                              k, hidden, inter, Wr, br, W_gu, b_gu, W_down, b_down, alpha, limit, x, n_tok, y, ids,
                              gates, ws, static_cast<cudaStream_t>(stream));
    if (rc == -2) return fail(QMV_ERR_SHAPE, "%s: a projection needs more shared memory than one SM has", name);
    if (rc == -8) return fail(QMV_ERR_CUDA, "%s: could not build a TMA tensor map", name);
    if (rc) return cuda_fail(name);
    return ok();
}

size_t qmv_moe_block_workspace_size(int fmt, int n_expert, int k, int64_t hidden, int64_t inter, int64_t n_tok)
{
    if (n_expert < 1 || k < 1 || hidden <= 0 || inter <= 0 || n_tok <= 0) return 0;
    const int wtype = fmt & 0xff, atype = (fmt >> 8) & 0xff;
    const bool bf16 = atype == QMV_BF16 && (wtype == QMV_MXFP4 || wtype == QMV_MXFP4_R);
    const bool mx = atype == QMV_MXFP8 && (wtype == QMV_MXFP4 || wtype == QMV_MXFP4_R);
    return qmv_moe_block_workspace_bytes(bf16, mx, n_expert, hidden, inter, n_tok, k);
}

size_t qmv_workspace_size(int op, int fmt, int64_t rows, int64_t cols, int64_t n)
{
    if (op == QMV_OP_MOE && rows > 0 && n > 0 && cols >= 0)
        return qmv_moe_workspace_bytes(((fmt >> 8) & 0xff) == QMV_BF16, rows, cols, n,
                                       ((fmt >> 8) & 0xff) == QMV_MXFP8);
    if (op == QMV_OP_MATMUL && (fmt & 0xffff) == QMV_FMT(QMV_Q4_K, QMV_Q8_K) && rows > 0 && n > 0 && cols > 0 &&
        cols % 256 == 0)
        return qmv_w4a8_workspace_bytes(cols, n);
    if (op == QMV_OP_MATMUL && ((fmt >> 8) & 0xff) == QMV_BF16 && dequant_type(fmt & 0xff) && (fmt & 0xff) != QMV_Q4_K &&
        (fmt & 0xff) != QMV_BF16 && !fused_tile(fmt & 0xff, cols) && rows > 0 && n > 0 && cols > 0)
        return qmv_bf16_gemm_workspace_bytes(rows, cols);
    return 0;
}

int qmv_set_workspace(void* ptr, size_t bytes)
{
    if (ptr && !aligned(ptr, 256)) return fail(QMV_ERR_ALIGN, "workspace must be 256-byte aligned");
    const int d = qmv::current_device();
    if (d < 0 || d >= qmv::kMaxDevices) return fail(QMV_ERR_INVALID_ARG, "device %d out of range", d);
    std::lock_guard<std::mutex> lock(g_ws_mu);
    g_ws[d].ptr = ptr;
    g_ws[d].bytes = ptr ? bytes : 0;
    return ok();
}

int qmv_set_wait_limit(unsigned ns)
{
    const int d = qmv::current_device();
    if (d < 0 || d >= qmv::kMaxDevices) return fail(QMV_ERR_INVALID_ARG, "device %d out of range", d);
    qmv::set_wait_limit_ns(d, ns);
    return ok();
}

int qmv_get_status(void* stream)
{
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_fail("qmv_get_status (synchronize)");
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_qmv_status, sizeof v) != cudaSuccess) return cuda_fail("qmv_get_status (read)");
    if (v == 0) return ok();
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_qmv_status, &zero, sizeof zero) != cudaSuccess) return cuda_fail("qmv_get_status (clear)");
    std::string what;
    if (v & QMV_DEV_BAD_EXPERT) what += "an expert id was out of range; ";
    if (v & QMV_DEV_WAIT_TIMEOUT) what += "a pipeline wait gave up (a copy never landed); ";
    if (v & QMV_DEV_BAD_ARG) what += "a kernel saw an inconsistent argument; ";
    return fail(QMV_ERR_DEVICE_STATUS, "device status 0x%x: %s", v, what.c_str());
}

// ---- the MoE call that allocates nothing ------------------------------------------
}  // extern "C"

namespace {

// Device address of g_moe_noalloc_scratch on the current device, looked up
// once per device (with that device current) and cached.  In host code the
// array's name is only a stand-in for the symbol, never a device pointer.
void* moe_noalloc_scratch()
{
    static std::atomic<void*> cache[qmv::kMaxDevices];
    const int d = qmv::current_device();
    if (d < 0 || d >= qmv::kMaxDevices) return nullptr;
    void* p = cache[d].load(std::memory_order_acquire);
    if (!p) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_moe_noalloc_scratch) != cudaSuccess || !a) return nullptr;
        cache[d].store(a, std::memory_order_release);
        p = a;
    }
    return p;
}

}  // namespace

extern "C" {

int qmv_moe_matvec_noalloc(int fmt, const void* W3d, int n_expert, int64_t rows, int64_t cols, const int32_t* ids,
                           const float* gates, int k, const void* x, float* y, int64_t n_tok, const float* bias,
                           void* stream)
{
    MoeCall c;
    int rc = moe_check("qmv_moe_matvec_noalloc", fmt, W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias, c);
    if (rc || c.empty) return rc;
    if (c.need > QMV_MOE_NOALLOC_MAX_BYTES)
        return fail(QMV_ERR_SHAPE,
                    "qmv_moe_matvec_noalloc: %lld (token, slot) pairs x %lld rows need %zu bytes of scratch; the "
                    "built-in scratch holds %zu (about n_tok*k*rows*4 bytes are needed); use qmv_moe_matvec with a "
                    "workspace for larger calls",
                    (long long)(n_tok * k), (long long)rows, c.need, (size_t)QMV_MOE_NOALLOC_MAX_BYTES);
    void* ws = moe_noalloc_scratch();
    if (!ws) return cuda_fail("qmv_moe_matvec_noalloc (scratch address)");
    return moe_run("qmv_moe_matvec_noalloc", c, W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias, ws,
                   stream);
}

}  // extern "C"
