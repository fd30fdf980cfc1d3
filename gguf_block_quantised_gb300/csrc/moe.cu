// moe.cu -- grouping and combining for the mixture-of-experts matvec.
//
// "Models and formats" page, "Architectures": a router picks k of n experts
// per token (here: the ids and gates are inputs), experts are stacked 3-D
// tensors, and gpt-oss adds a bias on every expert projection.
//
//  k_moe_group    one block: validates the ids and sorts the n_tok*k (token,
//                 slot) pairs by expert with a stable counting sort (one warp
//                 per expert, ballots over the pairs in order), writing
//                 offsets[n_expert+1], the experts that received pairs
//                 (active[], in id order, and their count) and perm[n_pairs]
//                 to the workspace.
//  k_moe_gemv     (moe.cuh) the expert matvecs over grouped pairs.
//  k_moe_combine  down form only: y[t][r] = sum over slots s, in slot order, of
//                 gates[t][s] * (part[t*k+s][r] + bias[e][r]).
// Nothing here uses atomics on data, so results are deterministic.
#include "common.cuh"
#include "runtime.cuh"

namespace qmv {

// Expert ids staged in shared memory when they fit (the scans below read each
// id once per expert a warp handles).
constexpr int kGroupStageIds = 10240;   // 40 KB: with base[], under the 48 KB of static shared memory

__global__ void __launch_bounds__(1024) k_moe_group(const int32_t* __restrict__ ids_g, int n_pairs, int n_expert,
                                                    int* __restrict__ offsets, int* __restrict__ active,
                                                    int* __restrict__ perm, unsigned* status)
{
    __shared__ int base[1025];
    __shared__ int ids_s[kGroupStageIds];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    pdl_trigger();
    pdl_wait();
    const bool staged = n_pairs <= kGroupStageIds;
    for (int p = tid; p < n_pairs; p += blockDim.x) {
        const int e = ids_g[p];
        if (e < 0 || e >= n_expert) atomicOr(status, QMV_DEV_BAD_EXPERT);
        if (staged) ids_s[p] = e;
    }
    __syncthreads();
    const int32_t* ids = staged ? ids_s : ids_g;
    for (int e = warp; e < n_expert; e += nw) {
        int c = 0;
        int b = 0;
        for (; b + 96 < n_pairs; b += 128) {   // four independent loads and ballots per round
            const int v0 = ids[b + lane], v1 = ids[b + 32 + lane], v2 = ids[b + 64 + lane];
            const int p3 = b + 96 + lane;
            const int v3 = p3 < n_pairs ? ids[p3] : -1;
            c += __popc(__ballot_sync(0xffffffffu, v0 == e)) + __popc(__ballot_sync(0xffffffffu, v1 == e)) +
                 __popc(__ballot_sync(0xffffffffu, v2 == e)) + __popc(__ballot_sync(0xffffffffu, v3 == e));
        }
        for (; b < n_pairs; b += 32) {
            const int p = b + lane;
            c += __popc(__ballot_sync(0xffffffffu, p < n_pairs && ids[p] == e));
        }
        if (lane == 0) base[e] = c;
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0, na = 0;
        for (int e = 0; e < n_expert; ++e) {
            const int c = base[e];
            base[e] = run;
            offsets[e] = run;
            run += c;
            if (c > 0) active[1 + na++] = e;
        }
        offsets[n_expert] = run;   // pairs with a valid expert
        active[0] = na;
    }
    __syncthreads();
    const uint32_t lt = (1u << lane) - 1u;
    for (int e = warp; e < n_expert; e += nw) {
        int pos = base[e];
        for (int b = 0; b < n_pairs; b += 128) {   // four chunks of 32 pairs per round, placed in order
            bool m[4];
            uint32_t mask[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int p = b + 32 * j + lane;
                m[j] = p < n_pairs && ids[p] == e;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) mask[j] = __ballot_sync(0xffffffffu, m[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (m[j]) perm[pos + __popc(mask[j] & lt)] = b + 32 * j + lane;
                pos += __popc(mask[j]);
            }
        }
    }
}

__global__ void k_moe_combine(const float* __restrict__ part, const int32_t* __restrict__ ids,
                              const float* __restrict__ gates, const float* __restrict__ bias, int k, int64_t rows,
                              int64_t n_tok, int n_expert, float* __restrict__ y)
{
    pdl_trigger();
    pdl_wait();   // the slot outputs come from the kernel before this one
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_tok * rows) return;
    const int64_t t = i / rows, r = i % rows;
    float acc = 0.f;
    for (int s = 0; s < k; ++s) {
        const int64_t pr = t * k + s;
        const int e = ids[pr];
        if (e < 0 || e >= n_expert) continue;
        float v = part[pr * rows + r];
        if (bias) v += bias[(int64_t)e * rows + r];
        acc = __fmaf_rn(gates[pr], v, acc);
    }
    y[i] = acc;
}

inline size_t r256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace qmv

#define QMV_MOE_DECL(NAME)                                                                                      \
    int NAME(bool a8, bool quant_x, const void* W3d, int n_expert, int64_t rows, int64_t cols, const int* offsets, \
             const int* active, const int* perm, const int32_t* ids, bool self_group, int n_pairs, int n_tok,       \
             const void* x, size_t xrow, int kdiv, float* out, const float* bias, cudaStream_t st);
QMV_MOE_DECL(qmv_moe_q4_0)
QMV_MOE_DECL(qmv_moe_q5_0)
QMV_MOE_DECL(qmv_moe_q8_0)
QMV_MOE_DECL(qmv_moe_mxfp4)
QMV_MOE_DECL(qmv_moe_q4_k)
QMV_MOE_DECL(qmv_moe_q6_k)
QMV_MOE_DECL(qmv_moe_q4_1)
QMV_MOE_DECL(qmv_moe_q5_1)
QMV_MOE_DECL(qmv_moe_q8_1)
QMV_MOE_DECL(qmv_moe_q2_k)
QMV_MOE_DECL(qmv_moe_q3_k)
QMV_MOE_DECL(qmv_moe_q5_k)
QMV_MOE_DECL(qmv_moe_f32)
QMV_MOE_DECL(qmv_moe_f16)
QMV_MOE_DECL(qmv_moe_bf16)

size_t qmv_moe_gemm_extra_bytes(int64_t cols, int64_t n_pairs, bool mx);
int qmv_launch_moe_gemm_mxfp4(const void* W3d, bool planar, bool mx, int n_expert, int64_t rows, int64_t cols,
                              const void* x, int kdiv, int64_t n_pairs, const int* offsets, const int* active,
                              const int* perm, void* ws, float* out, const float* bias, cudaStream_t st);

// Workspace layout: offsets[1025] + active[1025] | perm[n_pairs] | per-slot
// outputs [n_pairs][rows] fp32 | (the grouped GEMM's activations, bf16 or
// MXFP8, only) its slot list and packed activations.
size_t qmv_moe_workspace_bytes(bool bf16, int64_t rows, int64_t cols, int64_t n_pairs, bool mx)
{
    using qmv::r256;
    const size_t base = r256(2050 * 4) + r256((size_t)n_pairs * 4) + r256((size_t)n_pairs * (size_t)rows * 4);
    return base + ((bf16 || mx) ? qmv_moe_gemm_extra_bytes(cols, n_pairs, mx) : 0);
}

// bf16: MXFP4 experts with bf16 activations, through the grouped tensor-core
// GEMM (moe_gemm.cu); mx: the same with fp32 activations quantised to MXFP8
// on the block-scaled MMA; otherwise the expert matvecs of moe.cuh.  grouped: the
// workspace already holds the grouping of these ids (an earlier call with the
// same ids, n_tok and k on this workspace), so it is not rebuilt.
// Returns 0, -2 (shape beyond the plan), -6 (launch failure), -8 (tensor map).
int qmv_launch_moe_ex(int wtype, bool a8, bool quant_x, bool bf16, bool mx, size_t act_block_bytes,
                      const void* W3d, int n_expert, int64_t rows, int64_t cols, const int32_t* ids,
                      const float* gates, int k, const void* x, float* y, int64_t n_tok, const float* bias, void* ws,
                      bool grouped, cudaStream_t st)
{
    using namespace qmv;
    const int64_t n_pairs = n_tok * k;
    if (n_pairs == 0 || rows == 0) return 0;
    uint8_t* w = static_cast<uint8_t*>(ws);
    int* offsets = reinterpret_cast<int*>(w);            // [n_expert + 1]
    int* active = offsets + 1025;                         // [0] = count, [1..] = expert ids
    int* perm = reinterpret_cast<int*>(w + r256(2050 * 4));
    float* part = reinterpret_cast<float*>(w + r256(2050 * 4) + r256((size_t)n_pairs * 4));
    // At most 32 pairs on the matvec path (decode): each expert CTA groups the
    // ids itself, so the grouping kernel is not launched.
    const bool self_group = !bf16 && !mx && n_pairs <= 32;
    if (!grouped && !self_group) {
        // every kernel of the chain waits for its predecessor before touching memory,
        // so each is launched as a programmatic dependent (its launch overlaps the
        // kernel before it)
        if (launch_ex(k_moe_group, dim3(1), dim3(1024), 0, st, true, ids, (int)n_pairs, n_expert, offsets, active, perm,
                      status_word()) != cudaSuccess)
            return -6;
    }
    const size_t xrow = (a8 && !quant_x) ? (size_t)(cols / (kq_rt(wtype) ? 256 : 32)) *
                                               act_block_bytes
                                         : (size_t)cols * 4;
    const int kdiv = gates ? 1 : k;
    float* out = gates ? part : y;
    const float* b = gates ? nullptr : bias;
    int rc = -3;
    if (bf16 || mx) {
        void* gws = w + r256(2050 * 4) + r256((size_t)n_pairs * 4) + r256((size_t)n_pairs * (size_t)rows * 4);
        rc = wtype == QMV_MXFP4 || wtype == QMV_MXFP4_R
                 ? qmv_launch_moe_gemm_mxfp4(W3d, wtype == QMV_MXFP4_R, mx, n_expert, rows, cols, x, kdiv, n_pairs,
                                             offsets, active, perm, gws, out, b, st)
                 : -3;
    }
#define QMV_MOE_CALL(NAME) \
    NAME(a8, quant_x, W3d, n_expert, rows, cols, offsets, active, perm, ids, self_group, (int)n_pairs, (int)n_tok, x, \
         xrow, kdiv, out, b, st)
    if (!bf16 && !mx) switch (wtype) {
    case QMV_Q4_0: rc = QMV_MOE_CALL(qmv_moe_q4_0); break;
    case QMV_Q5_0: rc = QMV_MOE_CALL(qmv_moe_q5_0); break;
    case QMV_Q8_0: rc = QMV_MOE_CALL(qmv_moe_q8_0); break;
    case QMV_MXFP4: rc = QMV_MOE_CALL(qmv_moe_mxfp4); break;
    case QMV_Q4_K: rc = QMV_MOE_CALL(qmv_moe_q4_k); break;
    case QMV_Q6_K: rc = QMV_MOE_CALL(qmv_moe_q6_k); break;
    case QMV_Q4_1: rc = QMV_MOE_CALL(qmv_moe_q4_1); break;
    case QMV_Q5_1: rc = QMV_MOE_CALL(qmv_moe_q5_1); break;
    case QMV_Q8_1: rc = QMV_MOE_CALL(qmv_moe_q8_1); break;
    case QMV_Q2_K: rc = QMV_MOE_CALL(qmv_moe_q2_k); break;
    case QMV_Q3_K: rc = QMV_MOE_CALL(qmv_moe_q3_k); break;
    case QMV_Q5_K: rc = QMV_MOE_CALL(qmv_moe_q5_k); break;
    case QMV_F32: rc = QMV_MOE_CALL(qmv_moe_f32); break;
    case QMV_F16: rc = QMV_MOE_CALL(qmv_moe_f16); break;
    case QMV_BF16: rc = QMV_MOE_CALL(qmv_moe_bf16); break;
    }
#undef QMV_MOE_CALL
    if (rc) return rc;
    if (gates) {
        const int64_t n = n_tok * rows;
        if (launch_ex(k_moe_combine, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, true, (const float*)part,
                      ids, gates, bias, k, rows, n_tok, n_expert, y) != cudaSuccess)
            return -6;
    }
    return 0;
}

int qmv_launch_moe(int wtype, bool a8, bool quant_x, bool bf16, size_t act_block_bytes, const void* W3d,
                   int n_expert, int64_t rows, int64_t cols, const int32_t* ids, const float* gates, int k,
                   const void* x, float* y, int64_t n_tok, const float* bias, void* ws, cudaStream_t st)
{
    return qmv_launch_moe_ex(wtype, a8, quant_x, bf16, false, act_block_bytes, W3d, n_expert, rows, cols, ids, gates,
                             k, x, y, n_tok, bias, ws, false, st);
}
