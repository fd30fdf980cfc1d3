// moe_block.cu -- a whole mixture-of-experts block: router, top-k, gate_up,
// clipped SwiGLU, down.
//
// "Models and formats" page, "Architectures": a router picks k of n experts
// per token from stacked 3-D expert tensors; gpt-oss adds a bias to every
// expert projection and gates with a clipped SwiGLU whose linear half is
// offset by one.  The pages print neither the router's arithmetic nor the
// clipping constants; the library takes these readings:
//
//   logit[t][e]  fp32: 32 partial sums, partial l over the elements
//                h = l, l + 32, ... by fused multiply-add from 0, then a
//                butterfly (partial l + partial l^o for o = 16, 8, 4, 2, 1),
//                then the router bias.  The top-k choice depends only on
//                this fixed order.
//   top k        the k largest logits, ties to the lower expert id, in
//                descending order (slot 0 = largest).
//   gates        softmax over the k kept logits in fp32:
//                exp(l_s - l_0) / (sum over s in slot order).
//   activation   rows [0, I) of each gate_up expert give g, rows [I, 2I)
//                give u: h = min(g, limit) * sigmoid(alpha * min(g, limit))
//                * (clamp(u, -limit, limit) + 1), in fp32; alpha and limit
//                are arguments.
//
//  k_router      (token tile of 8) x (8 experts) per block, one warp per
//                expert: the logits in the order above; the blocks of the
//                first expert group also round x to bf16 when the experts
//                run on the bf16 tensor-core GEMM.
//  k_topk        one warp per token: k rounds of a warp-wide arg-max over
//                the token's logits (staged in shared memory), then the
//                gates.
//  (moe.cu)      gate_up: the expert matvecs or grouped GEMM, up/gate form.
//  k_swiglu      the activation, fp32 or bf16 out.
//  (moe.cu)      down: the gate-weighted form, reusing the grouping.
#include <cuda_bf16.h>

#include "common.cuh"
#include "runtime.cuh"

namespace qmv {

constexpr int RT_TOK = 8;   // tokens per router block
constexpr int RT_EXP = 8;   // experts per router block (one per warp)

__global__ void __launch_bounds__(256) k_router(const float* __restrict__ x, const float* __restrict__ Wr,
                                                const float* __restrict__ br, int64_t n_tok, int64_t hidden, int E,
                                                float* __restrict__ logits, __nv_bfloat16* __restrict__ xb)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const int64_t t0 = (int64_t)blockIdx.x * RT_TOK;
    const int nt = (int)(n_tok - t0 < RT_TOK ? n_tok - t0 : RT_TOK);
    const int e = blockIdx.y * RT_EXP + warp;
    if (xb && blockIdx.y == 0)
        for (int64_t i = threadIdx.x; i < (int64_t)nt * hidden; i += blockDim.x)
            xb[t0 * hidden + i] = __float2bfloat16_rn(x[t0 * hidden + i]);
    if (e >= E) return;
    const float* w = Wr + (int64_t)e * hidden;
    const float* xt = x + t0 * hidden;
    float acc[RT_TOK];
#pragma unroll
    for (int j = 0; j < RT_TOK; ++j) acc[j] = 0.f;
    // Each lane's chain runs in ascending h; the loads of U steps are issued
    // before their multiply-adds so that one memory latency covers U steps.
    constexpr int U = 8;
    int64_t h = lane;
    if (nt == RT_TOK) {
        for (; h + (U - 1) * 32 < hidden; h += U * 32) {
            float wv[U], xv[U][RT_TOK];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                wv[u] = __ldg(w + h + u * 32);
#pragma unroll
                for (int j = 0; j < RT_TOK; ++j) xv[u][j] = __ldg(xt + j * hidden + h + u * 32);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < RT_TOK; ++j) acc[j] = __fmaf_rn(xv[u][j], wv[u], acc[j]);
        }
    } else if (nt == 1) {
        // one token (decode): 24 steps per memory round trip
        constexpr int U1 = 24;
        for (; h + (U1 - 1) * 32 < hidden; h += U1 * 32) {
            float wv[U1], xv[U1];
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                wv[u] = __ldg(w + h + u * 32);
                xv[u] = __ldg(xt + h + u * 32);
            }
#pragma unroll
            for (int u = 0; u < U1; ++u) acc[0] = __fmaf_rn(xv[u], wv[u], acc[0]);
        }
    }
    for (; h < hidden; h += 32) {   // the rest, and partial token tiles of more than one token
        const float wv = __ldg(w + h);
#pragma unroll
        for (int j = 0; j < RT_TOK; ++j)
            if (j < nt) acc[j] = __fmaf_rn(__ldg(xt + j * hidden + h), wv, acc[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < RT_TOK; ++j) acc[j] = __fadd_rn(acc[j], __shfl_xor_sync(0xffffffffu, acc[j], o));
    if (lane == 0) {
        const float b = br ? br[e] : 0.f;
#pragma unroll
        for (int j = 0; j < RT_TOK; ++j)
            if (j < nt) logits[(t0 + j) * E + e] = br ? __fadd_rn(acc[j], b) : acc[j];
    }
}

// (v, e) beats (v2, e2): a larger logit, or the same logit and a lower id; a
// candidate with e < 0 (none) never wins.
__device__ __forceinline__ bool beats(float v, int e, float v2, int e2)
{
    return e >= 0 && (e2 < 0 || v > v2 || (v == v2 && e < e2));
}

__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int64_t n_tok, int E, int k,
                                              int32_t* __restrict__ ids, float* __restrict__ gates)
{
    extern __shared__ float sm[];   // per warp: E logits, then 64 kept logits
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const int64_t t = (int64_t)blockIdx.x * 8 + warp;
    if (t >= n_tok) return;
    float* L = sm + warp * (E + 64);
    float* kept = L + E;
    for (int e = lane; e < E; e += 32) L[e] = logits[t * E + e];
    __syncwarp();
    uint32_t taken = 0;   // bit j: expert lane + 32 j is already kept
    int id_mine0 = 0, id_mine1 = 0;   // the ids of slots lane and lane + 32
    for (int s = 0; s < k; ++s) {
        float bv = 0.f;
        int be = -1;
        for (int j = 0, e = lane; e < E; ++j, e += 32)
            if (!((taken >> j) & 1u) && beats(L[e], e, bv, be)) {
                bv = L[e];
                be = e;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
            const int e2 = __shfl_xor_sync(0xffffffffu, be, o);
            if (beats(v2, e2, bv, be)) {
                bv = v2;
                be = e2;
            }
        }
        if (be >= 0 && (be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == 0) kept[s] = bv;
        if (s == lane) id_mine0 = be;
        if (s == lane + 32) id_mine1 = be;
    }
    __syncwarp();
    const float m = kept[0];
    const float e0 = lane < k ? expf(kept[lane] - m) : 0.f;
    const float e1 = lane + 32 < k ? expf(kept[lane + 32] - m) : 0.f;
    __syncwarp();
    if (lane < k) kept[lane] = e0;
    if (lane + 32 < k) kept[lane + 32] = e1;
    __syncwarp();
    float sum = 0.f;
    for (int s = 0; s < k; ++s) sum = __fadd_rn(sum, kept[s]);
    if (lane < k) {
        ids[t * k + lane] = id_mine0;
        gates[t * k + lane] = __fdiv_rn(e0, sum);
    }
    if (lane + 32 < k) {
        ids[t * k + lane + 32] = id_mine1;
        gates[t * k + lane + 32] = __fdiv_rn(e1, sum);
    }
}

template <bool BF>
__global__ void __launch_bounds__(256) k_swiglu(const float* __restrict__ y1, int64_t n_pairs, int64_t inter,
                                                float alpha, float limit, void* __restrict__ h)
{
    pdl_trigger();
    pdl_wait();
    const int64_t n = n_pairs * inter;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = i / inter, c = i - p * inter;
        const float g = y1[p * 2 * inter + c], u = y1[p * 2 * inter + inter + c];
        const float gc = fminf(g, limit);
        const float uc = fminf(fmaxf(u, -limit), limit);
        const float sig = __fdiv_rn(1.f, __fadd_rn(1.f, expf(__fmul_rn(-alpha, gc))));
        const float v = __fmul_rn(__fmul_rn(gc, sig), __fadd_rn(uc, 1.f));
        if constexpr (BF) static_cast<__nv_bfloat16*>(h)[i] = __float2bfloat16_rn(v);
        else static_cast<float*>(h)[i] = v;
    }
}

inline size_t r256b(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace qmv

size_t qmv_moe_workspace_bytes(bool bf16, int64_t rows, int64_t cols, int64_t n_pairs, bool mx);
int qmv_launch_moe_ex(int wtype, bool a8, bool quant_x, bool bf16, bool mx, size_t act_block_bytes,
                      const void* W3d, int n_expert, int64_t rows, int64_t cols, const int32_t* ids,
                      const float* gates, int k, const void* x, float* y, int64_t n_tok, const float* bias, void* ws,
                      bool grouped, cudaStream_t st);

// Workspace: logits [n_tok][n_expert] fp32 | gate_up outputs [n_pairs][2I]
// fp32 | activations [n_pairs][I] (fp32, or bf16) | (bf16) x [n_tok][hidden]
// bf16 | the scratch of the two expert calls (shared: they run in order).
size_t qmv_moe_block_workspace_bytes(bool bf16, bool mx, int n_expert, int64_t hidden, int64_t inter, int64_t n_tok,
                                     int k)
{
    using qmv::r256b;
    const int64_t n_pairs = n_tok * k;
    const int64_t mr = hidden > 2 * inter ? hidden : 2 * inter, mc = hidden > inter ? hidden : inter;
    return r256b((size_t)n_tok * n_expert * 4) + r256b((size_t)n_pairs * 2 * inter * 4) +
           r256b((size_t)n_pairs * inter * (bf16 ? 2 : 4)) + (bf16 ? r256b((size_t)n_tok * hidden * 2) : 0) +
           qmv_moe_workspace_bytes(bf16, mr, mc, n_pairs, mx);
}

// a8: both projections quantise their fp32 inputs to the paired 8-bit blocks
// inside the expert kernels.  bf16: MXFP4 experts on the grouped GEMM, x and
// the activations rounded to bf16.  mx: MXFP4 experts on the block-scaled
// GEMM, x and the activations quantised to MXFP8 by its gather.  Returns 0, or
// the codes of qmv_launch_moe.
int qmv_launch_moe_block(int wtype, bool a8, bool bf16, bool mx, size_t act_block_bytes, int n_expert, int k,
                         int64_t hidden, int64_t inter, const float* Wr, const float* br, const void* Wgu,
                         const float* bgu, const void* Wd, const float* bd, float alpha, float limit, const float* x,
                         int64_t n_tok, float* y, int32_t* ids, float* gates, void* ws, cudaStream_t st)
{
    using namespace qmv;
    if (n_tok == 0) return 0;
    const int64_t n_pairs = n_tok * k;
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* logits = reinterpret_cast<float*>(w);
    w += r256b((size_t)n_tok * n_expert * 4);
    float* y1 = reinterpret_cast<float*>(w);
    w += r256b((size_t)n_pairs * 2 * inter * 4);
    void* h = w;
    w += r256b((size_t)n_pairs * inter * (bf16 ? 2 : 4));
    __nv_bfloat16* xb = nullptr;
    if (bf16) {
        xb = reinterpret_cast<__nv_bfloat16*>(w);
        w += r256b((size_t)n_tok * hidden * 2);
    }
    void* inner = w;

    const dim3 rgrid((unsigned)((n_tok + RT_TOK - 1) / RT_TOK), (unsigned)((n_expert + RT_EXP - 1) / RT_EXP));
    // each kernel waits for its predecessor before touching memory: all are
    // launched as programmatic dependents
    if (launch_ex(k_router, rgrid, dim3(256), 0, st, true, x, Wr, br, n_tok, hidden, n_expert, logits, xb) !=
        cudaSuccess)
        return -6;
    const size_t tsm = (size_t)8 * (n_expert + 64) * 4;
    prepare_kernel(k_topk, 256, tsm);
    if (launch_ex(k_topk, dim3((unsigned)((n_tok + 7) / 8)), dim3(256), tsm, st, true, (const float*)logits, n_tok,
                  n_expert, k, ids, gates) != cudaSuccess)
        return -6;

    const void* xin = bf16 ? static_cast<const void*>(xb) : static_cast<const void*>(x);
    int rc = qmv_launch_moe_ex(wtype, a8, a8, bf16, mx, act_block_bytes, Wgu, n_expert, 2 * inter, hidden, ids, nullptr,
                               k, xin, y1, n_tok, bgu, inner, false, st);
    if (rc) return rc;
    const int64_t n = n_pairs * inter;
    const unsigned sg = (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    if (launch_ex(bf16 ? k_swiglu<true> : k_swiglu<false>, dim3(sg), dim3(256), 0, st, true, (const float*)y1, n_pairs,
                  inter, alpha, limit, h) != cudaSuccess)
        return -6;
    return qmv_launch_moe_ex(wtype, a8, a8, bf16, mx, act_block_bytes, Wd, n_expert, hidden, inter, ids, gates, k, h, y,
                             n_tok, bd, inner, true, st);
}
