/*
 * moeblock.c -- the router and the gated activation of a mixture-of-experts
 * block.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * "Models and formats" page, "Architectures": a router picks k of n experts
 * per token; gpt-oss has "a clipped SwiGLU gate whose linear half is offset by
 * one" and a bias on every expert projection.  The pages give neither the
 * clipping constants nor the router's arithmetic; the readings are:
 *
 *   router logit  l[t][e] = (sum_h x[t][h] * Wr[e][h]) + br[e], in fp32, in
 *                 the order the kernel that decides the top k uses, so that
 *                 the decision is the same on both sides: 32 partial sums, sum
 *                 l taking the elements h = l, l + 32, l + 64, ... with fused
 *                 multiply-adds from 0; then pairwise sums over the partials
 *                 in a fixed tree (partial i plus partial i ^ o, for o = 16, 8,
 *                 4, 2, 1, every level over all 32 partials); then the bias.
 *   top k         the k largest logits, ties to the lower expert id, in
 *                 descending order.
 *   gates         softmax over the k kept logits, in fp64.
 *   activation    for the gate half g and the linear half u of the first
 *                 projection (rows [0, I) and [I, 2I) of each expert):
 *                 g' = min(g, limit), u' = clamp(u, -limit, limit),
 *                 h = g' * sigmoid(alpha * g') * (u' + 1), in fp64.
 */
#include "oracle.h"
#include <math.h>
#include <string.h>

int orc_router(const float* x, const float* Wr, const float* br, int64_t n_tok, int64_t hidden, int64_t n_expert,
               float* logits)
{
    if (n_tok < 0 || hidden <= 0 || n_expert <= 0) return ORC_EINVAL;
    for (int64_t t = 0; t < n_tok; t++)
        for (int64_t e = 0; e < n_expert; e++) {
            float p[32];
            for (int l = 0; l < 32; l++) {
                float acc = 0.0f;
                for (int64_t h = l; h < hidden; h += 32) acc = fmaf(x[t * hidden + h], Wr[e * hidden + h], acc);
                p[l] = acc;
            }
            for (int o = 16; o > 0; o >>= 1) {
                float q[32];
                for (int l = 0; l < 32; l++) q[l] = p[l] + p[l ^ o];
                memcpy(p, q, sizeof p);
            }
            logits[t * n_expert + e] = br ? p[0] + br[e] : p[0];
        }
    return ORC_OK;
}

int orc_topk_softmax(const float* logits, int64_t n_tok, int64_t n_expert, int64_t k, int32_t* ids, double* gates)
{
    if (k <= 0 || k > n_expert || n_tok < 0) return ORC_EINVAL;
    for (int64_t t = 0; t < n_tok; t++) {
        const float* l = logits + t * n_expert;
        int32_t* id = ids + t * k;
        for (int64_t s = 0; s < k; s++) {
            int best = -1;
            for (int64_t e = 0; e < n_expert; e++) {
                int taken = 0;
                for (int64_t j = 0; j < s; j++) taken |= id[j] == e;
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = (int)e;   /* strictly greater: ties keep the lower id */
            }
            id[s] = best;
        }
        double m = (double)l[id[0]], sum = 0.0;
        for (int64_t s = 0; s < k; s++) sum += exp((double)l[id[s]] - m);
        for (int64_t s = 0; s < k; s++) gates[t * k + s] = exp((double)l[id[s]] - m) / sum;
    }
    return ORC_OK;
}

double orc_swiglu(double g, double u, double alpha, double limit)
{
    const double gc = g < limit ? g : limit;
    const double uc = u < -limit ? -limit : (u > limit ? limit : u);
    return gc * (1.0 / (1.0 + exp(-alpha * gc))) * (uc + 1.0);
}
