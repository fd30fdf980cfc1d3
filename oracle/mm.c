/*
 * mm.c -- integer block dots, matrix-vector and matrix-matrix products and the
 * mixture-of-experts product.  TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * What is computed ("Architecture" page, "The package map": pkg/tensor MatVec
 * for decode and MatMul for prefill, pkg/quant fused W4A8 kernels):
 *
 *   y[v][r] = sum_c w[r][c] * xhat[v][c]
 *
 * with w the exactly decoded weight and xhat the activation as consumed:
 * fp32 x (A32), bf16 x against bf16-rounded weights (the prefill tiles), or
 * d_x * xq (A8).  In the A8 form each block contributes
 *
 *   d_x * (d * S - dmin * Mn),  S = sum_i sub_scale_i * code_i * xq_i,
 *                               Mn = sum_i sub_min_i * xq_i,
 *
 * with S and Mn exact integers; everything after the integers is fp64.
 * There is no blocking or reordering beyond this definition: rows, vectors and
 * blocks are visited in order.
 *
 * Batched prefill equals sequential decode ("Architecture" page, "The forward
 * pass"): here that holds by construction, because every vector is computed
 * on its own.
 *
 * Mixture of experts ("Models and formats" page, "Architectures": a router
 * picks k of n experts per token from stacked 3-D tensors; gpt-oss has a bias
 * on every expert projection): each (token, slot) multiplies its expert's
 * matrix; with gates, the k slot outputs are combined in slot order.
 */
#include "oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

static int weight_type_ok(int t)
{
    return t == ORC_Q4_0 || t == ORC_Q5_0 || t == ORC_Q8_0 || t == ORC_MXFP4 || t == ORC_Q4_K || t == ORC_Q6_K ||
           t == ORC_Q4_1 || t == ORC_Q5_1 || t == ORC_Q5_K || t == ORC_Q2_K || t == ORC_Q3_K || t == ORC_Q8_1;
}

/* The 8-bit activation format that pairs with a weight format: the same block
 * length, so that weight block b meets activation block b. */
static int paired_act(int wtype) { return orc_block_elems(wtype) == 32 ? ORC_Q8_0 : ORC_Q8_K; }

int orc_block_dots(int wtype, const uint8_t* W, int64_t rows, int64_t cols,
                   const uint8_t* xq, int64_t n_vec, int64_t* out)
{
    if (!weight_type_ok(wtype)) return ORC_EUNSUP;
    int64_t bs = orc_block_elems(wtype), bb = orc_block_bytes(wtype);
    int at = paired_act(wtype);
    int64_t ab = orc_block_bytes(at);
    if (cols % bs) return ORC_ESHAPE;
    int64_t nb = cols / bs;
    orc_block wb;
    int32_t q[256];
    double dx;
    for (int64_t v = 0; v < n_vec; v++)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t b = 0; b < nb; b++) {
                orc_decode_block(wtype, W + (r * nb + b) * bb, &wb);
                orc_decode_act_block(at, xq + (v * nb + b) * ab, q, &dx, NULL);
                int64_t S = 0, Mn = 0;
                for (int i = 0; i < bs; i++) {
                    S += (int64_t)wb.sub_scale[i] * wb.code[i] * q[i];
                    Mn += (int64_t)wb.sub_min[i] * q[i];
                }
                int64_t* o = out + ((v * rows + r) * nb + b) * 2;
                o[0] = S;
                o[1] = Mn;
            }
    return ORC_OK;
}

/* One output: row `wrow` (nb blocks) against activation vector `xv`. */
static int dot_row(int wtype, int atype, const uint8_t* wrow, int64_t cols, const uint8_t* xv,
                   double* y, double* yabs)
{
    if (orc_plain_bytes(wtype)) {
        /* plain weights against fp32 activations: the definition, in fp64; against
           bf16 activations (the prefill product) the weight is first rounded to
           bf16 from its fp32 value, as the bf16 tile holds it */
        double acc = 0.0, aabs = 0.0;
        for (int64_t c = 0; c < cols; c++) {
            double p;
            if (atype == ORC_BF16) {
                const uint16_t xb = (uint16_t)(xv[2 * c] | (xv[2 * c + 1] << 8));
                const float wf = (float)orc_plain_weight(wtype, wrow, c);
                p = orc_bf16_to_f64(orc_f32_to_bf16_rn(wf)) * orc_bf16_to_f64(xb);
            } else {
                float xf;
                memcpy(&xf, xv + 4 * c, 4);
                p = orc_plain_weight(wtype, wrow, c) * (double)xf;
            }
            acc += p;
            aabs += fabs(p);
        }
        *y = acc;
        if (yabs) *yabs = aabs;
        return ORC_OK;
    }
    int64_t bs = orc_block_elems(wtype), bb = orc_block_bytes(wtype);
    int64_t nb = cols / bs;
    orc_block wb;
    double acc = 0.0, aabs = 0.0;
    if (atype == ORC_MXFP8) {
        /* block-scaled 8-bit activations: every product is exact in fp64 */
        for (int64_t b = 0; b < nb; b++) {
            orc_decode_block(wtype, wrow + b * bb, &wb);
            for (int i = 0; i < 32; i++) {
                const double p = orc_block_weight(&wb, i) * orc_mxfp8_value(xv + b * 33, i);
                acc += p;
                aabs += fabs(p);
            }
        }
    } else if (atype == ORC_F32 || atype == ORC_BF16) {
        for (int64_t b = 0; b < nb; b++) {
            orc_decode_block(wtype, wrow + b * bb, &wb);
            for (int i = 0; i < bs; i++) {
                int64_t c = b * bs + i;
                double w, xh;
                if (atype == ORC_F32) {
                    float xf;
                    memcpy(&xf, xv + 4 * c, 4);
                    w = orc_block_weight(&wb, i);
                    xh = (double)xf;
                } else {
                    uint16_t xb = (uint16_t)(xv[2 * c] | (xv[2 * c + 1] << 8));
                    /* the tile holds bf16(fp32 weight): two roundings for Q4_K, one or none otherwise */
                    float wf = (float)orc_block_weight(&wb, i);
                    w = orc_bf16_to_f64(orc_f32_to_bf16_rn(wf));
                    xh = orc_bf16_to_f64(xb);
                }
                acc += w * xh;
                aabs += fabs(w * xh);
            }
        }
    } else {
        int64_t ab = orc_block_bytes(atype);
        int32_t q[256];
        double dx;
        for (int64_t b = 0; b < nb; b++) {
            orc_decode_block(wtype, wrow + b * bb, &wb);
            orc_decode_act_block(atype, xv + b * ab, q, &dx, NULL);
            int64_t S = 0, Mn = 0;
            for (int i = 0; i < bs; i++) {
                S += (int64_t)wb.sub_scale[i] * wb.code[i] * q[i];
                Mn += (int64_t)wb.sub_min[i] * q[i];
                aabs += fabs(orc_block_weight(&wb, i) * dx * (double)q[i]);
            }
            if (S > INT32_MAX || S < INT32_MIN || Mn > INT32_MAX || Mn < INT32_MIN) return ORC_ERANGE;
            acc += dx * (wb.d * (double)S - wb.dmin * (double)Mn);
        }
    }
    *y = acc;
    if (yabs) *yabs = aabs;
    return ORC_OK;
}

static int64_t act_row_bytes(int atype, int64_t cols)
{
    if (atype == ORC_F32) return 4 * cols;
    if (atype == ORC_BF16) return 2 * cols;
    return cols / orc_block_elems(atype) * orc_block_bytes(atype);
}

static int64_t weight_row_bytes(int wtype, int64_t cols)
{
    if (orc_plain_bytes(wtype)) return cols * orc_plain_bytes(wtype);
    return cols / orc_block_elems(wtype) * orc_block_bytes(wtype);
}

static int check_pair(int wtype, int atype, int64_t cols)
{
    if (orc_plain_bytes(wtype)) return ((atype == ORC_F32 || atype == ORC_BF16) && cols > 0) ? ORC_OK : ORC_EUNSUP;
    if (!weight_type_ok(wtype)) return ORC_EUNSUP;
    if (atype == ORC_MXFP8 && orc_block_elems(wtype) != 32) return ORC_EUNSUP;
    if (atype != ORC_F32 && atype != ORC_BF16 && atype != ORC_MXFP8 && atype != paired_act(wtype)) return ORC_EUNSUP;
    if (cols <= 0 || cols % orc_block_elems(wtype)) return ORC_ESHAPE;
    return ORC_OK;
}

int orc_matvec(int wtype, int atype, const uint8_t* W, int64_t rows, int64_t cols,
               const void* x, int64_t n_vec, const int64_t* row_ids, int64_t n_rows,
               double* y, double* yabs)
{
    int rc = check_pair(wtype, atype, cols);
    if (rc) return rc;
    if (rows < 0 || n_vec < 0) return ORC_EINVAL;
    if (!row_ids) n_rows = rows;
    int64_t rb = weight_row_bytes(wtype, cols);
    int64_t xb = act_row_bytes(atype, cols);
    const uint8_t* X = (const uint8_t*)x;
    for (int64_t v = 0; v < n_vec; v++)
        for (int64_t j = 0; j < n_rows; j++) {
            int64_t r = row_ids ? row_ids[j] : j;
            if (r < 0 || r >= rows) return ORC_EINVAL;
            rc = dot_row(wtype, atype, W + r * rb, cols, X + v * xb, &y[v * n_rows + j],
                         yabs ? &yabs[v * n_rows + j] : NULL);
            if (rc) return rc;
        }
    return ORC_OK;
}

int orc_moe(int wtype, int atype, const uint8_t* W3d, int64_t n_expert,
            int64_t rows, int64_t cols, const int32_t* ids, const float* gates,
            int64_t k, const void* x, int64_t n_tok, const float* bias,
            double* y, double* yabs)
{
    int rc = check_pair(wtype, atype, cols);
    if (rc) return rc;
    if (n_expert <= 0 || rows < 0 || k <= 0 || n_tok < 0) return ORC_EINVAL;
    int64_t rb = weight_row_bytes(wtype, cols);
    int64_t xb = act_row_bytes(atype, cols);
    const uint8_t* X = (const uint8_t*)x;
    for (int64_t t = 0; t < n_tok; t++) {
        for (int64_t r = 0; r < rows; r++) {
            double comb = 0.0, comb_abs = 0.0;
            for (int64_t s = 0; s < k; s++) {
                int64_t e = ids[t * k + s];
                if (e < 0 || e >= n_expert) return ORC_ERANGE;
                const uint8_t* wrow = W3d + (e * rows + r) * rb;
                const uint8_t* xv = gates ? X + (t * k + s) * xb : X + t * xb;
                double v, va;
                rc = dot_row(wtype, atype, wrow, cols, xv, &v, &va);
                if (rc) return rc;
                if (bias) {
                    v += (double)bias[e * rows + r];
                    va += fabs((double)bias[e * rows + r]);
                }
                if (gates) {
                    double g = (double)gates[t * k + s];
                    comb += g * v;
                    comb_abs += fabs(g) * va;
                } else {
                    y[(t * k + s) * rows + r] = v;
                    if (yabs) yabs[(t * k + s) * rows + r] = va;
                }
            }
            if (gates) {
                y[t * rows + r] = comb;
                if (yabs) yabs[t * rows + r] = comb_abs;
            }
        }
    }
    return ORC_OK;
}
