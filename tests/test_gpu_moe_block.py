"""GPU parity of the whole mixture-of-experts block (router -> top k -> gate_up ->
clipped SwiGLU -> down) against the CPU oracle.

Bars:
  ids    bit-exact (the router's logit order is fixed, so the top-k decision is
         the same on both sides);
  gates  relative error <= (k + 8) * 2^-23 (fp32 exp, slot-order sum and one
         division against the oracle's fp64 softmax);
  y      |y - y_oracle| <= 1e-4 * sum_s g_s (sum|w*xhat| + |b|) + A, where A
         carries the difference of the activations h into the down projection:
         the GPU computes h in fp32 from its own fp32 gate_up outputs, the oracle
         in fp64 from exact ones.  With dh the bound on that difference (gate_up
         outputs within EPS_Y1 of their sums of magnitudes -- 20x the largest
         error the up-form expert parity sees -- propagated through the
         SwiGLU's derivative, which is 0 where the clip holds, plus a few
         roundings of h), A = sum_s g_s |W_down| (dh + a step where the rounding
         of h can go either way: one code step d of the 8-bit block, or one
         bf16 unit), computed from the oracle's own values.  Each case prints
         the largest err/bar and A/bar."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import TOL, dev, host, orc_t, workspace

pytestmark = pytest.mark.gpu

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16, MXFP4_R = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
Q5_K, MXFP8 = 16, 18
ALPHA, LIMIT = 1.702, 7.0
EPS_Y1 = 2e-6


def block_inputs(wt, E, hidden, inter, n_tok, seed):
    return dict(
        x=synth.activations(n_tok, hidden, seed=seed),
        Wr=synth.router_weights(E, hidden, seed=seed),
        br=synth.bias(1, E, seed=seed, tensor_id=4001)[0],
        Wgu=synth.weights(wt, E * 2 * inter, hidden, seed=seed, tensor_id=11),
        bgu=synth.bias(E, 2 * inter, seed=seed, tensor_id=12),
        Wd=synth.weights(wt, E * hidden, inter, seed=seed, tensor_id=13),
        bd=synth.bias(E, hidden, seed=seed, tensor_id=14),
    )


def experts_dev(qmv, wt, W, n_rows, cols):
    """Device experts: the GGUF rows, or for MXFP4_R their qmv_repack output."""
    Wd = dev(W)
    if wt != MXFP4_R:
        return Wd
    Wr = torch.empty(n_rows * qmv.qmv_row_bytes(MXFP4_R, cols), dtype=torch.uint8, device="cuda")
    qmv.qmv_repack(MXFP4, Wd, n_rows, cols, Wr)
    return Wr


def run_block(qmv, wt, at, E, k, hidden, inter, inp, n_tok, biases=True):
    fmt = qmv.FMT(wt, at)
    y = torch.full((n_tok, hidden), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((n_tok, k), -7, dtype=torch.int32, device="cuda")
    gates = torch.full((n_tok, k), float("nan"), dtype=torch.float32, device="cuda")
    need = qmv.qmv_moe_block_workspace_size(fmt, E, k, hidden, inter, n_tok)
    Wgu = experts_dev(qmv, wt, inp["Wgu"], E * 2 * inter, hidden)
    Wd = experts_dev(qmv, wt, inp["Wd"], E * hidden, inter)
    b = (lambda a: dev(a)) if biases else (lambda a: None)
    with workspace(qmv, need):
        qmv.qmv_moe_block(fmt, E, k, hidden, inter, dev(inp["Wr"]), b(inp["br"]), Wgu, b(inp["bgu"]), Wd,
                          b(inp["bd"]), ALPHA, LIMIT, dev(inp["x"]), n_tok, y, ids, gates)
        qmv.qmv_get_status()
        return host(y), host(ids), host(gates)


def _nearest_half_distance(v):
    return np.abs(v - np.floor(v) - 0.5)


def propagation_allowance(orc, wt, at, E, k, hidden, inter, ids, gates, det):
    """A[t][r] of the module docstring, from the oracle's y1, y1abs and h."""
    y1, y1abs, h = det["y1"], det["y1abs"], det["h"].astype(np.float64)
    g, u = y1[..., :inter], y1[..., inter:]
    gc = np.minimum(g, LIMIT)
    uc = np.clip(u, -LIMIT, LIMIT)
    dg, du = EPS_Y1 * y1abs[..., :inter], EPS_Y1 * y1abs[..., inter:]
    # d/dg (g sigmoid(alpha g)) = s'(alpha g) with s(z) = z sigmoid(z), and |s'| <= 1.1
    # everywhere, <= e^z2 (1 + |z1|) on [z1, z2] below -1; both derivatives vanish
    # where the clip holds for every value within the error
    z1, z2 = ALPHA * (gc - dg), ALPHA * (gc + dg)
    ds = np.where(z2 < -1.0, np.exp(np.minimum(z2, 0.0)) * (1.0 + np.abs(z1)), 1.1)
    dh_dg = np.where(g - dg > LIMIT, 0.0, ds * (np.abs(uc) + du + 1.0))
    sig_hi = 1.0 / (1.0 + np.exp(-np.clip(z2, -700, 700)))
    dh_du = np.where(np.abs(u) - du > LIMIT, 0.0, (np.abs(gc) + dg) * sig_hi)
    dh = dh_dg * dg + dh_du * du + 16 * 2.0 ** -24 * np.abs(h)
    step = np.zeros_like(h)
    if at in (Q8_0, Q8_K):
        bs = 32 if at == Q8_0 else 256
        hb, dhb = h.reshape(h.shape[:-1] + (-1, bs)), dh.reshape(dh.shape[:-1] + (-1, bs))
        amax = np.abs(hb).max(axis=-1, keepdims=True)
        dmax = dhb.max(axis=-1, keepdims=True)
        safe = np.where(amax > 0, amax, 1.0)
        v = hb * 127.0 / safe
        dv = (127.0 * dhb + np.abs(v) * dmax) / safe
        flip = _nearest_half_distance(v) <= dv
        stepb = np.where(flip, amax / 127.0, 0.0)
        # x-hat = d q moves with d: |h| dmax / amax; and a Q8_0 scale whose fp16
        # rounding can go either way moves the whole block by 2^-10 relative
        dhb = dhb + np.abs(hb) * dmax / safe
        if at == Q8_0:
            d32 = (amax / 127.0)
            ulp = 2.0 ** (np.floor(np.log2(np.where(d32 > 0, d32, 1.0))) - 10)
            amb16 = _nearest_half_distance(d32 / ulp) * ulp <= dmax / 127.0
            stepb = stepb + np.where(amb16, np.abs(hb) * 2.0 ** -10, 0.0)
        step = stepb.reshape(h.shape)
        dh = dhb.reshape(h.shape)
        n_flag = int(flip.sum())
    elif at == MXFP8:
        hb, dhb = h.reshape(h.shape[:-1] + (-1, 32)), dh.reshape(dh.shape[:-1] + (-1, 32))
        amax = np.abs(hb).max(axis=-1, keepdims=True)
        dmax = dhb.max(axis=-1, keepdims=True)
        lg = np.floor(np.log2(np.where(amax > 0, amax, 1.0)))
        E = np.maximum(lg - 8, -127)
        v = np.abs(hb) * np.exp2(-E)
        sp = np.where(v < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3))
        frac = v / sp
        near = np.abs(frac - np.floor(frac) - 0.5) * sp * np.exp2(E) <= dhb
        flip = near & (v < 448)
        # a block whose largest magnitude is within reach of a power of two may
        # take the neighbouring scale: then any code may move (clamping included)
        amb = (amax - np.exp2(lg) <= dmax) | (np.exp2(lg + 1) - amax <= dmax)
        stepb = np.where(flip, sp * np.exp2(E), 0.0) + np.where(amb, np.abs(hb) * 0.125 + 2 * sp * np.exp2(E), 0.0)
        step = stepb.reshape(h.shape)
        n_flag = int(flip.sum()) + int(amb.sum()) * 32
    elif at == BF16:
        hf = h.astype(np.float32)
        lo = (hf.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
        ulp = np.abs(((hf.view(np.uint32) & np.uint32(0xFFFF0000)) + np.uint32(0x10000)).view(np.float32)
                     .astype(np.float64) - lo)
        mid = lo + np.sign(h) * ulp / 2
        flip = np.abs(h - mid) <= dh
        step = np.where(flip, ulp, 0.0)
        n_flag = int(flip.sum())
    else:
        n_flag = 0
    a = dh + step                                      # [n_tok][k][inter]
    n_tok = ids.shape[0]
    A = np.zeros((n_tok, hidden))
    geo = MXFP4 if wt == MXFP4_R else wt
    for e in np.unique(ids):
        rb = orc.row_bytes(orc_t(geo), inter)
        Wd_bytes = det["Wd"][e * hidden * rb:(e + 1) * hidden * rb]
        Dabs = np.abs(orc.dequant(orc_t(geo), Wd_bytes, hidden, inter).astype(np.float64))
        for t, s in zip(*np.nonzero(ids == e)):
            A[t] += np.float32(gates[t, s]) * (Dabs @ a[t, s])
    return A, n_flag


def check_block(qmv, orc, wt, at, E, k, hidden, inter, n_tok, seed=0, inp=None, biases=True):
    inp = inp or block_inputs(MXFP4 if wt == MXFP4_R else wt, E, hidden, inter, n_tok, seed)
    y, ids, gates = run_block(qmv, wt, at, E, k, hidden, inter, inp, n_tok, biases)
    geo = MXFP4 if wt == MXFP4_R else wt
    ow, oa = orc_t(geo), orc_t(at)
    B = (lambda a: a) if biases else (lambda a: None)
    yr, yabs, ids_r, gates_r, det = orc.moe_block(ow, oa, inp["x"], inp["Wr"], B(inp["br"]), inp["Wgu"],
                                                  B(inp["bgu"]), inp["Wd"], B(inp["bd"]), E, k, hidden, inter,
                                                  ALPHA, LIMIT, detail=True)
    assert np.array_equal(ids, ids_r), "top-k ids differ"
    rel = np.abs(gates.astype(np.float64) - gates_r) / gates_r
    assert rel.max() <= (k + 8) * 2.0 ** -23, f"gates: max relative error {rel.max():.3g}"
    det["Wd"] = inp["Wd"]
    A, n_flag = propagation_allowance(orc, wt, at, E, k, hidden, inter, ids_r, gates_r, det)
    err = np.abs(y.astype(np.float64) - yr)
    bound = TOL * yabs + A
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} outputs out of tolerance; worst err/bound "
                           f"{(err / np.maximum(bound, 1e-300)).max():.3g}; ambiguous roundings {n_flag}")
    return (float((err / np.maximum(TOL * yabs, 1e-300)).max()), float((A / np.maximum(TOL * yabs, 1e-300)).max()),
            n_flag)


CASES = [(Q4_0, F32), (Q8_0, F32), (Q4_K, F32), (Q6_K, F32), (MXFP4, F32), (Q5_K, F32),
         (Q4_0, Q8_0), (Q5_0, Q8_0), (MXFP4, Q8_0), (Q4_K, Q8_K), (Q6_K, Q8_K),
         (MXFP4, BF16), (MXFP4_R, BF16), (MXFP4, MXFP8), (MXFP4_R, MXFP8)]


@pytest.mark.parametrize("wt,at", CASES)
@pytest.mark.parametrize("n_tok", [1, 13])
def test_block_parity(qmv, orc, wt, at, n_tok):
    E, k = 32, 4
    hidden, inter = (512, 256)
    used, extra, n_flag = check_block(qmv, orc, wt, at, E, k, hidden, inter, n_tok, seed=n_tok)
    print(f"{wt}/{at} n_tok={n_tok}: err/bar {used:.3g}, allowance/bar {extra:.3g}, ambiguous roundings {n_flag}")


def test_block_without_biases(qmv, orc):
    check_block(qmv, orc, Q8_0, F32, 16, 2, 256, 128, 5, seed=3, biases=False)


@pytest.mark.parametrize("at", [F32, Q8_0, BF16, MXFP8])
def test_block_gpt_oss_shapes(qmv, orc, at):
    """gpt-oss-sized experts (hidden = inter = 2880, 32 experts, 4 per token)."""
    used, extra, n_flag = check_block(qmv, orc, MXFP4, at, 32, 4, 2880, 2880, 3, seed=9)
    print(f"gpt-oss shapes {at}: err/bar {used:.3g}, allowance/bar {extra:.3g}, ambiguous roundings {n_flag}")


def test_router_ties_go_to_the_lower_id(qmv, orc):
    E, k, hidden, inter, n_tok = 16, 4, 256, 64, 9
    inp = block_inputs(Q8_0, E, hidden, inter, n_tok, 4)
    Wr, br = inp["Wr"].copy(), inp["br"].copy()
    Wr[5], br[5] = Wr[2], br[2]          # experts 2 and 5, and 7 and 11, score the same
    Wr[11], br[11] = Wr[7], br[7]
    x = inp["x"].copy()
    # steer every token towards the tied experts
    x[:] = (Wr[2] + Wr[7]) * 40 + x * 0.01
    inp.update(Wr=Wr, br=br, x=x)
    y, ids, gates = run_block(qmv, Q8_0, F32, E, k, hidden, inter, inp, n_tok)
    for t in range(n_tok):
        row = list(ids[t])
        assert set(row) == {2, 5, 7, 11}
        assert row.index(2) < row.index(5) and row.index(7) < row.index(11)
    check_block(qmv, orc, Q8_0, F32, E, k, hidden, inter, n_tok, inp=inp)


def test_all_logits_equal(qmv, orc):
    """Zero router weights and bias: every logit ties, ids are 0..k-1, gates 1/k."""
    E, k, hidden, inter, n_tok = 8, 3, 64, 32, 4
    inp = block_inputs(Q4_0, E, hidden, inter, n_tok, 6)
    inp["Wr"][:] = 0
    inp["br"][:] = 0
    y, ids, gates = run_block(qmv, Q4_0, F32, E, k, hidden, inter, inp, n_tok)
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (n_tok, 1)))
    assert np.allclose(gates, 1.0 / k, rtol=4 * 2.0 ** -23, atol=0)
    check_block(qmv, orc, Q4_0, F32, E, k, hidden, inter, n_tok, inp=inp)


@pytest.mark.parametrize("E,k", [(1, 1), (1024, 64), (130, 7)])
def test_expert_count_edges(qmv, orc, E, k):
    check_block(qmv, orc, Q8_0, F32, E, k, 64, 32, 3, seed=E)


def test_empty_and_refusals(qmv):
    fmt = qmv.FMT(Q8_0, F32)
    E, k, hidden, inter, n_tok = 8, 2, 64, 32, 3
    inp = block_inputs(Q8_0, E, hidden, inter, n_tok, 1)
    args = dict(Wr=dev(inp["Wr"]), Wgu=dev(inp["Wgu"]), Wd=dev(inp["Wd"]), x=dev(inp["x"]))
    # no tokens: a no-op, even without x, y, ids and gates
    assert qmv.qmv_moe_block(fmt, E, k, hidden, inter, args["Wr"], None, args["Wgu"], None, args["Wd"], None,
                             ALPHA, LIMIT, None, 0, None, None, None) == 0
    y = torch.empty((n_tok, hidden), dtype=torch.float32, device="cuda")
    ids = torch.empty((n_tok, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((n_tok, k), dtype=torch.float32, device="cuda")
    qmv.qmv_set_workspace(None, 0)
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_moe_block(fmt, E, k, hidden, inter, args["Wr"], None, args["Wgu"], None, args["Wd"], None, ALPHA,
                          LIMIT, args["x"], n_tok, y, ids, gates)
    assert e.value.code == qmv.ERR_WORKSPACE
