"""GPU parity of the mixture-of-experts matvec against the CPU oracle.

Bar (per output): |y - y_oracle| <= 1e-4 * sum_s g_s (sum|w*xhat| + |b|)
(gates taken as 1 in the up form)."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu

MXFP4, Q8_0, F32, Q4_K, Q8_K = 6, 3, 8, 4, 7


@pytest.fixture(scope="module")
def workspace(qmv):
    buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # 256 MB
    qmv.qmv_set_workspace(buf, buf.numel())
    yield buf
    qmv.qmv_set_workspace(None, 0)


def moe_inputs(t, E, rows, cols, n_tok, k, seed):
    W3 = synth.weights(t, E * rows, cols, seed=seed, tensor_id=1)
    ids, gates = synth.router(n_tok, E, k, seed=seed)
    b = synth.bias(E, rows, seed=seed)
    return W3, ids, gates, b


def run_moe(qmv, fmt, W3d, E, rows, cols, ids, gates, k, x, n_tok, bias):
    shape = (n_tok, k, rows) if gates is None else (n_tok, rows)
    y = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    qmv.qmv_moe_matvec(fmt, W3d, E, rows, cols, dev(ids), None if gates is None else dev(gates), k, x, y, n_tok,
                       None if bias is None else dev(bias))
    return host(y)


@pytest.mark.parametrize("t", [MXFP4, Q4_K])
@pytest.mark.parametrize("mode", ["A32", "A8", "A8q"])
def test_moe_small_parity(qmv, orc, workspace, t, mode):
    E, rows, k, n_tok = 6, 48, 3, 9
    cols = 256 if t == Q4_K else 128
    at = {"A32": F32, "A8": Q8_0 if t == MXFP4 else Q8_K, "A8q": Q8_0 if t == MXFP4 else Q8_K}[mode]
    flags = qmv.FLAG_QUANTIZE_X if mode == "A8q" else 0
    W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 5)
    W3d = dev(W3)
    # up form: x shared by the slots of a token
    x = synth.activations(n_tok, cols, seed=5)
    xin_o = orc.quantize_act(at, x) if at != F32 else x
    xin_g = dev(x) if (at == F32 or flags) else dev(xin_o)
    y = run_moe(qmv, qmv.FMT(t, at) | flags, W3d, E, rows, cols, ids, None, k, xin_g, n_tok, b)
    yref, yabs = orc.moe(t, at, W3, E, rows, cols, ids, None, k, xin_o, n_tok, bias=b)
    assert_close(y, yref, yabs, what=f"up {mode}")
    # down form: one input per slot, gate-weighted
    h = synth.activations(n_tok * k, cols, seed=6).reshape(n_tok, k, cols)
    hin_o = orc.quantize_act(at, h) if at != F32 else h
    hin_g = dev(h) if (at == F32 or flags) else dev(hin_o)
    y = run_moe(qmv, qmv.FMT(t, at) | flags, W3d, E, rows, cols, ids, gates, k, hin_g, n_tok, b)
    yref, yabs = orc.moe(t, at, W3, E, rows, cols, ids, gates, k, hin_o, n_tok, bias=b)
    assert_close(y, yref, yabs, what=f"down {mode}")
    qmv.qmv_get_status()


def oracle_sampled(orc, t, at, W3, E, rows, cols, ids, gates, k, x_o, toks, rids, bias, down):
    """Expected values for sampled tokens and rows, composed from the oracle's
    matvec on each routed expert's slice of the stacked tensor."""
    rb = orc.row_bytes(t, cols)
    outs, absd = [], []
    for tok in toks:
        per, pera = [], []
        for s in range(k):
            e = int(ids[tok, s])
            We = W3[e * rows * rb:(e + 1) * rows * rb]
            xv = x_o[tok, s:s + 1] if down else x_o[tok:tok + 1]
            yv, ya = orc.matvec(t, at, We, rows, cols, xv, 1, row_ids=rids)
            per.append(yv[0] + bias[e, rids])
            pera.append(ya[0] + np.abs(bias[e, rids]))
        if down:
            g = gates[tok].astype(np.float64)
            outs.append(sum(g[s] * per[s] for s in range(k)))
            absd.append(sum(abs(g[s]) * pera[s] for s in range(k)))
        else:
            outs.append(np.stack(per))
            absd.append(np.stack(pera))
    return np.stack(outs), np.stack(absd)


@pytest.mark.parametrize("n_tok", [1, 64, 1024])
def test_moe_gpt_oss_shapes_sampled(qmv, orc, workspace, n_tok):
    """gpt-oss-20B-shaped experts: 32 MXFP4 experts, gate_up 5760x2880 and
    down 2880x2880 with biases, top-4 routing; W4A8 with the activations
    quantised inside the kernels.  Sampled tokens and rows are checked."""
    E, k, t, at = 32, 4, MXFP4, Q8_0
    fl = qmv.FLAG_QUANTIZE_X
    g = np.random.default_rng(n_tok)
    for rows, cols, down in ((5760, 2880, False), (2880, 2880, True)):
        W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 20 + rows)
        x = synth.activations(n_tok * (k if down else 1), cols, seed=21)
        x = x.reshape(n_tok, k, cols) if down else x
        y = run_moe(qmv, qmv.FMT(t, at) | fl, dev(W3), E, rows, cols, ids, gates if down else None, k, dev(x),
                    n_tok, b)
        toks = np.unique(np.concatenate([[0, n_tok - 1], g.integers(0, n_tok, 4)]))
        rids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 30)]))
        x_o = orc.quantize_act(at, x)
        yref, yabs = oracle_sampled(orc, t, at, W3, E, rows, cols, ids, gates, k, x_o, toks, rids, b, down)
        ysel = y[toks][..., rids]
        assert_close(ysel, yref, yabs, what=f"n_tok={n_tok} down={down}")
    qmv.qmv_get_status()


def test_moe_routing_invariance(qmv, orc, workspace):
    """A token's expert outputs do not depend on which other tokens were routed
    with it: the 16-token call equals 16 single-token calls bit for bit."""
    E, rows, cols, k, n_tok, t = 8, 96, 256, 2, 16, MXFP4
    W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 9)
    W3d = dev(W3)
    x = synth.activations(n_tok, cols, seed=9)
    fmt = qmv.FMT(t, Q8_0) | qmv.FLAG_QUANTIZE_X
    y = run_moe(qmv, fmt, W3d, E, rows, cols, ids, None, k, dev(x), n_tok, b)
    for tok in (0, 5, 15):
        y1 = run_moe(qmv, fmt, W3d, E, rows, cols, ids[tok:tok + 1], None, k, dev(x[tok:tok + 1]), 1, b)
        assert np.array_equal(y1[0].view(np.uint32), y[tok].view(np.uint32))


def test_moe_bad_expert_and_workspace(qmv, orc, workspace):
    E, rows, cols, k, n_tok, t = 4, 32, 64, 2, 3, MXFP4
    W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 4)
    W3d = dev(W3)
    x = synth.activations(n_tok, cols, seed=4)
    bad = ids.copy()
    bad[1, 0] = 7   # out of range
    y = run_moe(qmv, qmv.FMT(t, F32), W3d, E, rows, cols, bad, None, k, dev(x), n_tok, b)
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_get_status()
    assert e.value.code == qmv.ERR_DEVICE_STATUS and "expert id" in str(e.value)
    yref, yabs = orc.moe(t, F32, W3, E, rows, cols, ids, None, k, x, n_tok, bias=b)
    ok = [(0, 0), (0, 1), (1, 1), (2, 0), (2, 1)]   # every slot but the bad one
    for tok, s in ok:
        assert_close(y[tok, s], yref[tok, s], yabs[tok, s])
    qmv.qmv_get_status()   # cleared
    # a workspace that is too small is refused before launching
    need = qmv.qmv_workspace_size(qmv.OP_MOE, qmv.FMT(t, F32), rows, cols, n_tok * k)
    assert need > 0
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    qmv.qmv_set_workspace(small, small.numel())
    try:
        with pytest.raises(qmv.QmvError) as e:
            run_moe(qmv, qmv.FMT(t, F32), W3d, E, rows, cols, ids, None, k, dev(x), n_tok, b)
        assert e.value.code == qmv.ERR_WORKSPACE
    finally:
        qmv.qmv_set_workspace(workspace, workspace.numel())


# ---- MXFP4 experts x bf16 activations: the grouped tensor-core GEMM ---------------
BF16 = 9


def bf16_rows(n, cols, seed):
    """bf16 activation rows (torch's round-to-nearest of N(0,1)) and their bit
    patterns for the oracle."""
    xb = torch.from_numpy(synth.activations(n, cols, seed=seed)).to(torch.bfloat16)
    return xb, xb.view(torch.int16).numpy()


MXFP4_R = 10


def repack_reference(W, rows, cols):
    """MXFP4 GGUF rows -> MXFP4_R rows, by a plain reshuffle: per row the 16
    code bytes of each block in block order, then the exponent bytes, then
    zeros up to a multiple of 16 bytes."""
    nblk = cols // 32
    blocks = W.reshape(rows, nblk, 17)
    rb = (17 * nblk + 15) // 16 * 16
    out = np.zeros((rows, rb), dtype=np.uint8)
    out[:, :16 * nblk] = blocks[:, :, 1:].reshape(rows, 16 * nblk)
    out[:, 16 * nblk:17 * nblk] = blocks[:, :, 0]
    return out.reshape(-1)


def experts_on_device(qmv, W3, n_rows, cols, repacked):
    """(device weights, weight type): the GGUF rows, or their qmv_repack output."""
    Wd = dev(W3)
    if not repacked:
        return Wd, MXFP4
    Wr = torch.empty(n_rows * qmv.qmv_row_bytes(MXFP4_R, cols), dtype=torch.uint8, device="cuda")
    qmv.qmv_repack(MXFP4, Wd, n_rows, cols, Wr)
    return Wr, MXFP4_R


@pytest.mark.parametrize("rows,cols", [(37, 544), (5, 32), (64, 2880)])
def test_repack_bytes(qmv, rows, cols):
    """qmv_repack writes exactly the reshuffled bytes (padding zeroed)."""
    W = synth.weights(MXFP4, rows, cols, seed=81, tensor_id=cols)
    assert qmv.qmv_row_bytes(MXFP4_R, cols) == (17 * (cols // 32) + 15) // 16 * 16
    Wr = torch.full((rows * qmv.qmv_row_bytes(MXFP4_R, cols),), 0xAB, dtype=torch.uint8, device="cuda")
    qmv.qmv_repack(MXFP4, dev(W), rows, cols, Wr)
    assert np.array_equal(host(Wr), repack_reference(W, rows, cols))


def test_repack_refusals(qmv):
    W = torch.zeros(4 * 144, dtype=torch.uint8, device="cuda")
    out = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmv.QmvError) as e:   # no repacked layout for Q4_K
        qmv.qmv_repack(Q4_K, W, 4, 256, out)
    assert e.value.code == qmv.ERR_UNSUPPORTED
    with pytest.raises(qmv.QmvError) as e:   # output overlapping the input
        qmv.qmv_repack(MXFP4, out, 4, 64, out[16:])
    assert e.value.code == qmv.ERR_INVALID_ARG
    y = torch.zeros((1, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(qmv.QmvError) as e:   # MXFP4_R is a MoE bf16 operand only
        qmv.qmv_matvec(qmv.FMT(MXFP4_R, Q8_0), out, 32, 64, y, y, 1)
    assert e.value.code == qmv.ERR_UNSUPPORTED
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_moe_matvec(qmv.FMT(MXFP4_R, Q8_0), out, 1, 32, 64, ids, None, 1, y, y, 1, None)
    assert e.value.code == qmv.ERR_UNSUPPORTED


@pytest.mark.parametrize("repacked", [False, True])
@pytest.mark.parametrize("rows,cols,n_tok", [(296, 544, 1), (128, 256, 37), (200, 2880, 9), (136, 320, 300)])
def test_moe_bf16_gemm_parity(qmv, orc, workspace, rows, cols, n_tok, repacked):
    """Ragged row tiles, an odd number of blocks per row (a half 64-k chunk and
    a short last raw stage), experts with more than one 128-token tile, both
    forms, with biases; GGUF rows and repacked MXFP4_R rows."""
    E, k, t = 8, 4, MXFP4
    W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 40 + cols)
    W3d, wt = experts_on_device(qmv, W3, E * rows, cols, repacked)
    fmt = qmv.FMT(wt, BF16)
    xb, xbits = bf16_rows(n_tok, cols, 41)
    y = run_moe(qmv, fmt, W3d, E, rows, cols, ids, None, k, xb.cuda(), n_tok, b)
    yref, yabs = orc.moe(t, BF16, W3, E, rows, cols, ids, None, k, xbits, n_tok, bias=b)
    assert_close(y, yref, yabs, what="up")
    hb, hbits = bf16_rows(n_tok * k, cols, 42)
    y = run_moe(qmv, fmt, W3d, E, rows, cols, ids, gates, k, hb.reshape(n_tok, k, cols).cuda(), n_tok, b)
    yref, yabs = orc.moe(t, BF16, W3, E, rows, cols, ids, gates, k, hbits.reshape(n_tok, k, cols), n_tok, bias=b)
    assert_close(y, yref, yabs, what="down")
    qmv.qmv_get_status()


@pytest.mark.parametrize("repacked", [False, True])
def test_moe_bf16_exponent_range(qmv, orc, workspace, repacked):
    """E8M0 exponents across 0..200: the table path (2..252) at both ends of its
    range and the exact fallback for the zero and subnormal scales (0, 1)."""
    E, rows, cols, k, n_tok, t = 4, 160, 512, 2, 20, MXFP4
    W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 50)
    blocks = W3.reshape(-1, 17)
    g = np.random.default_rng(50)
    blocks[:, 0] = g.integers(0, 201, size=blocks.shape[0], dtype=np.uint8)
    blocks[::7, 0] = 2
    blocks[3::11, 0] = g.integers(0, 2, size=blocks[3::11].shape[0], dtype=np.uint8)
    W3 = blocks.reshape(-1)
    xb, xbits = bf16_rows(n_tok, cols, 51)
    W3d, wt = experts_on_device(qmv, W3, E * rows, cols, repacked)
    y = run_moe(qmv, qmv.FMT(wt, BF16), W3d, E, rows, cols, ids, None, k, xb.cuda(), n_tok, None)
    yref, yabs = orc.moe(t, BF16, W3, E, rows, cols, ids, None, k, xbits, n_tok)
    assert_close(y, yref, yabs, what="exponents")
    qmv.qmv_get_status()


@pytest.mark.parametrize("repacked", [False, True])
@pytest.mark.parametrize("n_tok", [1, 64, 1024])
def test_moe_bf16_gpt_oss_shapes_sampled(qmv, orc, workspace, n_tok, repacked):
    """gpt-oss-20B-shaped experts with bf16 activations through the grouped
    GEMM: gate_up 5760x2880 (up form) and down 2880x2880 (gate-weighted),
    biases, top-4 of 32; sampled tokens and rows against the oracle."""
    E, k, t = 32, 4, MXFP4
    g = np.random.default_rng(100 + n_tok)
    for rows, cols, down in ((5760, 2880, False), (2880, 2880, True)):
        W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 60 + rows)
        xb, xbits = bf16_rows(n_tok * (k if down else 1), cols, 61)
        if down:
            xb, xbits = xb.reshape(n_tok, k, cols), xbits.reshape(n_tok, k, cols)
        W3d, wt = experts_on_device(qmv, W3, E * rows, cols, repacked)
        y = run_moe(qmv, qmv.FMT(wt, BF16), W3d, E, rows, cols, ids, gates if down else None, k, xb.cuda(),
                    n_tok, b)
        toks = np.unique(np.concatenate([[0, n_tok - 1], g.integers(0, n_tok, 4)]))
        rids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 30)]))
        yref, yabs = oracle_sampled(orc, t, BF16, W3, E, rows, cols, ids, gates, k, xbits, toks, rids, b, down)
        assert_close(y[toks][..., rids], yref, yabs, what=f"n_tok={n_tok} down={down}")
    qmv.qmv_get_status()


def test_moe_bf16_routing_invariance(qmv, orc, workspace):
    """A token's outputs from the grouped GEMM do not depend on the other
    tokens routed with it (its column of the expert's tile): a 200-token call
    equals single-token calls bit for bit."""
    E, rows, cols, k, n_tok, t = 4, 256, 512, 2, 200, MXFP4
    W3, ids, gates, b = moe_inputs(t, E, rows, cols, n_tok, k, 70)
    W3d = dev(W3)
    xb, _ = bf16_rows(n_tok, cols, 71)
    y = run_moe(qmv, qmv.FMT(t, BF16), W3d, E, rows, cols, ids, None, k, xb.cuda(), n_tok, b)
    for tok in (0, 77, 199):
        y1 = run_moe(qmv, qmv.FMT(t, BF16), W3d, E, rows, cols, ids[tok:tok + 1], None, k, xb[tok:tok + 1].cuda(),
                     1, b)
        assert np.array_equal(y1[0].view(np.uint32), y[tok].view(np.uint32))


def test_moe_bf16_refusals(qmv, workspace):
    W = torch.zeros(64 * 17, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 2, 32), dtype=torch.float32, device="cuda")
    ids = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(qmv.QmvError) as e:   # BF16 activations are for MXFP4 experts only
        qmv.qmv_moe_matvec(qmv.FMT(Q4_K, BF16), W, 1, 32, 256, ids, None, 2, x, y, 1, None)
    assert e.value.code == qmv.ERR_UNSUPPORTED
    with pytest.raises(qmv.QmvError) as e:   # nothing to quantise
        qmv.qmv_moe_matvec(qmv.FMT(MXFP4, BF16) | qmv.FLAG_QUANTIZE_X, W, 1, 32, 64, ids, None, 2, x, y, 1, None)
    assert e.value.code == qmv.ERR_INVALID_ARG
