"""GPU parity of the MXFP8 activation path: the quantiser bit for bit, and the
grouped mixture-of-experts GEMM on the block-scaled MMA (MXFP4 experts x
MXFP8 tokens) against the oracle's exact products.

Bar (per output): |y - y_oracle| <= 1e-4 * sum|w * xhat| (+ |b|), x-hat the
MXFP8 value the oracle's quantiser gives; with gates, gate-weighted."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host, orc_t, workspace

pytestmark = pytest.mark.gpu

MXFP4, MXFP4_R, MXFP8 = 6, 10, 18
O_MXFP8 = 17   # the oracle's number


def quant_gpu(qmv, x):
    xd = dev(np.ascontiguousarray(x, dtype=np.float32))
    out = torch.empty(x.size // 32 * 33, dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_act(MXFP8, xd, out, x.size)
    return host(out)


def adversarial_rows(g, n, cols):
    x = g.standard_normal((n, cols)).astype(np.float32)
    x[0] = 0.0                                                    # zero blocks
    x[1] *= np.float32(2.0 ** -135)                               # subnormal inputs, scale held at -127
    x[2] *= np.float32(1e30)                                      # large scales
    x[3] = np.exp2(g.integers(-20, 20, cols)).astype(np.float32)  # powers of two (exact codes, amax on 2^n)
    x[4, ::32] = 1.9999                                           # clamped to 448
    # ties of the E4M3 grid: midpoints between codes at the block's scale
    vals = torch.arange(0x7f, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (vals[1:] + vals[:-1]) / 2
    t = g.choice(mids[mids > 0], cols) * np.where(g.random(cols) < 0.5, -1, 1)
    t[::32] = 256.0                                               # amax 256 keeps the scale at 2^0
    x[5] = t.astype(np.float32)
    return x


@pytest.mark.parametrize("n,cols", [(1, 32), (7, 2880), (64, 4096)])
def test_quantize_mxfp8_bit_exact(qmv, orc, n, cols):
    g = np.random.default_rng(cols + n)
    x = adversarial_rows(g, max(n, 6), cols)[:max(n, 6)] if n >= 6 else g.standard_normal((n, cols)).astype(np.float32)
    got = quant_gpu(qmv, x)
    want = orc.quantize_act(O_MXFP8, x).reshape(-1)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"


def moe_case(qmv, orc, wt, E, rows, cols, n_tok, k, seed, down):
    W3 = synth.weights(MXFP4, E * rows, cols, seed=seed, tensor_id=1)
    ids, gates = synth.router(n_tok, E, k, seed=seed + 1)
    b = synth.bias(E, rows, seed=seed + 2)
    x = synth.activations(n_tok * (k if down else 1), cols, seed=seed + 3) * np.float32(2.0)
    x = x.reshape(n_tok, k, cols) if down else x
    W3d = dev(W3)
    if wt == MXFP4_R:
        Wr = torch.empty(E * rows * qmv.qmv_row_bytes(MXFP4_R, cols), dtype=torch.uint8, device="cuda")
        qmv.qmv_repack(MXFP4, W3d, E * rows, cols, Wr)
        W3d = Wr
    fmt = qmv.FMT(wt, MXFP8)
    shape = (n_tok, rows) if down else (n_tok, k, rows)
    y = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    with workspace(qmv, qmv.qmv_workspace_size(qmv.OP_MOE, fmt, rows, cols, n_tok * k)):
        qmv.qmv_moe_matvec(fmt, W3d, E, rows, cols, dev(ids), dev(gates) if down else None, k, dev(x), y, n_tok,
                           dev(b))
        qmv.qmv_get_status()
        got = host(y)
    xq = orc.quantize_act(O_MXFP8, x)
    return got, (W3, ids, gates, b, xq)


@pytest.mark.parametrize("wt", [MXFP4, MXFP4_R])
@pytest.mark.parametrize("cols", [128, 2880, 4096])
@pytest.mark.parametrize("down", [False, True])
def test_moe_mx_parity(qmv, orc, wt, cols, down):
    E, rows, k, n_tok = 6, 256, 3, 9
    got, (W3, ids, gates, b, xq) = moe_case(qmv, orc, wt, E, rows, cols, n_tok, k, cols + 7, down)
    yref, yabs = orc.moe(MXFP4, O_MXFP8, W3, E, rows, cols, ids, gates if down else None, k, xq, n_tok, bias=b)
    assert_close(got, yref, yabs, what=f"cols={cols} down={down}")


def test_moe_mx_many_tiles(qmv, orc):
    """Experts with several 128-token tiles, ragged rows (not a multiple of 128)."""
    E, rows, cols, k, n_tok = 3, 200, 512, 2, 300
    got, (W3, ids, gates, b, xq) = moe_case(qmv, orc, MXFP4, E, rows, cols, n_tok, k, 31, False)
    yref, yabs = orc.moe(MXFP4, O_MXFP8, W3, E, rows, cols, ids, None, k, xq, n_tok, bias=b)
    assert_close(got, yref, yabs, what="many tiles")


@pytest.mark.parametrize("n_tok", [64, 1024])
def test_moe_mx_gpt_oss_sampled(qmv, orc, n_tok):
    """gpt-oss-20B-shaped experts (32 x 5760 x 2880 gate_up, 32 x 2880 x 2880
    down, top 4): sampled tokens and rows against the oracle's matvec on each
    routed expert."""
    E, k = 32, 4
    g = np.random.default_rng(n_tok + 5)
    for rows, cols, down in ((5760, 2880, False), (2880, 2880, True)):
        got, (W3, ids, gates, b, xq) = moe_case(qmv, orc, MXFP4_R, E, rows, cols, n_tok, k, rows + n_tok, down)
        toks = np.unique(np.concatenate([[0, n_tok - 1], g.integers(0, n_tok, 4)]))
        rids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 24)]))
        rb = orc.row_bytes(MXFP4, cols)
        xq3 = xq.reshape(n_tok, k if down else 1, -1)
        for t in toks:
            per, pera = [], []
            for s in range(k):
                e = int(ids[t, s])
                We = W3[e * rows * rb:(e + 1) * rows * rb]
                yv, ya = orc.matvec(MXFP4, O_MXFP8, We, rows, cols, xq3[t, s if down else 0][None], 1, row_ids=rids)
                per.append(yv[0] + b[e, rids])
                pera.append(ya[0] + np.abs(b[e, rids]))
            if down:
                gt = gates[t].astype(np.float32).astype(np.float64)
                yref = sum(gt[s] * per[s] for s in range(k))
                yabs = sum(abs(gt[s]) * pera[s] for s in range(k))
                assert_close(got[t, rids], yref, yabs, what=f"down t={t}")
            else:
                assert_close(got[t][:, rids], np.stack(per), np.stack(pera), what=f"up t={t}")


def test_moe_mx_refusals(qmv):
    fmt = qmv.FMT(MXFP4, MXFP8)
    with pytest.raises(qmv.QmvError) as e:   # cols beyond the staged scale rows
        qmv.qmv_moe_matvec(fmt, 4096, 2, 64, 4128, 4096, None, 1, 4096, 4096, 1)
    assert e.value.code == qmv.ERR_SHAPE
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_moe_matvec(qmv.FMT(4, MXFP8), 4096, 2, 64, 256, 4096, None, 1, 4096, 4096, 1)   # Q4_K experts
    assert e.value.code == qmv.ERR_UNSUPPORTED
