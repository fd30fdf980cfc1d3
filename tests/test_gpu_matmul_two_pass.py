"""GPU parity of the prefill product for every weight format without a fused
tile dequantiser (all GGUF block types but Q4_K, and plain F32/F16/BF16 rows)
with bf16 activations: one pass writes bf16(w) tiles into the workspace, a
bf16 x bf16 tcgen05 GEMM multiplies them.  The oracle multiplies bf16(w), w
rounded from its fp32 value, by the bf16 activations in fp64.  Bar:
|Y - Y_oracle| <= 1e-4 * sum|bf16(w) x| for every output checked
("Architecture" page, "The two phases": prefill multiplies a whole prompt)."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host, orc_t, workspace

pytestmark = pytest.mark.gpu

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, F32, BF16, MXFP4_R = 1, 2, 3, 4, 5, 6, 8, 9, 10
Q4_1, Q5_1, Q8_1, Q2_K, Q3_K, Q5_K, F16 = 11, 12, 13, 14, 15, 16, 17
TYPES = [Q4_0, Q5_0, Q8_0, Q6_K, MXFP4, Q4_1, Q5_1, Q8_1, Q2_K, Q3_K, Q5_K, F32, F16, BF16]
K_TYPES = {Q6_K, Q2_K, Q3_K, Q5_K}


def bf16_x(m, cols, seed):
    x = synth.activations(m, cols, seed=seed, tensor_id=m + cols)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    return xb, xb.view(torch.int16).numpy()


def run(qmv, t, Wd, rows, cols, xb, m):
    Y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    need = qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(t, BF16), rows, cols, m)
    assert need >= rows * cols * 2
    with workspace(qmv, need):
        qmv.qmv_matmul(qmv.FMT(t, BF16), Wd, rows, cols, xb.cuda(), Y, m)
        qmv.qmv_get_status()
    return host(Y)


def check(qmv, orc, t, rows, cols, m, seed):
    W = synth.weights(t, rows, cols, seed=seed, tensor_id=rows + t)
    xb, xbits = bf16_x(m, cols, seed)
    Y = run(qmv, t, dev(W), rows, cols, xb, m)
    yref, yabs = orc.matvec(orc_t(t), BF16, W, rows, cols, xbits, m)
    assert_close(Y, yref, yabs, what=f"type {t} {rows}x{cols} m={m}")


@pytest.mark.parametrize("t", TYPES)
@pytest.mark.parametrize("rows,cols,m", [(130, 512, 300), (300, 768, 1), (256, 1024, 129)])
def test_two_pass_parity(qmv, orc, t, rows, cols, m):
    """Ragged row tiles (130, 300), ragged token tiles (1, 129, 300), several
    128-k stages per tile; every output checked."""
    check(qmv, orc, t, rows, cols, m, 21)


@pytest.mark.parametrize("t,cols", [(Q8_0, 32), (Q4_0, 96), (MXFP4, 160), (F32, 8), (BF16, 40), (F16, 1032),
                                    (Q6_K, 256), (Q3_K, 1280)])
def test_two_pass_ragged_k(qmv, orc, t, cols):
    """K that is not a multiple of the 128-k stage (and for the plain rows not
    of a 64-k box): the tensor maps fill the missing k with zeros."""
    check(qmv, orc, t, 200, cols, 77, 22)


@pytest.mark.parametrize("t,rows,m", [(Q8_0, 9700, 500), (Q5_0, 19500, 200), (Q6_K, 4000, 1100)])
def test_two_pass_many_tiles(qmv, orc, t, rows, m):
    """More tiles than SMs with 256-token tiles (9700 x 500, 4000 x 1100) and
    with 128-token tiles (19500 x 200), ragged in both directions."""
    check(qmv, orc, t, rows, 256, m, 23)


@pytest.mark.parametrize("t,rows,cols,m", [(Q5_0, 4864, 896, 512), (Q8_0, 896, 4864, 512), (Q8_0, 151936, 896, 64),
                                           (Q5_0, 896, 896, 2048), (Q6_K, 4096, 14336, 512)])
def test_two_pass_model_shapes_sampled(qmv, orc, t, rows, cols, m):
    """Qwen2-0.5B-shaped matrices in its GGUF formats (the layers in Q5_0, the
    vocabulary projection in Q8_0: 896 is not a multiple of the 256-element
    K-quant super-block) and a 14336-wide Q6_K down projection: 40 sampled rows
    for 64 sampled tokens checked by the oracle, first and last of each
    included."""
    W = synth.weights(t, rows, cols, seed=24, tensor_id=rows * 3 + cols)
    xb, xbits = bf16_x(m, cols, 24)
    Y = run(qmv, t, dev(W), rows, cols, xb, m)
    assert np.isfinite(Y).all()
    g = np.random.default_rng(rows + m)
    rids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 38)]))
    toks = np.unique(np.concatenate([[0, m - 1], g.integers(0, m, 62)]))
    yref, yabs = orc.matvec(orc_t(t), BF16, W, rows, cols, xbits[toks], len(toks), row_ids=rids)
    assert_close(Y[np.ix_(toks, rids)], yref, yabs, what=f"type {t} {rows}x{cols} m={m}")


def test_two_pass_deterministic_and_token_independent(qmv):
    """Repeated calls are bit-identical, and a token's outputs do not depend on
    how many tokens share the call (no split of K, one accumulation order)."""
    rows, cols, m = 1000, 1536, 300
    Wd = dev(synth.weights(Q5_0, rows, cols, seed=25))
    xb, _ = bf16_x(m, cols, 25)
    Y = run(qmv, Q5_0, Wd, rows, cols, xb, m)
    for _ in range(2):
        assert np.array_equal(run(qmv, Q5_0, Wd, rows, cols, xb, m).view(np.uint32), Y.view(np.uint32))
    for t0, n in [(0, 1), (299, 1), (17, 40)]:
        part = run(qmv, Q5_0, Wd, rows, cols, xb[t0:t0 + n], n)
        assert np.array_equal(part.view(np.uint32), Y[t0:t0 + n].view(np.uint32))


def test_two_pass_equals_rowwise_decode(qmv, orc):
    """Prefill against sequential fp32 decode of the same bf16 token values: the
    GEMM multiplies bf16-rounded weights and the A32 matvec exact ones, so they
    differ by at most the weight rounding, 2^-9 * sum|w x| (plus fp32 noise)."""
    rows, cols, m = 512, 2048, 48
    W = synth.weights(Q8_0, rows, cols, seed=26)
    Wd = dev(W)
    xb, _ = bf16_x(m, cols, 26)
    Y = run(qmv, Q8_0, Wd, rows, cols, xb, m)
    xf = xb.float().cuda()
    yv = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    for t in range(m):
        qmv.qmv_matvec(qmv.FMT(Q8_0, F32), Wd, rows, cols, xf[t], yv[t], 1)
    yv = host(yv)
    _, yabs = orc.matvec(Q8_0, F32, W, rows, cols, xf.cpu().numpy(), m)
    assert (np.abs(Y - yv) <= (2.0 ** -9 + 2e-6) * yabs).all()


def test_two_pass_edge_cases_and_refusals(qmv):
    rows, cols = 128, 256
    W = dev(synth.weights(Q8_0, rows, cols, seed=27))
    Y = torch.full((1, rows), 5.0, device="cuda")
    x1 = torch.zeros((1, cols), dtype=torch.bfloat16, device="cuda")
    # m = 0 and rows = 0 do nothing, and need no workspace
    qmv.qmv_matmul(qmv.FMT(Q8_0, BF16), W, rows, cols, x1, Y, 0)
    qmv.qmv_matmul(qmv.FMT(Q8_0, BF16), W, 0, cols, x1, Y, 1)
    assert (host(Y) == 5).all()
    # zero activations give exact zeros
    assert (run(qmv, Q8_0, W, rows, cols, torch.zeros((3, cols), dtype=torch.bfloat16), 3) == 0).all()
    # no workspace, or too little, is refused before any launch
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matmul(qmv.FMT(Q8_0, BF16), W, rows, cols, x1, Y, 1)
    assert e.value.code == qmv.ERR_WORKSPACE
    with workspace(qmv, rows * cols * 2 - 512):
        with pytest.raises(qmv.QmvError) as e:
            qmv.qmv_matmul(qmv.FMT(Q8_0, BF16), W, rows, cols, x1, Y, 1)
        assert e.value.code == qmv.ERR_WORKSPACE
    with workspace(qmv, 1 << 20):
        # plain rows must be 16-byte rows of bf16 tiles: cols a multiple of 8
        Wf = dev(synth.weights(F32, rows, 12, seed=1))
        with pytest.raises(qmv.QmvError) as e:
            qmv.qmv_matmul(qmv.FMT(F32, BF16), Wf, rows, 12, torch.zeros((1, 12), dtype=torch.bfloat16,
                                                                          device="cuda"), Y, 1)
        assert e.value.code == qmv.ERR_SHAPE
        # repacked MXFP4 rows belong to the mixture of experts only; MXFP8 and
        # other activation types are not prefill formats
        for fmt in (qmv.FMT(MXFP4_R, BF16), qmv.FMT(Q8_0, F32), qmv.FMT(Q8_0, Q8_0)):
            with pytest.raises(qmv.QmvError) as e:
                qmv.qmv_matmul(fmt, W, rows, cols, x1, Y, 1)
            assert e.value.code == qmv.ERR_UNSUPPORTED
    assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(Q8_0, BF16), rows, cols, 1) >= rows * cols * 2
    assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(Q4_K, BF16), rows, cols, 1) == 0
    qmv.qmv_get_status()
