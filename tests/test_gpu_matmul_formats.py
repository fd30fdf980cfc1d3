"""GPU parity of the prefill product for the weight formats other than Q4_K
(Q4_0, Q5_0, Q8_0 and Q6_K rows of a whole number of 16 bytes dequantised
tile by tile into TMEM inside a tcgen05 GEMM; BF16 rows multiplied as they
are; the other types and row lengths converted to bf16 in the workspace
first), with bf16 activations.  The oracle
multiplies bf16(w), w rounded from its fp32 value, by the bf16 activations in
fp64.  Bar:
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
BB = {Q4_0: (32, 18), Q5_0: (32, 22), Q8_0: (32, 34), Q6_K: (256, 210)}


def two_pass(t, cols):
    """Whether the product converts the weights to bf16 in the workspace first
    (every type but Q4_K and BF16 rows, except Q4_0 / Q5_0 / Q8_0 / Q6_K rows of
    a whole number of 16 bytes, which are dequantised inside the GEMM)."""
    if t in (Q4_K, BF16):
        return False
    if t in BB:
        bs, bb = BB[t]
        return (cols // bs) * bb % 16 != 0
    return True


def bf16_x(m, cols, seed):
    x = synth.activations(m, cols, seed=seed, tensor_id=m + cols)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    return xb, xb.view(torch.int16).numpy()


def run(qmv, t, Wd, rows, cols, xb, m):
    Y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    need = qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(t, BF16), rows, cols, m)
    assert need == ((rows * cols * 2 + 255) // 256 * 256 if two_pass(t, cols) else 0)
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
def test_formats_parity(qmv, orc, t, rows, cols, m):
    """Ragged row tiles (130, 300), ragged token tiles (1, 129, 300), several
    128-k stages per tile; every output checked."""
    check(qmv, orc, t, rows, cols, m, 21)


@pytest.mark.parametrize("t,cols", [(Q8_0, 32), (Q4_0, 96), (Q5_0, 224), (Q8_0, 4064), (MXFP4, 160), (F32, 8),
                                    (BF16, 40), (F16, 1032), (Q6_K, 256), (Q3_K, 1280)])
def test_formats_ragged_k(qmv, orc, t, cols):
    """K that is not a multiple of the 128-k stage (and for the plain rows not
    of a 64-k box): the tensor maps fill the missing k with zeros."""
    check(qmv, orc, t, 200, cols, 77, 22)


@pytest.mark.parametrize("t,rows,cols,m", [(Q8_0, 9700, 256, 500), (Q5_0, 19500, 256, 200), (Q5_0, 9600, 256, 300),
                                           (Q6_K, 4000, 256, 1100), (Q6_K, 5000, 2048, 300), (Q4_0, 4000, 512, 1100),
                                           (BF16, 9700, 256, 600), (F16, 5000, 512, 700)])
def test_formats_many_tiles(qmv, orc, t, rows, cols, m):
    """More tiles than SMs with 256-token tiles (9700 x 500, 19500 x 200,
    4000 x 1100) and with 128-token tiles (9600 x 300: 225 tiles, two on some
    CTAs; 5000 x 300), ragged in both directions; Q6_K both in two passes
    (256 k: 210-byte rows) and inside the GEMM; the plain bf16 GEMM's two
    accumulators over several tiles per CTA (BF16 rows as they are, F16 rows
    through the workspace)."""
    check(qmv, orc, t, rows, cols, m, 23)


@pytest.mark.parametrize("t,rows,cols,m", [(Q6_K, 130, 2048, 300), (Q6_K, 300, 4096, 1), (Q6_K, 256, 6144, 129),
                                           (Q8_0, 129, 2304, 257), (Q5_0, 257, 1280, 33), (Q4_0, 1, 256, 5)])
def test_formats_fused_tiles(qmv, orc, t, rows, cols, m):
    """The tile dequantisers inside the GEMM: Q6_K rows of whole 16 bytes
    (cols a multiple of 2048; two A stages per super-block) and odd numbers of
    128-k stages for the 32-element formats, ragged rows and tokens."""
    check(qmv, orc, t, rows, cols, m, 29)


@pytest.mark.parametrize("t,rows,cols,m", [(Q5_0, 4864, 896, 512), (Q8_0, 896, 4864, 512), (Q8_0, 151936, 896, 64),
                                           (Q5_0, 896, 896, 2048), (Q6_K, 4096, 14336, 512),
                                           (BF16, 14336, 4096, 2048), (BF16, 4096, 14336, 512),
                                           (MXFP4, 14336, 4096, 512)])
def test_formats_model_shapes_sampled(qmv, orc, t, rows, cols, m):
    """Qwen2-0.5B-shaped matrices in its GGUF formats (the layers in Q5_0, the
    vocabulary projection in Q8_0: 896 is not a multiple of the 256-element
    K-quant super-block), a 14336-wide Q6_K down projection, and the
    configuration's full-size shapes as BF16 rows (the plain GEMM's 64-k stages
    at 256-token tiles, its 128-k stages at 128-token tiles) and as MXFP4 rows
    (two passes): 40 sampled rows for 64 sampled tokens checked by the oracle,
    first and last of each included."""
    W = synth.weights(t, rows, cols, seed=24, tensor_id=rows * 3 + cols)
    xb, xbits = bf16_x(m, cols, 24)
    Y = run(qmv, t, dev(W), rows, cols, xb, m)
    assert np.isfinite(Y).all()
    g = np.random.default_rng(rows + m)
    rids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 38)]))
    toks = np.unique(np.concatenate([[0, m - 1], g.integers(0, m, 62)]))
    yref, yabs = orc.matvec(orc_t(t), BF16, W, rows, cols, xbits[toks], len(toks), row_ids=rids)
    assert_close(Y[np.ix_(toks, rids)], yref, yabs, what=f"type {t} {rows}x{cols} m={m}")


def test_formats_deterministic_and_token_independent(qmv):
    """Repeated calls are bit-identical, and a token's outputs do not depend on
    how many tokens share the call (one accumulation order per output)."""
    rows, cols, m = 1000, 1536, 300
    Wd = dev(synth.weights(Q5_0, rows, cols, seed=25))
    xb, _ = bf16_x(m, cols, 25)
    Y = run(qmv, Q5_0, Wd, rows, cols, xb, m)
    for _ in range(2):
        assert np.array_equal(run(qmv, Q5_0, Wd, rows, cols, xb, m).view(np.uint32), Y.view(np.uint32))
    for t0, n in [(0, 1), (299, 1), (17, 40)]:
        part = run(qmv, Q5_0, Wd, rows, cols, xb[t0:t0 + n], n)
        assert np.array_equal(part.view(np.uint32), Y[t0:t0 + n].view(np.uint32))


@pytest.mark.parametrize("t,rows,cols,m", [(Q8_0, 200, 8192, 300), (Q6_K, 96, 16384, 1), (Q5_0, 1024, 8704, 77),
                                           (Q5_0, 896, 4864, 130), (Q8_0, 2600, 8192, 40)])
def test_formats_k_split(qmv, orc, t, rows, cols, m):
    """Rows much shorter than K: few row tiles run as four K parts on the CTAs
    of a thread-block cluster, summed in part order through its shared memory
    (200 x 8192, 96 x 16384, 1024 x 8704, the Qwen2-0.5B down projection 896 x
    4864 with unequal parts); more row tiles with cols >= 8192 and >= 2 rows as
    two halves adding into a zeroed Y (2600 x 8192).  Every output checked,
    repeated calls bit-identical, and the last token's outputs the same when it
    is multiplied alone (the split follows the weight's shape)."""
    W = synth.weights(t, rows, cols, seed=28, tensor_id=rows + cols)
    Wd = dev(W)
    xb, xbits = bf16_x(m, cols, 28)
    Y = run(qmv, t, Wd, rows, cols, xb, m)
    yref, yabs = orc.matvec(orc_t(t), BF16, W, rows, cols, xbits, m)
    assert_close(Y, yref, yabs, what=f"type {t} {rows}x{cols} m={m}")
    for _ in range(2):
        assert np.array_equal(run(qmv, t, Wd, rows, cols, xb, m).view(np.uint32), Y.view(np.uint32))
    one = run(qmv, t, Wd, rows, cols, xb[m - 1:m], 1)
    assert np.array_equal(one[0].view(np.uint32), Y[m - 1].view(np.uint32))


def test_formats_equals_rowwise_decode(qmv, orc):
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


def test_formats_edge_cases_and_refusals(qmv):
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
    # F32 / F16 rows without workspace, or with too little, are refused
    # before any launch; block types and BF16 rows need none
    Wf32 = dev(synth.weights(F32, rows, cols, seed=27))
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matmul(qmv.FMT(F32, BF16), Wf32, rows, cols, x1, Y, 1)
    assert e.value.code == qmv.ERR_WORKSPACE
    with workspace(qmv, rows * cols * 2 - 512):
        with pytest.raises(qmv.QmvError) as e:
            qmv.qmv_matmul(qmv.FMT(F32, BF16), Wf32, rows, cols, x1, Y, 1)
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
    assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(F16, BF16), rows, cols, 1) == rows * cols * 2
    for t in (Q4_0, Q5_0, Q8_0, BF16, Q4_K):
        assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(t, BF16), rows, cols, 1) == 0
    for t in (Q4_1, MXFP4, Q5_K, Q6_K):   # Q6_K: 256 k = 210 bytes per row
        assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(t, BF16), rows, cols, 1) == rows * cols * 2
    assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(Q6_K, BF16), rows, 2048, 1) == 0
    assert qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(Q8_0, BF16), rows, 896, 1) == rows * 896 * 2
    qmv.qmv_get_status()
