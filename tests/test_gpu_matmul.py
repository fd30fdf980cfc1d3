"""GPU parity of the prefill GEMM (Q4_K weights, bf16 activations, tcgen05)
against the CPU oracle, which multiplies bf16(w) by the bf16 activations in
fp64.  Bar: |Y - Y_oracle| <= 1e-4 * sum|bf16(w) x| for every output checked.
Invariant: prefill equals row-by-row decode ("Architecture" page, "The forward
pass") within the bf16 rounding of the weights."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host, workspace

pytestmark = pytest.mark.gpu

Q4_K, F32, BF16 = 4, 8, 9


def bf16_x(m, cols, seed):
    x = synth.activations(m, cols, seed=seed, tensor_id=m + cols)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    return xb, xb.view(torch.int16).numpy()


def run_matmul(qmv, Wd, rows, cols, xb, m):
    Y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    qmv.qmv_matmul(qmv.FMT(Q4_K, BF16), Wd, rows, cols, xb.cuda(), Y, m)
    return host(Y)


@pytest.mark.parametrize("rows,cols,m", [(128, 256, 256), (300, 512, 1), (256, 1024, 100), (130, 768, 300),
                                         (512, 2048, 513)])
def test_matmul_bf16_parity(qmv, orc, rows, cols, m):
    """Small shapes covering ragged row tiles (130, 300), ragged token tiles
    (1, 100, 300, 513) and several super-blocks per row; every output checked."""
    W = synth.weights(Q4_K, rows, cols, seed=7, tensor_id=rows)
    xb, xbits = bf16_x(m, cols, 7)
    Y = run_matmul(qmv, dev(W), rows, cols, xb, m)
    yref, yabs = orc.matvec(Q4_K, BF16, W, rows, cols, xbits, m)
    assert_close(Y, yref, yabs, what=f"{rows}x{cols} m={m}")
    qmv.qmv_get_status()


@pytest.mark.parametrize("rows,cols,m", [(200, 8192, 300), (1024, 8704, 77), (96, 16384, 1)])
def test_matmul_k_split_parity(qmv, orc, rows, cols, m):
    """Rows much shorter than K (cols >= 8192 and >= 2 rows) run as two K halves on
    different SMs that add into a zeroed Y: every output checked, repeated calls
    bit-identical (two addends commute, whichever lands first), and a token's
    outputs the same whatever m is (the split follows the weight's shape)."""
    W = synth.weights(Q4_K, rows, cols, seed=8, tensor_id=rows + cols)
    Wd = dev(W)
    xb, xbits = bf16_x(m, cols, 8)
    Y = run_matmul(qmv, Wd, rows, cols, xb, m)
    yref, yabs = orc.matvec(Q4_K, BF16, W, rows, cols, xbits, m)
    assert_close(Y, yref, yabs, what=f"{rows}x{cols} m={m}")
    for _ in range(3):
        assert np.array_equal(run_matmul(qmv, Wd, rows, cols, xb, m).view(np.uint32), Y.view(np.uint32))
    one = run_matmul(qmv, Wd, rows, cols, xb[m - 1:m], 1)
    assert np.array_equal(one[0].view(np.uint32), Y[m - 1].view(np.uint32))
    qmv.qmv_get_status()


@pytest.mark.parametrize("rows,m", [(9700, 500), (19500, 200), (9600, 300)])
def test_matmul_many_tiles_parity(qmv, orc, rows, m):
    """More tiles than SMs: 256-token tiles (the wide tile of the large prefill
    shapes; 9700 x 500, and 19500 x 200 in partly empty 256-token tiles) and
    128-token tiles with two per CTA on some SMs (9600 x 300: 75 row tiles give
    fewer than one 256-token tile per SM, so 225 tiles of 128 tokens), each with a
    ragged last row tile and a ragged last token tile; every output checked."""
    cols = 256
    W = synth.weights(Q4_K, rows, cols, seed=8, tensor_id=rows)
    xb, xbits = bf16_x(m, cols, 8)
    Y = run_matmul(qmv, dev(W), rows, cols, xb, m)
    yref, yabs = orc.matvec(Q4_K, BF16, W, rows, cols, xbits, m)
    assert_close(Y, yref, yabs, what=f"{rows}x{cols} m={m}")
    qmv.qmv_get_status()


@pytest.mark.parametrize("rows,cols,m", [(14336, 4096, 512), (4096, 14336, 512), (14336, 4096, 2048),
                                         (4096, 14336, 2048)])
def test_matmul_config_shapes_sampled(qmv, orc, rows, cols, m):
    """The prefill configuration's shapes at full size; the oracle checks 40
    sampled rows for 64 sampled tokens (first and last of each included)."""
    W = synth.weights(Q4_K, rows, cols, seed=3, tensor_id=rows * 3 + cols)
    xb, xbits = bf16_x(m, cols, 3)
    Y = run_matmul(qmv, dev(W), rows, cols, xb, m)
    assert np.isfinite(Y).all()
    g = np.random.default_rng(rows + m)
    rids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 38)]))
    toks = np.unique(np.concatenate([[0, m - 1], g.integers(0, m, 62)]))
    yref, yabs = orc.matvec(Q4_K, BF16, W, rows, cols, xbits[toks], len(toks), row_ids=rids)
    assert_close(Y[np.ix_(toks, rids)], yref, yabs, what=f"{rows}x{cols} m={m}")
    qmv.qmv_get_status()


def test_matmul_equals_rowwise_decode(qmv, orc):
    """Prefill vs sequential decode of the same bf16 token values: the GEMM
    multiplies bf16-rounded weights, the A32 matvec exact ones, so they may
    differ by at most the weight rounding, 2^-9 * sum|w x| (plus fp32 noise)."""
    rows, cols, m = 512, 2048, 64
    W = synth.weights(Q4_K, rows, cols, seed=11)
    Wd = dev(W)
    xb, _ = bf16_x(m, cols, 11)
    Y = run_matmul(qmv, Wd, rows, cols, xb, m)
    xf = xb.float().cuda()
    yv = torch.empty((m, rows), dtype=torch.float32, device="cuda")
    for t in range(m):   # one token at a time, as decode runs
        qmv.qmv_matvec(qmv.FMT(Q4_K, F32), Wd, rows, cols, xf[t], yv[t], 1)
    yv = host(yv)
    _, yabs = orc.matvec(Q4_K, F32, W, rows, cols, xf.cpu().numpy(), m)
    assert (np.abs(Y - yv) <= (2.0 ** -9 + 2e-6) * yabs).all()


def test_matmul_edge_cases(qmv, orc):
    rows, cols = 128, 256
    W = dev(synth.weights(Q4_K, rows, cols, seed=1))
    # m = 0 and rows = 0 do nothing
    Y = torch.full((1, rows), 5.0, device="cuda")
    qmv.qmv_matmul(qmv.FMT(Q4_K, BF16), W, rows, cols, torch.zeros((1, cols), dtype=torch.bfloat16, device="cuda"), Y, 0)
    qmv.qmv_matmul(qmv.FMT(Q4_K, BF16), W, 0, cols, torch.zeros((1, cols), dtype=torch.bfloat16, device="cuda"), Y, 1)
    assert (host(Y) == 5).all()
    # zero activations give exact zeros
    assert (run_matmul(qmv, W, rows, cols, torch.zeros((3, cols), dtype=torch.bfloat16), 3) == 0).all()
    # unsupported pairs and shapes are refused before any launch
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matmul(qmv.FMT(Q4_K, F32), W, rows, cols, W, Y, 1)
    assert e.value.code == qmv.ERR_UNSUPPORTED
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matmul(qmv.FMT(Q4_K, BF16), W, rows, 300, W, Y, 1)
    assert e.value.code == qmv.ERR_SHAPE
    qmv.qmv_get_status()


Q8_K = 7


def run_w4a8(qmv, Wd, rows, cols, xq_dev, m):
    Y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    need = qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(Q4_K, Q8_K), rows, cols, m)
    with workspace(qmv, need):
        qmv.qmv_matmul(qmv.FMT(Q4_K, Q8_K), Wd, rows, cols, xq_dev, Y, m)
        qmv.qmv_get_status()
    return host(Y)


@pytest.mark.parametrize("rows,cols,m", [(128, 256, 1), (300, 1024, 37), (130, 768, 300), (1000, 512, 129),
                                         (9700, 256, 500)])
def test_matmul_w4a8_parity(qmv, orc, rows, cols, m):
    """W4A8 prefill (Q4_K x Q8_K) on the tensor cores, every output against the
    oracle's exact integer dots: ragged row tiles (130, 300, 1000, 9700), ragged
    token tiles (1, 37, 129, 300, 500), one to four super-blocks per row, and
    more tiles than SMs (9700 x 500); plus every token's row within the same
    bar of its own W4A8 decode (both exact in integers; only the fp32
    accumulation order differs)."""
    W = synth.weights(Q4_K, rows, cols, seed=12, tensor_id=rows)
    Wd = dev(W)
    x = synth.activations(m, cols, seed=12)
    xq = orc.quantize_act(Q8_K, x)
    Y = run_w4a8(qmv, Wd, rows, cols, dev(xq), m)
    yref, yabs = orc.matvec(Q4_K, Q8_K, W, rows, cols, xq, m)
    assert_close(Y, yref, yabs, what=f"w4a8 {rows}x{cols} m={m}")
    xqd = dev(xq)
    toks = sorted({0, m // 2, m - 1})
    for t in toks:
        y1 = torch.empty((1, rows), dtype=torch.float32, device="cuda")
        qmv.qmv_matvec(qmv.FMT(Q4_K, Q8_K), Wd, rows, cols, xqd[t], y1, 1)
        assert_close(Y[t], host(y1)[0].astype(np.float64), yabs[t], what=f"prefill vs decode token {t}")
    qmv.qmv_get_status()


def test_matmul_w4a8_integer_exactness(qmv, orc):
    """The tensor cores return the integer sums exactly.  Weights with d = 1,
    dmin = 1, every sub-block scale and min 63 and every code 15, against
    activations whose codes are all +127 in the first half of each super-block
    and -127 in the second (scale d_x = 1/127 in fp32): each super-block's S is
    +15.36M - 15.36M and its Mn +/- sums that cancel, so every output is an
    exact small integer combination that any lost low bit would change.  Plus
    rows and tokens with mixed codes, compared exactly where the oracle's value
    is an integer below 2^24."""
    rows, cols, m = 256, 1024, 130
    blk = np.zeros(rows * cols // 256, dtype=synth.block_dtype(Q4_K))
    blk["d"] = np.float16(1.0)
    blk["dmin"] = np.float16(1.0)
    blk["scales"] = 0xFF              # every 6-bit scale and min = 63
    blk["qs"] = 0xFF                  # every code 15
    g = np.random.default_rng(77)
    mix = blk.reshape(rows, -1)[rows // 2:]
    mix["qs"] = g.integers(0, 256, mix["qs"].shape, dtype=np.uint8)
    mix["scales"] = g.integers(0, 256, mix["scales"].shape, dtype=np.uint8)
    W = blk.view(np.uint8).reshape(-1)
    x = np.empty((m, cols), dtype=np.float32)
    x.reshape(m, -1, 2, 128)[:, :, 0, :] = 1.0
    x.reshape(m, -1, 2, 128)[:, :, 1, :] = -1.0
    x[m // 2:] = g.integers(-127, 128, (m - m // 2, cols)).astype(np.float32) / np.float32(127.0)
    x[m // 2:, 0] = 1.0               # amax = 1, d_x = 1/127
    xq = orc.quantize_act(Q8_K, x)
    Y = run_w4a8(qmv, dev(W), rows, cols, dev(xq), m)
    yref, yabs = orc.matvec(Q4_K, Q8_K, W, rows, cols, xq, m)
    assert_close(Y, yref, yabs, what="w4a8 adversarial")
    # the all-maximal quarter: S cancels per super-block, leaving -d_x*dmin*Mn
    # with Mn = 63 * (sum of the 16 bsums) = 0, so exactly zero
    assert (Y[: m // 2, : rows // 2] == 0).all() and (yref[: m // 2, : rows // 2] == 0).all()
