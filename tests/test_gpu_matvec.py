"""GPU parity of the activation quantiser, dequantisation, the W4A8 integer
block dots and the decode matvec against the CPU oracle, through the C ABI.

Bars: bit-exact for quantised activations, dequantised weights and integer
dots; |y - y_oracle| <= 1e-4 * sum|w*xhat| for every matvec output; decode
bit-identical whatever n_vec (batch invariance)."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host, orc_t

pytestmark = pytest.mark.gpu

W32 = [1, 2, 3, 6, 11, 12, 13]   # Q4_0, Q5_0, Q8_0, MXFP4, Q4_1, Q5_1, Q8_1
WK = [4, 5, 14, 15, 16]          # Q4_K, Q6_K, Q2_K, Q3_K, Q5_K
PLAIN = [8, 17, 9]               # F32, F16, BF16 weights (fp32 activations only)
ALLW = W32 + WK


def act_for(t):
    return 3 if t in W32 else 7   # Q8_0 / Q8_K


def shapes_for(t):
    if t in W32:
        # ragged tile (37 rows), C1/C2 width, several K-chunks with a ragged last chunk
        return [(1, 32), (37, 96), (300, 896), (45, 8288)]
    return [(1, 256), (37, 512), (70, 4096), (19, 14336)]


@pytest.mark.parametrize("atype", [3, 7])
@pytest.mark.parametrize("n", [32 * 7, 256 * 3, 256 * 64])
def test_quantize_act_bit_exact(qmv, orc, atype, n):
    if n % (32 if atype == 3 else 256):
        pytest.skip("n not a multiple of the block")
    g = np.random.default_rng(n + atype)
    x = (g.standard_normal(n) * np.exp2(g.integers(-6, 6, n // 32).repeat(32))).astype(np.float32)
    x[:32] = 0.0                      # an all-zero block
    x[32:64] = np.float32(2.5)        # ties of x*id
    ref = orc.quantize_act(atype, x)
    xq = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_act(atype, dev(x), xq, n)
    assert np.array_equal(host(xq), ref)


@pytest.mark.parametrize("atype", [3, 7])
def test_quantize_act_scale_below_2_pow_minus_128(qmv, orc, atype):
    """Blocks whose amax/127 is below 2^-128, so that 1/d overflows: the codes
    are round(x / d) (zeros stay 0), byte for byte the oracle's, both from
    qmv_quantize_act and when the matvec quantises its fp32 input itself
    (QMV_FLAG_QUANTIZE_X gives the same output bits)."""
    bs = 32 if atype == 3 else 256
    n_vec, cols = 3, 1024
    g = np.random.default_rng(31)
    x = (g.uniform(-1, 1, (n_vec, cols)) * 1e-37).astype(np.float32)
    x[:, ::5] = 0.0
    x[0, :bs] = g.standard_normal(bs).astype(np.float32)     # one block with an ordinary scale
    x[2, bs:2 * bs] = 0.0                                      # and an all-zero block
    ref = orc.quantize_act(atype, x)
    xd = dev(x)
    xq = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_act(atype, xd, xq, x.size)
    assert np.array_equal(host(xq), ref.reshape(-1))
    t = 2 if atype == 3 else 4
    rows = 70
    W = dev(synth.weights(t, rows, cols, seed=32))
    y1 = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    y2 = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, atype), W, rows, cols, xq, y1, n_vec)
    qmv.qmv_matvec(qmv.FMT(t, atype) | qmv.FLAG_QUANTIZE_X, W, rows, cols, xd, y2, n_vec)
    assert np.array_equal(host(y1).view(np.uint32), host(y2).view(np.uint32))
    if atype == 7:
        assert (host(y1)[1:] != 0).any()   # the tiny Q8_K scales still reach the output


@pytest.mark.parametrize("t", ALLW)
def test_dequantize_bit_exact(qmv, orc, t):
    for rows, cols in shapes_for(t)[:3]:
        W = synth.weights(t, rows, cols, seed=1, tensor_id=t)
        ref = orc.dequant(orc_t(t), W, rows, cols)
        out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
        qmv.qmv_dequantize(t, dev(W), rows, cols, out)
        assert np.array_equal(host(out).view(np.uint32), ref.view(np.uint32)), (t, rows, cols)


@pytest.mark.parametrize("t", ALLW)
def test_block_dots_bit_exact(qmv, orc, t):
    rows, cols = shapes_for(t)[1]
    n_vec = 3
    W = synth.weights(t, rows, cols, seed=2, tensor_id=t)
    x = synth.activations(n_vec, cols, seed=2)
    xq = orc.quantize_act(act_for(t), x)
    ref = orc.block_dots(orc_t(t), W, rows, cols, xq, n_vec)
    assert np.abs(ref).max() < 2 ** 31
    out = torch.empty(ref.shape, dtype=torch.int32, device="cuda")
    qmv.qmv_block_dots(t, dev(W), rows, cols, dev(xq), n_vec, out)
    assert np.array_equal(host(out).astype(np.int64), ref)


@pytest.mark.parametrize("a8", [True, False], ids=["A8", "A32"])
@pytest.mark.parametrize("t", ALLW)
def test_matvec_parity(qmv, orc, t, a8):
    at = act_for(t) if a8 else 8
    for rows, cols in shapes_for(t):
        for n_vec in (1, 3, 16):
            W = synth.weights(t, rows, cols, seed=3, tensor_id=rows)
            x = synth.activations(n_vec, cols, seed=3, tensor_id=cols)
            xin = orc.quantize_act(at, x) if a8 else x
            yref, yabs = orc.matvec(orc_t(t), at, W, rows, cols, xin, n_vec)
            y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_matvec(qmv.FMT(t, at), dev(W), rows, cols, dev(xin), y, n_vec)
            assert_close(host(y), yref, yabs, what=f"t={t} a8={a8} {rows}x{cols} n_vec={n_vec}")
    qmv.qmv_get_status()


@pytest.mark.parametrize("a8", [True, False], ids=["A8", "A32"])
@pytest.mark.parametrize("t", ALLW)
def test_matvec_batch_invariance(qmv, orc, t, a8):
    """Output (v, r) is bit-identical whether v is decoded alone or with others
    (the pages' determinism claim: "regardless of ... batch composition")."""
    at = act_for(t) if a8 else 8
    rows, cols = shapes_for(t)[2]
    n_vec = 20
    W = dev(synth.weights(t, rows, cols, seed=4))
    x = synth.activations(n_vec, cols, seed=4)
    xin = orc.quantize_act(at, x) if a8 else x
    xd = dev(xin)
    y = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, at), W, rows, cols, xd, y, n_vec)
    ys = host(y)
    for v in (0, 7, 19):
        y1 = torch.empty((1, rows), dtype=torch.float32, device="cuda")
        qmv.qmv_matvec(qmv.FMT(t, at), W, rows, cols, xd[v], y1, 1)
        assert np.array_equal(host(y1)[0].view(np.uint32), ys[v].view(np.uint32)), v
    # and across vector groups of a different composition
    y5 = torch.empty((5, rows), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, at), W, rows, cols, xd[3:8], y5, 5)
    assert np.array_equal(host(y5).view(np.uint32), ys[3:8].view(np.uint32))


def test_matvec_quantised_pipeline(qmv, orc):
    """fp32 x -> qmv_quantize_act -> qmv_matvec on the device equals the oracle's
    quantise-then-multiply (the W4A8 hot path end to end)."""
    t, rows, cols, n_vec = 2, 256, 896, 8
    W = synth.weights(t, rows, cols, seed=5)
    x = synth.activations(n_vec, cols, seed=5)
    xq = torch.empty(n_vec * 28 * 34, dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_act(3, dev(x), xq, n_vec * cols)
    y = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, 3), dev(W), rows, cols, xq, y, n_vec)
    yref, yabs = orc.matvec(orc_t(t), 3, W, rows, cols, orc.quantize_act(3, x), n_vec)
    assert_close(host(y), yref, yabs)


def test_matvec_edge_cases(qmv, orc):
    # odd MXFP4 rows: the matrix ends off a 16-byte boundary (ragged tail path)
    for rows in (1, 15, 17, 33):
        t, cols = 6, 32
        W = synth.weights(t, rows, cols, seed=rows)
        x = synth.activations(2, cols, seed=rows)
        yref, yabs = orc.matvec(orc_t(t), 8, W, rows, cols, x, 2)
        y = torch.empty((2, rows), dtype=torch.float32, device="cuda")
        qmv.qmv_matvec(qmv.FMT(t, 8), dev(W), rows, cols, dev(x), y, 2)
        assert_close(host(y), yref, yabs, what=f"mxfp4 rows={rows}")
    # zero activations give exact zeros
    t, rows, cols = 4, 40, 512
    W = dev(synth.weights(t, rows, cols, seed=9))
    xq = dev(orc.quantize_act(7, np.zeros((2, cols), np.float32)))
    y = torch.full((2, rows), 7.0, dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, 7), W, rows, cols, xq, y, 2)
    assert (host(y) == 0).all()
    # n_vec = 0 and rows = 0 are no-ops that leave y alone
    y = torch.full((1, rows), 7.0, dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, 7), W, rows, cols, xq, y, 0)
    qmv.qmv_matvec(qmv.FMT(t, 7), W, 0, cols, xq, y, 1)
    assert (host(y) == 7).all()
    # misaligned weights are refused, not read
    buf = torch.zeros(100000, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matvec(qmv.FMT(1, 8), buf.data_ptr() + 8, 4, 32, dev(np.zeros(32, np.float32)), y, 1)
    assert e.value.code == qmv.ERR_ALIGN
    qmv.qmv_get_status()


# ---- the configurations' full shapes, checked on sampled rows ----------------------

CONFIG_SHAPES = [
    # single Q4_0 GEMV 896x896 (A32 and A8)
    (1, 896, 896, (1,)),
    # Qwen2.5-0.5B-shaped decode: q/o, k/v, gate/up, down in Q5_0; lm_head in Q8_0
    (2, 896, 896, (1, 8)), (2, 128, 896, (1, 8)), (2, 4864, 896, (1, 8)), (2, 896, 4864, (1, 8)),
    (3, 151936, 896, (1, 8)),
    # Llama-3-8B-shaped decode in K-quants
    (4, 4096, 4096, (1, 4, 16)), (4, 1024, 4096, (1, 16)), (4, 14336, 4096, (1, 16)),
    (4, 4096, 14336, (1, 4, 16)), (5, 128256, 4096, (1, 4, 16)),
]


@pytest.mark.parametrize("cfg", CONFIG_SHAPES, ids=lambda c: f"t{c[0]}_{c[1]}x{c[2]}")
def test_config_shapes_sampled(qmv, orc, cfg):
    t, rows, cols, nvecs = cfg
    W = synth.weights(t, rows, cols, seed=1, tensor_id=rows * 7 + cols)
    Wd = dev(W)
    g = np.random.default_rng(rows + cols)
    ids = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, 48)]))
    for a8 in (True, False):
        at = act_for(t) if a8 else 8
        for n_vec in nvecs:
            x = synth.activations(n_vec, cols, seed=1)
            xin = orc.quantize_act(at, x) if a8 else x
            y = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
            qmv.qmv_matvec(qmv.FMT(t, at), Wd, rows, cols, dev(xin), y, n_vec)
            yref, yabs = orc.matvec(orc_t(t), at, W, rows, cols, xin, n_vec, row_ids=ids)
            assert_close(host(y)[:, ids], yref, yabs, what=f"{cfg} a8={a8} n_vec={n_vec}")
    qmv.qmv_get_status()


@pytest.mark.parametrize("t", ALLW)
def test_quantize_x_flag_bit_identical(qmv, orc, t):
    """QMV_FLAG_QUANTIZE_X (quantise fp32 activations inside the matvec) gives
    the same bits as qmv_quantize_act followed by qmv_matvec.  The vector
    counts and widths reach every thread-per-block split of the in-kernel
    quantiser (8, 4, 2, 1 threads per 32-element block; 32, 16, 8 per 256)."""
    at = act_for(t)
    for (rows, cols), n_vec in [(rc, n) for rc in shapes_for(t)[1:] for n in (1, 2, 5)]:
        W = dev(synth.weights(t, rows, cols, seed=6))
        x = synth.activations(n_vec, cols, seed=6)
        x[n_vec - 1, :64] = 0.0       # an all-zero block
        xd = dev(x)
        xq = torch.empty(n_vec * qmv.qmv_row_bytes(at, cols), dtype=torch.uint8, device="cuda")
        qmv.qmv_quantize_act(at, xd, xq, n_vec * cols)
        y1 = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
        y2 = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
        qmv.qmv_matvec(qmv.FMT(t, at), W, rows, cols, xq, y1, n_vec)
        qmv.qmv_matvec(qmv.FMT(t, at) | qmv.FLAG_QUANTIZE_X, W, rows, cols, xd, y2, n_vec)
        assert np.array_equal(host(y1).view(np.uint32), host(y2).view(np.uint32)), (t, rows, cols)


def test_pdl_flag_same_results(qmv, orc):
    """Programmatic dependent launch changes scheduling only: a chain of
    dependent quantise + matvec launches gives the same bits with and without
    it, including when each matvec reads the previous one's output."""
    t, at, n = 2, 3, 896
    Ws = [dev(synth.weights(t, n, n, seed=10 + i)) for i in range(6)]
    x0 = dev(synth.activations(1, n, seed=10))

    def chain(flags):
        x = x0.clone()
        for W in Ws:
            y = torch.empty((1, n), dtype=torch.float32, device="cuda")
            xq = torch.empty(qmv.qmv_row_bytes(at, n), dtype=torch.uint8, device="cuda")
            qmv.qmv_quantize_act(at | flags, x, xq, n)
            qmv.qmv_matvec(qmv.FMT(t, at) | flags, W, n, n, xq, y, 1)
            x = y * 0.05
        return host(x)

    a = chain(0)
    b = chain(qmv.FLAG_PDL)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    qmv.qmv_get_status()


# ---- degenerate blocks, many vectors, the longest rows ------------------------------

@pytest.mark.parametrize("t", [1, 2, 3, 4, 5, 6])
def test_matvec_degenerate_blocks(qmv, orc, t):
    """Rows whose blocks all have a zero scale (Q4_K: zero d and dmin; MXFP4:
    zero codes) give exactly zero, with 8-bit and fp32 activations; the other
    rows are unaffected."""
    rows, cols = 12, 512
    blocks = synth.weights(t, rows, cols, seed=60 + t).view(synth.block_dtype(t)).reshape(rows, -1)
    zero_rows = [0, 5, 11]
    for r in zero_rows:
        if t == 6:
            blocks[r]["qs"] = 0
        else:
            blocks[r]["d"] = 0
            if t == 4:
                blocks[r]["dmin"] = 0
    W = blocks.view(np.uint8).reshape(-1)
    at8 = 7 if t in (4, 5) else 3
    x = synth.activations(3, cols, seed=61)
    for at in (at8, 8):
        xin = orc.quantize_act(at, x) if at != 8 else x
        yref, yabs = orc.matvec(orc_t(t), at, W, rows, cols, xin, 3)
        y = torch.full((3, rows), float("nan"), dtype=torch.float32, device="cuda")
        qmv.qmv_matvec(qmv.FMT(t, at) | (qmv.FLAG_QUANTIZE_X if at != 8 else 0), dev(W), rows, cols, dev(x), y, 3)
        yh = host(y)
        assert (yh[:, zero_rows] == 0).all() and (yref[:, zero_rows] == 0).all()
        assert_close(yh, yref, yabs, what=f"t={t} at={at}")


def test_matvec_mxfp4_nan_exponent(qmv, orc):
    """An E8M0 exponent of 255 is NaN (OCP): the row holding that block is NaN
    on both sides, the other rows are finite and match."""
    rows, cols = 6, 256
    blocks = synth.weights(6, rows, cols, seed=70).view(synth.block_dtype(6)).reshape(rows, -1)
    blocks[2, 3]["e"] = 255
    W = blocks.view(np.uint8).reshape(-1)
    x = synth.activations(2, cols, seed=71)
    for at in (3, 8):
        xin = orc.quantize_act(at, x) if at != 8 else x
        yref, yabs = orc.matvec(6, at, W, rows, cols, xin, 2)
        y = torch.empty((2, rows), dtype=torch.float32, device="cuda")
        qmv.qmv_matvec(qmv.FMT(6, at) | (qmv.FLAG_QUANTIZE_X if at != 8 else 0), dev(W), rows, cols, dev(x), y, 2)
        yh = host(y)
        assert np.isnan(yref[:, 2]).all() and np.isnan(yh[:, 2]).all()
        keep = [r for r in range(rows) if r != 2]
        assert_close(yh[:, keep], yref[:, keep], yabs[:, keep], what=f"at={at}")


@pytest.mark.parametrize("t,at", [(2, 3), (4, 7), (6, 8)])
def test_matvec_many_vectors(qmv, orc, t, at):
    """37 vectors: several launches of up to 16 vectors each, a ragged last group."""
    rows, cols, n_vec = 70, 512, 37
    W = synth.weights(t, rows, cols, seed=80 + t)
    x = synth.activations(n_vec, cols, seed=81)
    xin = orc.quantize_act(at, x) if at != 8 else x
    yref, yabs = orc.matvec(orc_t(t), at, W, rows, cols, xin, n_vec)
    y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, at) | (qmv.FLAG_QUANTIZE_X if at != 8 else 0), dev(W), rows, cols, dev(x), y, n_vec)
    assert_close(host(y), yref, yabs, what=f"t={t} at={at}")


def test_matvec_longest_rows(qmv, orc):
    """A row of 65536 elements stages its 8-bit activations in one SM's shared
    memory and is computed; rows whose staged activations cannot fit are
    refused with QMV_ERR_SHAPE before anything is launched."""
    rows, cols = 3, 65536
    W = synth.weights(1, rows, cols, seed=90)
    x = synth.activations(1, cols, seed=91)
    yref, yabs = orc.matvec(1, 3, W, rows, cols, orc.quantize_act(3, x), 1)
    y = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(1, 3) | qmv.FLAG_QUANTIZE_X, dev(W), rows, cols, dev(x), y, 1)
    assert_close(host(y), yref, yabs, what="65536 cols")
    big = torch.zeros(rows * qmv.qmv_row_bytes(1, 1 << 17), dtype=torch.uint8, device="cuda")
    xb = torch.zeros((1, 1 << 17), dtype=torch.float32, device="cuda")
    yb = torch.zeros((1, rows), dtype=torch.float32, device="cuda")
    for fmt, c in ((qmv.FMT(1, 3) | qmv.FLAG_QUANTIZE_X, 1 << 17), (qmv.FMT(1, 8), 1 << 16)):
        with pytest.raises(qmv.QmvError) as e:
            qmv.qmv_matvec(fmt, big, rows, c, xb, yb, 1)
        assert e.value.code == qmv.ERR_SHAPE and "shared memory" in str(e.value)
    qmv.qmv_get_status()


# ---- plain F32 / F16 / BF16 weights (fp32 activations) -------------------------------

@pytest.mark.parametrize("t", PLAIN)
def test_plain_weights(qmv, orc, t):
    """Plain weights: dequantisation is the exact conversion; the matvec
    matches the oracle within the bar on ragged tiles, several K-chunks and
    16 vectors; decode is batch-invariant bit for bit; 8-bit activations and
    rows that are not multiples of 8 are refused."""
    for rows, cols in [(1, 8), (37, 96), (300, 896), (45, 8288)]:
        W = synth.weights(t, rows, cols, seed=21, tensor_id=rows)
        out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
        qmv.qmv_dequantize(t, dev(W), rows, cols, out)
        assert np.array_equal(host(out).view(np.uint32), orc.dequant(orc_t(t), W, rows, cols).view(np.uint32))
        for n_vec in (1, 3, 16):
            x = synth.activations(n_vec, cols, seed=22, tensor_id=cols)
            yref, yabs = orc.matvec(orc_t(t), 8, W, rows, cols, x, n_vec)
            y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_matvec(qmv.FMT(t, 8), dev(W), rows, cols, dev(x), y, n_vec)
            assert_close(host(y), yref, yabs, what=f"t={t} {rows}x{cols} n_vec={n_vec}")
            if n_vec == 16:
                y1 = torch.empty((1, rows), dtype=torch.float32, device="cuda")
                qmv.qmv_matvec(qmv.FMT(t, 8), dev(W), rows, cols, dev(x[7:8]), y1, 1)
                assert np.array_equal(host(y1)[0].view(np.uint32), host(y)[7].view(np.uint32))
    Wd = dev(synth.weights(t, 4, 64, seed=1))
    y = torch.empty((1, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matvec(qmv.FMT(t, 3), Wd, 4, 64, Wd, y, 1)
    assert e.value.code == qmv.ERR_UNSUPPORTED
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_matvec(qmv.FMT(t, 8), Wd, 4, 60, Wd, y, 1)
    assert e.value.code == qmv.ERR_SHAPE
    qmv.qmv_get_status()


@pytest.mark.parametrize("t", [11, 12, 13, 14, 15, 16, 17])
def test_new_formats_in_the_expert_matvec(qmv, orc, t):
    """The mixture-of-experts matvec over stacked experts of the later formats,
    up and down forms, against the oracle."""
    E, rows, k, n_tok = 5, 40, 2, 7
    cols = 64 if t in (11, 12, 13, 17) else 512
    W3 = synth.weights(t, E * rows, cols, seed=33, tensor_id=t)
    ids, gates = synth.router(n_tok, E, k, seed=34)
    b = synth.bias(E, rows, seed=35)
    at = 8 if t == 17 else act_for(t)
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    qmv.qmv_set_workspace(buf, buf.numel())
    try:
        for down in (False, True):
            x = synth.activations(n_tok * k if down else n_tok, cols, seed=36)
            if down:
                x = x.reshape(n_tok, k, cols)
            fl = qmv.FLAG_QUANTIZE_X if at != 8 else 0
            shape = (n_tok, rows) if down else (n_tok, k, rows)
            y = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_moe_matvec(qmv.FMT(t, at) | fl, dev(W3), E, rows, cols, dev(ids), dev(gates) if down else None,
                               k, dev(x), y, n_tok, dev(b))
            x_o = orc.quantize_act(at, x) if at != 8 else x
            yref, yabs = orc.moe(orc_t(t), at, W3, E, rows, cols, ids, gates if down else None, k, x_o, n_tok, bias=b)
            assert_close(host(y), yref, yabs, what=f"t={t} down={down}")
        qmv.qmv_get_status()
    finally:
        qmv.qmv_set_workspace(None, 0)
