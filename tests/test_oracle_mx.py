"""Pins of the oracle's MXFP8 activations (OCP Microscaling v1.0: E4M3 codes with
one E8M0 scale per 32), no GPU.

The pages name MXFP4 weights but print no activation format for a
block-scaled tensor-core product; the reading is the OCP specification's
MXFP8 and its conversion (scale 2^(floor(log2 amax) - 8), elements rounded to
nearest even E4M3 and clamped to 448).  Pinned by torch's own float8_e4m3fn
conversions (every code decoded, values encoded), hand-worked blocks
(clamping, the scale's lower limit, zero blocks), scale and sign invariance,
the half-unit error bound, and dense fp64 products of independently decoded
operands."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth

MXFP4_LIB, MXFP4, MXFP8, F32 = 6, 6, 17, 8


def test_e4m3_decode_every_code(orc):
    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_to_f64(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_below_the_clamp(orc):
    g = np.random.default_rng(7)
    v = np.concatenate([
        np.exp2(g.uniform(-12, np.log2(447.9), 4000)) * g.choice([-1, 1], 4000),
        # every midpoint between neighbouring codes (ties) and points just beside them
    ]).astype(np.float32)
    vals = np.array([orc.e4m3_to_f64(b) for b in range(0x7f)])       # 0 .. 448, increasing
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    v = v[np.abs(v) < 448]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.f64_to_e4m3(float(t)) for t in v], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_clamps_to_448(orc):
    for t in (448.0, 463.9, 464.0, 480.0, 511.0, 1e6):
        assert orc.f64_to_e4m3(t) == 0x7e and orc.f64_to_e4m3(-t) == 0xfe


def block_of(x):
    return np.asarray(x, dtype=np.float32).reshape(1, 32)


def test_hand_worked_blocks(orc):
    x = np.zeros(32, np.float32)
    x[0] = 1.0                                   # amax 1: E = -8, 1 * 2^8 = 256 -> 0x78
    b = orc.quantize_act(MXFP8, block_of(x))[0]
    assert b[0] == 119 and b[1] == 0x78 and not b[2:].any()
    x[5] = -1.96                                 # amax 1.96: E = -8, 501.8 clamps to 448
    b = orc.quantize_act(MXFP8, block_of(x))[0]
    assert b[0] == 119 and b[6] == 0xfe and b[1] == 0x78
    z = orc.quantize_act(MXFP8, block_of(np.zeros(32)))[0]   # zeros: the lowest scale, codes 0
    assert z[0] == 0 and not z[1:].any()
    t = np.full(32, 2.0 ** -130, np.float32)     # E would be -138: held at -127
    b = orc.quantize_act(MXFP8, block_of(t))[0]
    assert b[0] == 0 and all(c == 0x20 for c in b[1:])   # 2^-130 * 2^127 = 2^-3
    big = np.full(32, 3.0e38, np.float32)        # E = 127 - 8 = 119: byte 246
    b = orc.quantize_act(MXFP8, block_of(big))[0]
    assert b[0] == 246


def test_scale_and_sign_invariance(orc):
    g = np.random.default_rng(8)
    x = g.standard_normal((16, 32)).astype(np.float32)
    base = orc.quantize_act(MXFP8, x)
    for k in (-20, -3, 5, 40):
        s = orc.quantize_act(MXFP8, (x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(s[:, 1:], base[:, 1:])
        assert np.array_equal(s[:, 0].astype(int), base[:, 0].astype(int) + k)
    neg = orc.quantize_act(MXFP8, -x)
    assert np.array_equal(neg[:, 0], base[:, 0])
    assert np.array_equal(orc.mxfp8_values(neg), -orc.mxfp8_values(base))


def test_error_bound_and_positions(orc):
    g = np.random.default_rng(9)
    x = (g.standard_normal((64, 256)) * np.exp2(g.uniform(-30, 30, (64, 1)))).astype(np.float32)
    q = orc.quantize_act(MXFP8, x)
    v = orc.mxfp8_values(q)
    E = (q.reshape(64, 8, 33)[:, :, 0].astype(np.int64) - 127)
    E = np.repeat(E, 32, axis=1)
    scaled = np.abs(x.astype(np.float64)) * np.exp2(-E)
    clipped = scaled >= 448
    # unclipped: half a unit of E4M3 (2^-4 relative, or 2^-10 absolute below 2^-6)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.exp2(E - 10))
    assert np.all(np.abs(v - x)[~clipped] <= bound[~clipped])
    assert np.all(np.abs(v[clipped]) == 448 * np.exp2(E[clipped]))
    assert clipped.any()
    # one element changed (not the block's largest) changes one code
    y = x.copy()
    y[3, 37] *= 0.5
    q2 = orc.quantize_act(MXFP8, y)
    diff = np.nonzero(q2[3] != q[3])[0]
    assert list(diff) == [33 + 1 + 5]


def test_products_against_dense_fp64(orc):
    rows, cols, n = 24, 256, 3
    W = synth.weights(MXFP4_LIB, rows, cols, seed=12)
    x = (synth.activations(n, cols, seed=13) * 3).astype(np.float32)
    xq = orc.quantize_act(MXFP8, x)
    # x-hat decoded independently with torch's E4M3 and the E8M0 exponent
    codes = torch.from_numpy(xq.reshape(n, cols // 32, 33)[:, :, 1:].copy()).view(torch.float8_e4m3fn)
    sc = np.exp2(xq.reshape(n, cols // 32, 33)[:, :, :1].astype(np.float64) - 127)
    xhat = (codes.to(torch.float64).numpy() * sc).reshape(n, cols)
    Wd = orc.dequant(MXFP4, W, rows, cols).astype(np.float64)
    y, yabs = orc.matvec(MXFP4, MXFP8, W, rows, cols, xq, n)
    want = xhat @ Wd.T
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12 * np.abs(Wd).sum() * np.abs(xhat).max())
    np.testing.assert_allclose(yabs, np.abs(xhat) @ np.abs(Wd).T, rtol=1e-12)
    # the mixture of experts composes the same products per slot
    E, k = 3, 2
    W3 = synth.weights(MXFP4_LIB, E * rows, cols, seed=14)
    ids, gates = synth.router(n, E, k, seed=15)
    ym, _ = orc.moe(MXFP4, MXFP8, W3, E, rows, cols, ids, None, k, xq, n)
    for t in range(n):
        for s in range(k):
            e = ids[t, s]
            We = W3[e * rows * orc.row_bytes(MXFP4, cols):(e + 1) * rows * orc.row_bytes(MXFP4, cols)]
            yv, _ = orc.matvec(MXFP4, MXFP8, We, rows, cols, xq[t:t + 1], 1)
            assert np.array_equal(ym[t, s], yv[0])


def test_refusals(orc):
    with pytest.raises(Exception):
        orc.quantize_act(MXFP8, np.full((1, 32), np.inf, np.float32))
    with pytest.raises(Exception):
        orc.matvec(4, MXFP8, np.zeros(144, np.uint8), 1, 256, np.zeros(8 * 33, np.uint8), 1)   # Q4_K: 256 blocks
