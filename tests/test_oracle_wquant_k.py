"""Pins of the oracle's Q4_1 / Q5_1 and K-quant (Q4_K, Q5_K, Q6_K) weight
writers, no GPU.

"Models and formats" page, "Tensor formats": llamay quantize writes Q4_0/1,
Q5_0/1, Q8_0 and the K-quants; the pages print no procedure.  The reading
(one pass of min/max rules per run, no search) is pinned by:
  * closed forms: weights that lie exactly on a block's grid -- scales that
    are powers of two, sub-block scales and mins whose extremes are 63 (or -128
    for Q6_K), every run holding its lowest and highest code -- are written back
    to exactly the block an independent packer builds (tests/packers.py);
  * every code is a nearest point of its run's decoded grid (or the clamped
    end), on random data across magnitudes;
  * zero blocks decode to zero."""
import numpy as np
import pytest

import packers as P
from oracle import oracle as O


def _q45k_exact(g, bits):
    top = (1 << bits) - 1
    d, dmin = 2.0 ** -6, 2.0 ** -7
    sc = g.integers(1, 64, 8)
    m = g.integers(0, 64, 8)
    sc[g.integers(0, 8)] = 63
    m[g.integers(0, 8)] = 63
    q = g.integers(0, top + 1, 256)
    for j in range(8):                       # each sub-block holds its lowest and highest code
        i0, i1 = g.choice(32, 2, replace=False)
        q[32 * j + i0], q[32 * j + i1] = 0, top
    x = np.array([d * sc[i // 32] * q[i] - dmin * m[i // 32] for i in range(256)], dtype=np.float64)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)   # exact in fp32
    pack = P.pack_q4_k if bits == 4 else P.pack_q5_k
    return x.astype(np.float32), pack(d, dmin, sc, m, q)


@pytest.mark.parametrize("t,bits", [(O.Q4_K, 4), (O.Q5_K, 5)])
def test_q45k_closed_form(t, bits):
    g = np.random.default_rng(300 + bits)
    for _ in range(200):
        x, ref = _q45k_exact(g, bits)
        got = O.quantize_weights(t, x[None, :]).tobytes()
        assert got == ref
        assert np.array_equal(O.dequant(t, np.frombuffer(got, dtype=np.uint8), 1, 256)[0], x)


def test_q6k_closed_form():
    g = np.random.default_rng(306)
    d = 2.0 ** -8
    for _ in range(200):
        sc = g.integers(-127, 128, 16)
        sc[sc == 0] = 5
        sc[g.integers(0, 16)] = -128
        q = g.integers(1, 64, 256)               # |q - 32| <= 31 except the run extreme
        for j in range(16):
            q[16 * j + g.integers(0, 16)] = 0    # the run's extreme, -32 * D_j
        x = np.array([d * sc[i // 16] * (q[i] - 32) for i in range(256)], dtype=np.float64)
        assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
        got = O.quantize_weights(O.Q6_K, x.astype(np.float32)[None, :]).tobytes()
        assert got == P.pack_q6_k(d, sc, q)


@pytest.mark.parametrize("t,bits", [(O.Q4_1, 4), (O.Q5_1, 5)])
def test_q_1_closed_form(t, bits):
    g = np.random.default_rng(310 + bits)
    top = (1 << bits) - 1
    for _ in range(300):
        d = 2.0 ** int(g.integers(-12, 0))
        m = float(np.float16(g.normal() * 0.5))
        q = g.integers(0, top + 1, 32)
        i0, i1 = g.choice(32, 2, replace=False)
        q[i0], q[i1] = 0, top
        x = np.array([d * v + m for v in q], dtype=np.float64)
        if not np.array_equal(x.astype(np.float32).astype(np.float64), x):
            continue
        got = O.quantize_weights(t, x.astype(np.float32)[None, :]).tobytes()
        assert got == (P.pack_q4_1(d, m, q) if bits == 4 else P.pack_q5_1(d, m, q))


def _random_rows(seed, n, bs):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, bs)).astype(np.float32)
    x *= np.exp2(g.integers(-10, 6, (n, 1))).astype(np.float32)
    x[::5] = np.abs(x[::5])                      # all-positive blocks
    x[1::7] = -np.abs(x[1::7])                   # all-negative blocks
    x[2::9, : bs // 2] = 0.0                     # half-zero blocks
    return x


@pytest.mark.parametrize("t", [O.Q4_1, O.Q5_1])
def test_q_1_codes_are_nearest_on_the_fp32_grid(t):
    """Q4_1 / Q5_1 take their codes from the fp32 d = (max - min)/top and
    m = min (then store both in fp16, as Q4_0 does): each code is a nearest
    point of that fp32 grid, computed here from the block's own values."""
    top = 15 if t == O.Q4_1 else 31
    x = _random_rows(330 + t, 600, 32)
    out = O.quantize_weights(t, x)
    for i in range(len(x)):
        xi = x[i]
        m32, d32 = xi.min(), (xi.max() - xi.min()) / np.float32(top)
        blk = O.decode_block(t, out[i * O.BLOCK_BYTES[t]:(i + 1) * O.BLOCK_BYTES[t]].tobytes())
        assert blk["d"] == float(np.float16(d32)) and -blk["dmin"] == float(np.float16(m32))
        q = blk["code"]
        err = np.abs(xi.astype(np.float64) - (float(d32) * q + float(m32)))
        assert (err <= float(d32) * (0.5 + 1e-5) + 1e-30).all(), i


@pytest.mark.parametrize("t", [O.Q4_K, O.Q5_K, O.Q6_K])
def test_codes_are_nearest_grid_points(t):
    """Each element's decoded weight is a nearest point of its run's grid
    (built from the block's own decoded fields), or the grid's clamped end."""
    bs = O.BLOCK_ELEMS[t]
    x = _random_rows(320 + t, 400, bs)
    out = O.quantize_weights(t, x)
    bb = O.BLOCK_BYTES[t]
    run = {O.Q4_K: 32, O.Q5_K: 32, O.Q6_K: 16}[t]
    ncode = {O.Q4_K: 16, O.Q5_K: 32, O.Q6_K: 64}[t]
    for i in range(len(x)):
        blk = O.decode_block(t, out[i * bb:(i + 1) * bb].tobytes())
        for r in range(bs // run):
            sl = slice(run * r, run * (r + 1))
            scale = blk["d"] * blk["sub_scale"][sl][0]
            off = blk["dmin"] * blk["sub_min"][sl][0]
            base = -32 if t == O.Q6_K else 0
            grid = scale * (np.arange(ncode) + base) - off
            w = scale * blk["code"][sl] - off
            xi = x[i, sl].astype(np.float64)
            err = np.abs(xi[:, None] - grid[None, :])
            got = np.abs(xi - w)
            best = err.min(axis=1)
            lo, hi = grid.min(), grid.max()
            tol = 1e-6 * max(abs(scale), 1e-30) + 1e-30
            ok = (got <= best + tol) | (xi >= hi - tol) & (w == hi) | (xi <= lo + tol) & (w == lo)
            assert ok.all(), (t, i, r)


@pytest.mark.parametrize("t", [O.Q4_1, O.Q5_1, O.Q4_K, O.Q5_K, O.Q6_K])
def test_zero_blocks_decode_to_zero(t):
    bs = O.BLOCK_ELEMS[t]
    out = O.quantize_weights(t, np.zeros((3, bs), dtype=np.float32))
    assert not O.dequant(t, out, 3, bs).any()
