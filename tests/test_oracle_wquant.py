"""Pins of the oracle's weight quantisers (fp32 -> Q4_0 / Q5_0 / Q8_0), no GPU.

Each test fixes the oracle against something other than its own formula:
hand-built blocks whose codes are known exactly, the zero block, the sign and
tie rule of the block extreme, a brute-force nearest-grid-point check, the
round-trip error bound, and the decoders of blocks.c (pinned elsewhere)."""
import numpy as np
import pytest

from oracle import oracle as O


def _scale(blk: bytes) -> float:
    return float(np.frombuffer(blk[:2], dtype=np.float16)[0])


def test_known_q4_0_block():
    # -4, -3.5, ..., 3.5 twice: m = -4 (first of two), d = 0.5, codes 0..15
    x = (np.arange(32) % 16 * 0.5 - 4).astype(np.float32)
    assert O.quantize_weights(O.Q4_0, x).tobytes().hex() == "0038" + "00112233445566778899aabbccddeeff"


def test_known_q5_0_block():
    # (i - 16) / 4: m = -4, d = 0.25, codes 0..31: fifth bits set for i >= 16
    x = ((np.arange(32) - 16) * 0.25).astype(np.float32)
    assert O.quantize_weights(O.Q5_0, x).tobytes().hex() == \
        "0034" + "0000ffff" + "00112233445566778899aabbccddeeff"


def test_zero_block():
    z = np.zeros(32, dtype=np.float32)
    # m = 0 and d = 0 / -8 is -0 in IEEE arithmetic: fp16 0x8000; every code is the zero point
    assert O.quantize_weights(O.Q4_0, z).tobytes().hex() == "0080" + "88" * 16      # code 8 = 0
    assert O.quantize_weights(O.Q5_0, z).tobytes().hex() == "0080" + "ffffffff" + "00" * 16   # code 16 = 0


def test_extreme_sign_and_ties():
    x = np.full(32, 0.01, dtype=np.float32)
    x[0] = 2.0                       # positive extreme: d = 2 / -8 = -0.25
    b = O.quantize_weights(O.Q4_0, x).tobytes()
    assert b[:2].hex() == "00b4" and (b[2] & 15) == 0
    y = np.full(32, 0.01, dtype=np.float32)
    y[3], y[7] = -3.0, 3.0           # equal magnitudes: the first one decides, d = -3 / -8 = 0.375
    assert O.quantize_weights(O.Q4_0, y).tobytes()[:2].hex() == "0036"
    y[3], y[7] = 3.0, -3.0
    assert O.quantize_weights(O.Q4_0, y).tobytes()[:2].hex() == "00b6"


@pytest.mark.parametrize("t,half", [(O.Q4_0, 8), (O.Q5_0, 16)])
def test_scale_below_2_pow_minus_128(t, half):
    """A block extreme so small that 1/d overflows: zero weights still land on
    the zero point (code 8 / 16), the extreme on code 0, and every code is a
    nearest grid point of the exact quotient x/d."""
    g = np.random.default_rng(23)
    m = np.float32(-2e-38)
    x = (g.uniform(-1, 1, 32) * np.float32(1.9e-38)).astype(np.float32)
    x[5] = m
    x[0] = 0.0
    x[9] = -0.0
    d = m / np.float32(-half)
    assert float(abs(d)) < 2.0 ** -128 and np.isinf(np.float32(1) / d)
    b = O.quantize_weights(t, x).tobytes()
    nib = np.frombuffer(b[2 if t == O.Q4_0 else 6:], dtype=np.uint8)
    q = np.concatenate([nib & 15, nib >> 4]).astype(int)
    if t == O.Q5_0:
        qh = int.from_bytes(b[2:6], "little")
        q += np.array([(qh >> i) & 1 for i in range(32)]) * 16
    assert q[0] == half and q[9] == half and q[5] == 0
    exact = x.astype(np.float64) / float(d) + half
    top = 2 * half - 1
    assert (np.abs(np.clip(exact, 0, top) - q) <= 0.5 + 1e-5).all()


def _blocks(seed, n):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, 32)).astype(np.float32)
    x *= np.exp2(g.integers(-12, 8, (n, 1))).astype(np.float32)
    x[::7] = g.uniform(-1, 1, (len(x[::7]), 32)).astype(np.float32)
    x[::11, 5] = -x[::11, 9]         # magnitude ties
    return x


@pytest.mark.parametrize("t,half,top", [(O.Q4_0, 8, 15), (O.Q5_0, 16, 31)])
def test_codes_are_nearest_grid_points(t, half, top):
    """Every code is a nearest point of the block's grid d*(q - half), q in
    0..top (the fp32 d), except past the grid's top end, where it clamps."""
    x = _blocks(1, 2000)
    out = O.quantize_weights(t, x).reshape(len(x), -1)
    W = O.dequant(t, out.reshape(-1), len(x), 32).astype(np.float64)
    for i in range(len(x)):
        xi = x[i].astype(np.float64)
        m = xi[np.argmax(np.abs(xi))]            # numpy's argmax takes the first of equal values
        d = np.float64(np.float32(np.float32(m) / np.float32(-half)))
        if d == 0:
            assert np.all(W[i] == 0)
            continue
        grid = d * (np.arange(top + 1) - half)
        err = np.abs(xi[:, None] - grid[None, :])
        q = np.rint(W[i] / np.float64(_scale(out[i].tobytes())) + half).astype(int)
        got = err[np.arange(32), q]
        best = err.min(axis=1)
        clamped = xi / d > top - half + 0.5 - 1e-6
        ok = (got <= best + 1e-5 * abs(d)) | (clamped & (q == top))
        assert ok.all(), (i, np.flatnonzero(~ok))


@pytest.mark.parametrize("t,half", [(O.Q4_0, 8), (O.Q5_0, 16)])
def test_extreme_lands_on_code_zero_and_error_bound(t, half):
    x = _blocks(2, 1000)
    out = O.quantize_weights(t, x).reshape(len(x), -1)
    W = O.dequant(t, out.reshape(-1), len(x), 32).astype(np.float64)
    for i in range(len(x)):
        xi = x[i].astype(np.float64)
        k = int(np.argmax(np.abs(xi)))
        d16 = _scale(out[i].tobytes())
        d32 = float(np.float32(np.float32(xi[k]) / np.float32(-half)))
        # the extreme decodes to -half * d16, i.e. to m up to the fp16 rounding of d
        assert W[i, k] == -half * d16
        assert abs(W[i, k] - xi[k]) <= half * abs(d16 - d32) + 1e-6 * abs(xi[k])
        # every element within one grid step (half a step except at the clamped end)
        assert np.all(np.abs(W[i] - xi) <= abs(d32) + half * abs(d16 - d32) + 1e-5 * abs(d32))


def test_q8_0_weights_are_the_symmetric_8bit_form():
    x = _blocks(3, 300)
    assert np.array_equal(O.quantize_weights(O.Q8_0, x), O.quantize_act(O.Q8_0, x).reshape(-1))


def test_refusals():
    with pytest.raises(O.OracleError):
        O.quantize_weights(O.Q6_K, np.zeros(200, dtype=np.float32))   # not a whole super-block
    with pytest.raises(O.OracleError):
        O.quantize_weights(O.Q8_K, np.zeros(256, dtype=np.float32))   # an activation-only type
    with pytest.raises(O.OracleError):
        O.lib()   # loads
        O._check(O.lib().orc_quantize_weights(O.Q4_0, O._ptr(np.zeros(48, dtype=np.float32)), 48,
                                              O._ptr(np.zeros(64, dtype=np.uint8))), "quantize_weights")
