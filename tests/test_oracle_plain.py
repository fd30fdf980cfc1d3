"""Pins of the oracle's Q8_1 blocks and its plain F32 / F16 / BF16 weights, no GPU.

"Models and formats" page, "Tensor formats": Q8_1 is among the formats read;
F32, F16 and BF16 are read and accelerated on every backend.  Q8_1 is the GGUF
block fp16 d | fp16 s | int8[32] with w = d*q (s, the block's code sum times
d, belongs to activation blocks and a weight ignores it); the plain types are
one little-endian value per element.  Pinned by hand-built blocks, numpy's
and torch's own conversions, the position bijection, brute-force integer dots
and dense fp64 products computed here from independently decoded weights."""
import numpy as np
import pytest
import torch

Q8_0, F32, BF16, Q8_1, F16 = 3, 8, 9, 15, 16


def pack_q8_1(d, s, q):
    return np.float16(d).tobytes() + np.float16(s).tobytes() + np.asarray(q, dtype=np.int8).tobytes()


def test_handbuilt_q8_1(orc):
    # d = 0.5, s = +inf (must not matter), codes -16..15: w = q / 2
    q = np.arange(-16, 16)
    blob = bytes.fromhex("0038" + "007c") + q.astype(np.int8).tobytes()
    w = orc.dequant(Q8_1, np.frombuffer(blob, dtype=np.uint8), 1, 32)[0]
    assert np.array_equal(w, (q * 0.5).astype(np.float32))


def test_q8_1_closed_form_and_positions(orc):
    g = np.random.default_rng(41)
    for _ in range(200):
        d, s = np.float16(g.normal() * 0.05), np.float16(g.normal() * 9)
        q = g.integers(-128, 128, 32)
        w = orc.dequant(Q8_1, np.frombuffer(pack_q8_1(d, s, q), dtype=np.uint8), 1, 32)[0]
        assert np.array_equal(w, (float(d) * q.astype(np.float64)).astype(np.float32))
    for pos in range(32):
        base = np.full(32, 3)
        alt = base.copy()
        alt[pos] = -77
        wa = orc.dequant(Q8_1, np.frombuffer(pack_q8_1(1.0, 0.0, base), dtype=np.uint8), 1, 32)[0]
        wb = orc.dequant(Q8_1, np.frombuffer(pack_q8_1(1.0, 0.0, alt), dtype=np.uint8), 1, 32)[0]
        assert list(np.nonzero(wa != wb)[0]) == [pos]


def _q8_1_matrix(rows, cols, seed):
    g = np.random.default_rng(seed)
    blobs, ws = [], []
    for _ in range(rows * cols // 32):
        d, s, q = np.float16(abs(g.normal()) * 0.02), np.float16(g.normal()), g.integers(-127, 128, 32)
        blobs.append(pack_q8_1(d, s, q))
        ws.append(float(d) * q.astype(np.float64))
    return np.frombuffer(b"".join(blobs), dtype=np.uint8).copy(), np.array(ws).reshape(rows, cols)


def test_q8_1_dots_and_products(orc):
    rows, cols = 6, 128
    W, Wd = _q8_1_matrix(rows, cols, 42)
    x = np.random.default_rng(43).standard_normal((2, cols)).astype(np.float32)
    xq = orc.quantize_act(Q8_0, x)
    out = orc.block_dots(Q8_1, W, rows, cols, xq, 2)
    xc = np.frombuffer(xq.tobytes(), dtype=np.uint8).reshape(2, cols // 32, 34)[:, :, 2:].view(np.int8).astype(np.int64)
    codes = W.reshape(rows, cols // 32, 36)[:, :, 4:].view(np.int8).astype(np.int64)
    for v in range(2):
        for r in range(rows):
            for b in range(cols // 32):
                assert tuple(out[v, r, b]) == (int(codes[r, b] @ xc[v, b]), 0)
    y, _ = orc.matvec(Q8_1, F32, W, rows, cols, x, 2)
    assert np.allclose(y, x.astype(np.float64) @ Wd.T, rtol=0, atol=1e-10)


@pytest.mark.parametrize("t", [F32, F16, BF16])
def test_plain_weights_decode(orc, t):
    g = np.random.default_rng(50 + t)
    rows, cols = 5, 48
    if t == F32:
        w = g.standard_normal((rows, cols)).astype(np.float32)
        raw, ref = w.view(np.uint8).reshape(-1), w
    else:
        bits = g.integers(0, 1 << 16, (rows, cols), dtype=np.uint16)
        bits[(bits & 0x7c00) == 0x7c00] &= 0x3fff if t == F16 else 0xffff   # finite fp16 only
        if t == BF16:
            bits[(bits & 0x7f80) == 0x7f80] &= 0x3fff                          # finite bf16 only
        raw = bits.view(np.uint8).reshape(-1)
        ref = bits.view(np.float16).astype(np.float32) if t == F16 else \
            torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    out = orc.dequant(t, raw, rows, cols)
    assert np.array_equal(out.view(np.uint32), ref.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("t", [F32, F16, BF16])
def test_plain_weights_matvec_dense(orc, t):
    g = np.random.default_rng(60 + t)
    rows, cols, n = 9, 96, 3
    w32 = g.standard_normal((rows, cols)).astype(np.float32)
    if t == F32:
        raw, wd = w32.view(np.uint8).reshape(-1), w32.astype(np.float64)
    elif t == F16:
        w16 = w32.astype(np.float16)
        raw, wd = w16.view(np.uint8).reshape(-1), w16.astype(np.float64)
    else:
        wb = torch.from_numpy(w32).to(torch.bfloat16)
        raw, wd = wb.view(torch.int16).numpy().view(np.uint8).reshape(-1), wb.double().numpy()
    x = g.standard_normal((n, cols)).astype(np.float32)
    y, yabs = orc.matvec(t, F32, raw, rows, cols, x, n)
    assert np.allclose(y, x.astype(np.float64) @ wd.T, rtol=0, atol=1e-11)
    assert np.allclose(yabs, np.abs(x.astype(np.float64)) @ np.abs(wd).T, rtol=1e-12, atol=0)
    with pytest.raises(Exception):
        orc.matvec(t, Q8_0, raw, rows, cols, orc.quantize_act(Q8_0, x), n)   # plain weights pair with F32 only


@pytest.mark.parametrize("t", [F32, F16, BF16])
def test_plain_weights_bf16_activations(orc, t):
    """Plain rows against bf16 activations (the prefill product): each weight is
    rounded to bf16 from its fp32 value, nearest-even (torch's conversion), and
    the products are summed in fp64.  F32 rows include exact halfway cases
    (1 + 2^-8 rounds down to 1, 1 + 3*2^-8 up to 1 + 2^-6) so a truncating or
    ties-away rounding fails."""
    g = np.random.default_rng(70 + t)
    rows, cols, n = 7, 64, 3
    w32 = g.standard_normal((rows, cols)).astype(np.float32)
    w32[0, :4] = [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.0 * (1 + 2.0 ** -8)]
    if t == F32:
        raw, wf = w32.view(np.uint8).reshape(-1), w32
    elif t == F16:
        w16 = w32.astype(np.float16)
        raw, wf = w16.view(np.uint8).reshape(-1), w16.astype(np.float32)
    else:
        wb = torch.from_numpy(w32).to(torch.bfloat16)
        raw, wf = wb.view(torch.int16).numpy().view(np.uint8).reshape(-1), wb.float().numpy()
    wd = torch.from_numpy(wf).to(torch.bfloat16).double().numpy()
    if t == F32:
        assert wd[0, 0] == 1.0 and wd[0, 1] == 1 + 2.0 ** -6 and wd[0, 2] == -1.0
    xb = torch.from_numpy(g.standard_normal((n, cols)).astype(np.float32)).to(torch.bfloat16)
    y, yabs = orc.matvec(t, BF16, raw, rows, cols, xb.view(torch.int16).numpy(), n)
    xd = xb.double().numpy()
    assert np.allclose(y, xd @ wd.T, rtol=0, atol=1e-12)
    assert np.allclose(yabs, np.abs(xd) @ np.abs(wd).T, rtol=1e-12, atol=0)
