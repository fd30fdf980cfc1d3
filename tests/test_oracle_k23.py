"""Pins of the oracle's Q2_K and Q3_K decoding and products, no GPU.

Both are K-quants the "Models and formats" page lists ("Q2_K through Q8_K").
The byte layouts are the GGUF ones (2-bit codes in 128-element halves; Q2_K
with 4-bit sub-block scales and mins, Q3_K with a high-bit mask and sixteen
6-bit scales centred on 32).  Pinned by literal blocks, closed forms on
independently packed blocks, the position bijection, brute-force integer dots
against Q8_K activations and dense fp64 products."""
import numpy as np
import pytest

import packers as P

Q2_K, Q3_K, Q8_K, F32 = 13, 14, 7, 8
# code byte 0xE4 holds 0, 1, 2, 3 in its bit pairs: element 128n+32j+l gets code j
PATTERN = np.tile(np.repeat(np.arange(4), 32), 2).astype(np.float32)


def test_literal_q2_k(orc):
    # every scale byte 0x01 (scale 1, min 0), d = 1, dmin = 0
    blob = bytes.fromhex("01" * 16 + "e4" * 64 + "003c" + "0000")
    w = orc.dequant(Q2_K, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
    assert np.array_equal(w, PATTERN)
    # scale 1, min 1, dmin = 0.5: every weight lowered by 0.5
    blob = bytes.fromhex("11" * 16 + "e4" * 64 + "003c" + "0038")
    w = orc.dequant(Q2_K, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
    assert np.array_equal(w, PATTERN - 0.5)


def test_literal_q3_k(orc):
    # every 6-bit scale 33 (factor 1): low nibbles 1 (bytes 0x11), high bits 2 (bytes 0xaa); d = 1
    scales = "11" * 8 + "aa" * 4
    blob = bytes.fromhex("ff" * 32 + "e4" * 64 + scales + "003c")      # mask set: code = low bits
    w = orc.dequant(Q3_K, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
    assert np.array_equal(w, PATTERN)
    blob = bytes.fromhex("00" * 32 + "e4" * 64 + scales + "003c")      # mask clear: code = low bits - 4
    w = orc.dequant(Q3_K, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
    assert np.array_equal(w, PATTERN - 4)


def _random(t, g):
    d = float(np.float16(abs(g.normal()) * 0.02))
    if t == Q2_K:
        dmin = float(np.float16(abs(g.normal()) * 0.02))
        sc, m, q = g.integers(0, 16, 16), g.integers(0, 16, 16), g.integers(0, 4, 256)
        return P.pack_q2_k(d, dmin, sc, m, q), P.closed_q2_k(d, dmin, sc, m, q), ("q2", sc, m, q)
    s6, code = g.integers(0, 64, 16), g.integers(-4, 4, 256)
    return P.pack_q3_k(d, s6, code), P.closed_q3_k(d, s6, code), ("q3", s6, code)


@pytest.mark.parametrize("t", [Q2_K, Q3_K])
def test_closed_form_random_blocks(orc, t):
    g = np.random.default_rng(700 + t)
    for _ in range(200):
        blob, ref, _ = _random(t, g)
        w = orc.dequant(t, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
        assert np.array_equal(w, np.array(ref, dtype=np.float64).astype(np.float32)), t


@pytest.mark.parametrize("t", [Q2_K, Q3_K])
def test_each_position_moves_one_element(orc, t):
    for pos in range(256):
        if t == Q2_K:
            sc, m = [i % 15 + 1 for i in range(16)], [0] * 16   # 4-bit scales, none zero
            base = np.full(256, 1)
            alt = base.copy()
            alt[pos] = 3
            a, b = P.pack_q2_k(1.0, 0.0, sc, m, base), P.pack_q2_k(1.0, 0.0, sc, m, alt)
        else:
            s6 = list(range(33, 49))
            base = np.full(256, 1)
            alt = base.copy()
            alt[pos] = -3                    # changes both the low bits and the mask bit
            a, b = P.pack_q3_k(1.0, s6, base), P.pack_q3_k(1.0, s6, alt)
        wa = orc.dequant(t, np.frombuffer(a, dtype=np.uint8), 1, 256)[0]
        wb = orc.dequant(t, np.frombuffer(b, dtype=np.uint8), 1, 256)[0]
        assert list(np.nonzero(wa != wb)[0]) == [pos], (t, pos)


def _matrix(t, rows, cols, seed):
    g = np.random.default_rng(seed)
    blobs, ws, fields = [], [], []
    for _ in range(rows * cols // 256):
        b, w, f = _random(t, g)
        blobs.append(b)
        ws.append(w)
        fields.append(f)
    return np.frombuffer(b"".join(blobs), dtype=np.uint8).copy(), np.array(ws, dtype=np.float64).reshape(rows, cols), fields


def _xq_codes(xq, n_vec, nb):
    blocks = np.frombuffer(xq.tobytes(), dtype=np.uint8).reshape(n_vec, nb, 292)
    d = blocks[:, :, :4].copy().view(np.float32)[:, :, 0].astype(np.float64)
    return d, blocks[:, :, 4:260].view(np.int8).astype(np.int64)


@pytest.mark.parametrize("t", [Q2_K, Q3_K])
def test_block_dots_brute_force(orc, t):
    rows, cols, n_vec = 3, 512, 2
    W, _, fields = _matrix(t, rows, cols, 11)
    x = np.random.default_rng(12).standard_normal((n_vec, cols)).astype(np.float32)
    xq = orc.quantize_act(Q8_K, x)
    out = orc.block_dots(t, W, rows, cols, xq, n_vec)
    _, xc = _xq_codes(xq, n_vec, cols // 256)
    sub = [P._k23_pos(e)[2] for e in range(256)]
    for v in range(n_vec):
        for r in range(rows):
            for b in range(cols // 256):
                f = fields[r * (cols // 256) + b]
                if f[0] == "q2":
                    _, sc, m, q = f
                    S = sum(int(sc[sub[e]]) * int(q[e]) * int(xc[v, b, e]) for e in range(256))
                    Mn = sum(int(m[sub[e]]) * int(xc[v, b, e]) for e in range(256))
                else:
                    _, s6, code = f
                    S = sum((int(s6[sub[e]]) - 32) * int(code[e]) * int(xc[v, b, e]) for e in range(256))
                    Mn = 0
                assert tuple(out[v, r, b]) == (S, Mn)


@pytest.mark.parametrize("t", [Q2_K, Q3_K])
def test_matvec_dense_brute_force(orc, t):
    rows, cols, n_vec = 5, 512, 3
    W, Wd, _ = _matrix(t, rows, cols, 13)
    x = np.random.default_rng(14).standard_normal((n_vec, cols)).astype(np.float32)
    y, _ = orc.matvec(t, F32, W, rows, cols, x, n_vec)
    assert np.allclose(y, x.astype(np.float64) @ Wd.T, rtol=0, atol=1e-9)
    xq = orc.quantize_act(Q8_K, x)
    d, xc = _xq_codes(xq, n_vec, cols // 256)
    y8, _ = orc.matvec(t, Q8_K, W, rows, cols, xq, n_vec)
    assert np.allclose(y8, (d[:, :, None] * xc).reshape(n_vec, cols) @ Wd.T, rtol=0, atol=1e-9)
