"""Pins of the oracle's Q5_K decoding and products, no GPU.

Q5_K is one of the K-quants the "Models and formats" page lists ("Q2_K through
Q8_K"); the byte layout is the GGUF one: Q4_K's fields (fp16 d, fp16 dmin, the
12 bytes of 6-bit sub-block scales and mins, the nibbles) plus 32 bytes of
fifth bits, w = d*sc*q - dmin*m with 5-bit q.  Pinned by a literal block,
closed forms on independently packed blocks, the position bijection,
brute-force integer dots against Q8_K activations and dense fp64 products."""
import numpy as np
import pytest

import packers as P

Q5_K, Q8_K, F32 = 12, 7, 8


def test_literal_block(orc):
    # d = 1, dmin = 0, every sub-block scale 1 and min 0, codes i mod 32: w = i mod 32
    blob = bytes.fromhex("003c" + "0000" + "01010101" + "00000000" + "01010101"
                         + "00" * 16 + "ff" * 16
                         + "00112233445566778899aabbccddeeff" * 8)
    assert len(blob) == 176
    w = orc.dequant(Q5_K, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
    assert np.array_equal(w, (np.arange(256) % 32).astype(np.float32))


def _random(g):
    d = float(np.float16(abs(g.normal()) * 0.02))
    dmin = float(np.float16(abs(g.normal()) * 0.02))
    sc = g.integers(0, 64, 8)
    m = g.integers(0, 64, 8)
    q = g.integers(0, 32, 256)
    closed = [P.f16_val(d) * int(sc[i // 32]) * int(q[i]) - P.f16_val(dmin) * int(m[i // 32]) for i in range(256)]
    return P.pack_q5_k(d, dmin, sc, m, q), closed, (sc, m, q)


def test_closed_form_random_blocks(orc):
    g = np.random.default_rng(512)
    for _ in range(200):
        blob, ref, _ = _random(g)
        w = orc.dequant(Q5_K, np.frombuffer(blob, dtype=np.uint8), 1, 256)[0]
        # one rounding of the exact d*sc*q - dmin*m, as for Q4_K
        assert np.array_equal(w, np.array(ref, dtype=np.float64).astype(np.float32))


def test_each_position_moves_one_element(orc):
    sc, m = list(range(1, 9)), list(range(8))
    for pos in range(256):
        base = np.full(256, 3)
        alt = base.copy()
        alt[pos] = 29                      # changes both the nibble and the fifth bit
        wa = orc.dequant(Q5_K, np.frombuffer(P.pack_q5_k(1.0, 0.5, sc, m, base), dtype=np.uint8), 1, 256)[0]
        wb = orc.dequant(Q5_K, np.frombuffer(P.pack_q5_k(1.0, 0.5, sc, m, alt), dtype=np.uint8), 1, 256)[0]
        assert list(np.nonzero(wa != wb)[0]) == [pos]


def _matrix(rows, cols, seed):
    g = np.random.default_rng(seed)
    blobs, ws, fields = [], [], []
    for _ in range(rows * cols // 256):
        b, w, f = _random(g)
        blobs.append(b)
        ws.append(w)
        fields.append(f)
    W = np.frombuffer(b"".join(blobs), dtype=np.uint8).copy()
    return W, np.array(ws, dtype=np.float64).reshape(rows, cols), fields


def _xq_codes(xq, n_vec, nb):
    blocks = np.frombuffer(xq.tobytes(), dtype=np.uint8).reshape(n_vec, nb, 292)
    d = blocks[:, :, :4].copy().view(np.float32)[:, :, 0].astype(np.float64)
    q = blocks[:, :, 4:260].view(np.int8).astype(np.int64)
    return d, q


def test_block_dots_brute_force(orc):
    rows, cols, n_vec = 3, 512, 2
    W, _, fields = _matrix(rows, cols, 1)
    x = np.random.default_rng(2).standard_normal((n_vec, cols)).astype(np.float32)
    xq = orc.quantize_act(Q8_K, x)
    out = orc.block_dots(Q5_K, W, rows, cols, xq, n_vec)
    _, xc = _xq_codes(xq, n_vec, cols // 256)
    for v in range(n_vec):
        for r in range(rows):
            for b in range(cols // 256):
                sc, m, q = fields[r * (cols // 256) + b]
                S = sum(int(sc[i // 32]) * int(q[i]) * int(xc[v, b, i]) for i in range(256))
                Mn = sum(int(m[i // 32]) * int(xc[v, b, i]) for i in range(256))
                assert tuple(out[v, r, b]) == (S, Mn)


def test_matvec_dense_brute_force(orc):
    rows, cols, n_vec = 5, 512, 3
    W, Wd, _ = _matrix(rows, cols, 3)
    x = np.random.default_rng(4).standard_normal((n_vec, cols)).astype(np.float32)
    y, _ = orc.matvec(Q5_K, F32, W, rows, cols, x, n_vec)
    assert np.allclose(y, x.astype(np.float64) @ Wd.T, rtol=0, atol=1e-9)
    xq = orc.quantize_act(Q8_K, x)
    d, xc = _xq_codes(xq, n_vec, cols // 256)
    xhat = (d[:, :, None] * xc).reshape(n_vec, cols)
    y8, _ = orc.matvec(Q5_K, Q8_K, W, rows, cols, xq, n_vec)
    assert np.allclose(y8, xhat @ Wd.T, rtol=0, atol=1e-9)
