"""Pins of the oracle's Q4_1 / Q5_1 decoding and products, no GPU.

The formats are on the "Models and formats" page ("Tensor formats": Q4_0/1 and
Q5_0/1 are read and written); the byte layout is the GGUF one (fp16 d, fp16 m,
for Q5_1 the 32 fifth bits, then the nibbles as in Q4_0), w = d*q + m.  Pinned
by hand-built blocks, closed forms on independently packed blocks, the
position bijection, brute-force integer dots and dense fp64 products."""
import numpy as np
import pytest

import packers as P

Q4_1, Q5_1, Q8_0, F32 = 10, 11, 3, 8


def test_handbuilt_q4_1(orc):
    # d = 0.5, m = -4, codes 0..15 twice: w = q/2 - 4
    blob = bytes.fromhex("0038" + "00c4" + "00112233445566778899aabbccddeeff")
    w = orc.dequant(Q4_1, np.frombuffer(blob, dtype=np.uint8), 1, 32)[0]
    assert np.array_equal(w, (np.arange(32) % 16 * 0.5 - 4).astype(np.float32))


def test_handbuilt_q5_1(orc):
    # d = 0.25, m = -4, codes 0..31: w = q/4 - 4
    blob = bytes.fromhex("0034" + "00c4" + "0000ffff" + "00112233445566778899aabbccddeeff")
    w = orc.dequant(Q5_1, np.frombuffer(blob, dtype=np.uint8), 1, 32)[0]
    assert np.array_equal(w, (np.arange(32) * 0.25 - 4).astype(np.float32))


def _random(t, g):
    d = float(np.float16(g.normal() * 0.05))
    m = float(np.float16(g.normal() * 0.5))
    q = g.integers(0, 16 if t == Q4_1 else 32, 32)
    blob = P.pack_q4_1(d, m, q) if t == Q4_1 else P.pack_q5_1(d, m, q)
    return blob, P.closed_q_1(d, m, q)


@pytest.mark.parametrize("t", [Q4_1, Q5_1])
def test_closed_form_random_blocks(orc, t):
    g = np.random.default_rng(200 + t)
    for _ in range(300):
        blob, ref = _random(t, g)
        w = orc.dequant(t, np.frombuffer(blob, dtype=np.uint8), 1, 32)[0]
        # one rounding of the exact d*q + m
        assert np.array_equal(w, np.array(ref, dtype=np.float64).astype(np.float32)), t


@pytest.mark.parametrize("t", [Q4_1, Q5_1])
def test_each_position_moves_one_element(orc, t):
    pack = P.pack_q4_1 if t == Q4_1 else P.pack_q5_1
    hi = 12 if t == Q4_1 else 29
    for pos in range(32):
        base = np.full(32, 3)
        alt = base.copy()
        alt[pos] = hi
        wa = orc.dequant(t, np.frombuffer(pack(1.0, 0.5, base), dtype=np.uint8), 1, 32)[0]
        wb = orc.dequant(t, np.frombuffer(pack(1.0, 0.5, alt), dtype=np.uint8), 1, 32)[0]
        assert list(np.nonzero(wa != wb)[0]) == [pos]


def _matrix(t, rows, cols, seed):
    g = np.random.default_rng(seed)
    blobs, ws = [], []
    for _ in range(rows * cols // 32):
        b, w = _random(t, g)
        blobs.append(b)
        ws.append(w)
    return np.frombuffer(b"".join(blobs), dtype=np.uint8).copy(), np.array(ws, dtype=np.float64).reshape(rows, cols)


@pytest.mark.parametrize("t", [Q4_1, Q5_1])
def test_block_dots_brute_force(orc, t):
    """S = sum q * xq (exact) and Mn = sum xq per block."""
    rows, cols = 5, 96
    W, _ = _matrix(t, rows, cols, 3)
    x = np.random.default_rng(4).standard_normal((2, cols)).astype(np.float32)
    xq = orc.quantize_act(Q8_0, x)
    out = orc.block_dots(t, W, rows, cols, xq, 2)
    codes = np.zeros((rows, cols), dtype=np.int64)
    bb = 20 if t == Q4_1 else 24
    for r in range(rows):
        for b in range(cols // 32):
            blk = W[(r * (cols // 32) + b) * bb:(r * (cols // 32) + b + 1) * bb]
            qs = blk[4:20] if t == Q4_1 else blk[8:24]
            lo, hi = (qs & 15).astype(np.int64), (qs >> 4).astype(np.int64)
            q = np.concatenate([lo, hi])
            if t == Q5_1:
                qh = int.from_bytes(bytes(blk[4:8]), "little")
                q = q + 16 * np.array([(qh >> i) & 1 for i in range(32)])
            codes[r, 32 * b:32 * b + 32] = q
    xc = np.frombuffer(xq.tobytes(), dtype=np.uint8).reshape(2, cols // 32, 34)[:, :, 2:].view(np.int8).astype(np.int64)
    for v in range(2):
        for r in range(rows):
            for b in range(cols // 32):
                S = int(np.dot(codes[r, 32 * b:32 * b + 32], xc[v, b]))
                Mn = int(xc[v, b].sum())
                assert tuple(out[v, r, b]) == (S, Mn)


@pytest.mark.parametrize("t", [Q4_1, Q5_1])
def test_matvec_dense_brute_force(orc, t):
    rows, cols = 7, 128
    W, Wd = _matrix(t, rows, cols, 5)
    x = np.random.default_rng(6).standard_normal((3, cols)).astype(np.float32)
    y, _ = orc.matvec(t, F32, W, rows, cols, x, 3)
    assert np.allclose(y, x.astype(np.float64) @ Wd.T, rtol=0, atol=1e-9)
    xq = orc.quantize_act(Q8_0, x)
    xhat = np.zeros_like(x, dtype=np.float64)
    blocks = np.frombuffer(xq.tobytes(), dtype=np.uint8).reshape(3, cols // 32, 34)
    for v in range(3):
        for b in range(cols // 32):
            d = float(np.frombuffer(blocks[v, b, :2].tobytes(), dtype=np.float16)[0])
            xhat[v, 32 * b:32 * b + 32] = d * blocks[v, b, 2:].view(np.int8).astype(np.float64)
    y8, _ = orc.matvec(t, Q8_0, W, rows, cols, xq, 3)
    assert np.allclose(y8, xhat @ Wd.T, rtol=0, atol=1e-9)
