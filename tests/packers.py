"""Test-side block packers and closed-form decoders.

Written independently of the oracle (no shared code) from the field layouts of
the GGUF block conventions, so that oracle tests can build blocks from chosen
field values and check the decoded weights against the closed forms:
  Q4_0 w = d*(q-8)      Q5_0 w = d*(q-16)     Q8_0 w = d*q
  Q4_K w = d*sc*q - dmin*m                    Q6_K w = d*sc*(q-32)
  MXFP4 w = 2^(e-127) * E2M1(code)
(the formats of the "Models and formats" page, "Tensor formats").
"""
import numpy as np

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16 = 1, 2, 3, 4, 5, 6, 7, 8, 9
TYPES = {"Q4_0": Q4_0, "Q5_0": Q5_0, "Q8_0": Q8_0, "Q4_K": Q4_K, "Q6_K": Q6_K, "MXFP4": MXFP4}

# OCP MX E2M1 values for codes 0..7 (codes 8..15 are the negatives).
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e2m1(code):
    v = E2M1[code & 7]
    return -v if code & 8 else v


def f16_bytes(d):
    return np.array([d], dtype="<f2").view(np.uint8).tobytes()


def f16_val(d):
    return float(np.float16(d))


def _nib_pack(q):
    """32 4-bit values -> 16 bytes, element j low nibble of byte j, j+16 high nibble."""
    q = np.asarray(q)
    return bytes(int(q[j]) | (int(q[j + 16]) << 4) for j in range(16))


def pack_q4_0(d, q):
    return f16_bytes(d) + _nib_pack(q)


def closed_q4_0(d, q):
    return [f16_val(d) * (int(x) - 8) for x in q]


def pack_q5_0(d, q):
    q = np.asarray(q)
    mask = 0
    for i in range(32):
        mask |= ((int(q[i]) >> 4) & 1) << i
    return f16_bytes(d) + int(mask).to_bytes(4, "little") + _nib_pack(q & 15)


def closed_q5_0(d, q):
    return [f16_val(d) * (int(x) - 16) for x in q]


def pack_q8_0(d, q):
    return f16_bytes(d) + np.asarray(q, dtype=np.int8).tobytes()


def closed_q8_0(d, q):
    return [f16_val(d) * int(x) for x in q]


def pack_mxfp4(e, codes):
    return bytes([e]) + _nib_pack(codes)


def closed_mxfp4(e, codes):
    return [2.0 ** (e - 127) * e2m1(int(c)) for c in codes]


def pack_q4_k_scales(sc, m):
    """Eight 6-bit scales and mins -> the 12-byte field (low 6 bits of bytes 0..7
    hold sc0..3 and m0..3; their top 2 bits the high bits of sc4..7 / m4..7;
    bytes 8..11 the low 4 bits of sc4..7 (low nibble) and m4..7 (high nibble))."""
    f = [0] * 12
    for j in range(4):
        f[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        f[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        f[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return bytes(f)


def pack_q4_k(d, dmin, sc, m, q):
    q = np.asarray(q)
    qs = bytearray(128)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = int(q[64 * c + l]) | (int(q[64 * c + 32 + l]) << 4)
    return f16_bytes(d) + f16_bytes(dmin) + pack_q4_k_scales(sc, m) + bytes(qs)


def closed_q4_k(d, dmin, sc, m, q):
    return [f16_val(d) * sc[i // 32] * int(q[i]) - f16_val(dmin) * m[i // 32] for i in range(256)]


def pack_q6_k(d, sc, q):
    q = np.asarray(q)
    ql = bytearray(128)
    qh = bytearray(64)
    for h in range(2):
        for l in range(32):
            b = 128 * h
            q0, q1, q2, q3 = (int(q[b + l]), int(q[b + l + 32]), int(q[b + l + 64]), int(q[b + l + 96]))
            ql[64 * h + l] = (q0 & 15) | ((q2 & 15) << 4)
            ql[64 * h + l + 32] = (q1 & 15) | ((q3 & 15) << 4)
            qh[32 * h + l] = (q0 >> 4) | ((q1 >> 4) << 2) | ((q2 >> 4) << 4) | ((q3 >> 4) << 6)
    return bytes(ql) + bytes(qh) + np.asarray(sc, dtype=np.int8).tobytes() + f16_bytes(d)


def closed_q6_k(d, sc, q):
    return [f16_val(d) * int(sc[i // 16]) * (int(q[i]) - 32) for i in range(256)]


def random_block(t, g):
    """Random field values for one block -> (bytes, closed-form weights as float64 list)."""
    d = float(np.float16(g.normal() * 0.05))
    if t == Q4_0:
        q = g.integers(0, 16, 32)
        return pack_q4_0(d, q), closed_q4_0(d, q)
    if t == Q5_0:
        q = g.integers(0, 32, 32)
        return pack_q5_0(d, q), closed_q5_0(d, q)
    if t == Q8_0:
        q = g.integers(-128, 128, 32)
        return pack_q8_0(d, q), closed_q8_0(d, q)
    if t == MXFP4:
        e = int(g.integers(100, 150))
        c = g.integers(0, 16, 32)
        return pack_mxfp4(e, c), closed_mxfp4(e, c)
    if t == Q4_K:
        dmin = float(np.float16(abs(g.normal()) * 0.01))
        sc = [int(v) for v in g.integers(0, 64, 8)]
        m = [int(v) for v in g.integers(0, 64, 8)]
        q = g.integers(0, 16, 256)
        return pack_q4_k(d, dmin, sc, m, q), closed_q4_k(d, dmin, sc, m, q)
    if t == Q6_K:
        sc = g.integers(-128, 128, 16)
        q = g.integers(0, 64, 256)
        return pack_q6_k(d, sc, q), closed_q6_k(d, sc, q)
    raise ValueError(t)


def random_matrix(t, rows, nblk, g):
    """rows x nblk random blocks -> (bytes as uint8 array, closed-form fp64 weights [rows][cols])."""
    data = bytearray()
    W = []
    for _ in range(rows):
        row = []
        for _ in range(nblk):
            b, w = random_block(t, g)
            data += b
            row += w
        W.append(row)
    return np.frombuffer(bytes(data), dtype=np.uint8).copy(), np.array(W, dtype=np.float64)


def read_golden(path):
    """Parse tests/golden/handbuilt_blocks.txt -> list of (name, type, bytes, expected)."""
    recs = []
    cur = {}

    def expand(tokens, conv):
        out = []
        for t in tokens:
            if "*" in t:
                n, v = t.split("*", 1)
                out += [conv(v)] * int(n)
            else:
                out.append(conv(t))
        return out

    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "name":
            cur = {"name": rest}
            recs.append(cur)
        elif key == "type":
            cur["type"] = TYPES[rest]
        elif key == "hex":
            parts = []
            for tok in rest.split():
                if "*" in tok:
                    n, v = tok.split("*", 1)
                    parts.append(v * int(n))
                else:
                    parts.append(tok)
            cur["bytes"] = bytes.fromhex("".join(parts))
        elif key == "expect":
            cur["expect"] = expand(rest.split(), float)
    return [(r["name"], r["type"], r["bytes"], r["expect"]) for r in recs]


# ---- Q4_1 / Q5_1: w = d*q + m (unsigned codes, a per-block offset) ----------------

def pack_q4_1(d, m, q):
    return f16_bytes(d) + f16_bytes(m) + _nib_pack(q)


def pack_q5_1(d, m, q):
    q = np.asarray(q)
    mask = 0
    for i in range(32):
        mask |= ((int(q[i]) >> 4) & 1) << i
    return f16_bytes(d) + f16_bytes(m) + int(mask).to_bytes(4, "little") + _nib_pack(q & 15)


def closed_q_1(d, m, q):
    return [f16_val(d) * int(x) + f16_val(m) for x in q]


# ---- Q5_K: Q4_K's fields plus a 32-byte field of fifth bits ---------------------

def pack_q5_k(d, dmin, sc, m, q):
    """Element 32j+l (sub-block j): low 4 bits as in Q4_K, bit 4 in bit j of byte l."""
    q = np.asarray(q)
    qh = bytearray(32)
    qs = bytearray(128)
    for j in range(8):
        for l in range(32):
            qh[l] |= ((int(q[32 * j + l]) >> 4) & 1) << j
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = (int(q[64 * c + l]) & 15) | ((int(q[64 * c + 32 + l]) & 15) << 4)
    return f16_bytes(d) + f16_bytes(dmin) + pack_q4_k_scales(sc, m) + bytes(qh) + bytes(qs)


# ---- Q2_K and Q3_K: 2-bit codes in 128-element halves --------------------------

def _k23_pos(e):
    """Element e -> (code byte 32n+l, bit shift 2j, sub-block 8n+2j+(l>=16), l, n, j)."""
    n, rem = divmod(e, 128)
    j, l = divmod(rem, 32)
    return 32 * n + l, 2 * j, 8 * n + 2 * j + (1 if l >= 16 else 0), l, n, j


def pack_q2_k(d, dmin, sc, m, q):
    """sc, m: sixteen 4-bit scales and mins; q: 256 codes 0..3."""
    scales = bytes((int(sc[i]) & 15) | ((int(m[i]) & 15) << 4) for i in range(16))
    qs = bytearray(64)
    for e in range(256):
        byte, shift, _, _, _, _ = _k23_pos(e)
        qs[byte] |= (int(q[e]) & 3) << shift
    return scales + bytes(qs) + f16_bytes(d) + f16_bytes(dmin)


def closed_q2_k(d, dmin, sc, m, q):
    out = []
    for e in range(256):
        s = _k23_pos(e)[2]
        out.append(f16_val(d) * int(sc[s]) * int(q[e]) - f16_val(dmin) * int(m[s]))
    return out


def pack_q3_k(d, s6, code):
    """s6: sixteen 6-bit scales (factor s6 - 32); code: 256 values in -4..3, kept
    as low 2 bits plus a mask bit that is set for codes 0..3."""
    hm = bytearray(32)
    qs = bytearray(64)
    for e in range(256):
        byte, shift, _, l, n, j = _k23_pos(e)
        c = int(code[e])
        qs[byte] |= ((c + 4) & 3 if c < 0 else c) << shift
        hm[l] |= (1 if c >= 0 else 0) << (4 * n + j)
    sf = bytearray(12)
    for s in range(16):
        v = int(s6[s])
        if s < 8:
            sf[s] |= v & 15
        else:
            sf[s - 8] |= (v & 15) << 4
        sf[8 + s % 4] |= ((v >> 4) & 3) << (2 * (s // 4))
    return bytes(hm) + bytes(qs) + bytes(sf) + f16_bytes(d)


def closed_q3_k(d, s6, code):
    return [f16_val(d) * (int(s6[_k23_pos(e)[2]]) - 32) * int(code[e]) for e in range(256)]

