"""Pins for the CPU oracle: it is checked against facts that do not come from
itself -- hand-built blocks (tests/golden), closed forms evaluated on fields
packed by an independent test-side packer, numpy/torch conversions, dense
fp64 products on tiny matrices, and invariants of the method.

Runs on CPU only (no GPU needed).
"""
import os

import numpy as np
import pytest
import torch

import packers as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "handbuilt_blocks.txt")
WEIGHT_TYPES = [P.Q4_0, P.Q5_0, P.Q8_0, P.MXFP4, P.Q4_K, P.Q6_K]


# ---- fp16 / bf16 ---------------------------------------------------------------

def test_f16_decode_exhaustive(orc):
    h = np.arange(65536, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(v)) for v in h])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_encode_matches_numpy(orc):
    g = np.random.default_rng(1)
    vals = np.concatenate([
        (g.standard_normal(20000) * np.exp2(g.integers(-30, 20, 20000))).astype(np.float32),
        np.float32([0.0, -0.0, 65504, 65519.996, 65520, 65536, 1e-8, 2.0 ** -24, 2.0 ** -25,
                    3 * 2.0 ** -26, 2.0 ** -14, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, np.inf, -np.inf]),
    ])
    # ties: odd multiples of half an fp16 ulp around several binades
    ties = np.float32([(1 + (2 * k + 1) * 2.0 ** -11) * 2.0 ** s for k in range(8) for s in (-20, -3, 0, 7)])
    vals = np.concatenate([vals, ties, -ties])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16_rn(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_decode_matches_torch(orc):
    g = np.random.default_rng(2)
    vals = (g.standard_normal(20000) * np.exp2(g.integers(-60, 60, 20000))).astype(np.float32)
    ties = np.float32([(1 + (2 * k + 1) * 2.0 ** -8) for k in range(16)])
    vals = np.concatenate([vals, ties, -ties, np.float32([0.0, 3.3895314e38, np.inf])])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16_rn(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([orc.bf16_to_f64(int(b)) for b in ref[:2000]])
    assert np.array_equal(back, torch.from_numpy(ref[:2000].view(np.int16)).view(torch.bfloat16).double().numpy())


# ---- hand-built blocks ----------------------------------------------------------

@pytest.mark.parametrize("rec", P.read_golden(GOLDEN), ids=lambda r: r[0])
def test_handbuilt_block(orc, rec):
    name, t, blob, expect = rec
    assert len(blob) == orc.BLOCK_BYTES[t], name
    n = orc.BLOCK_ELEMS[t]
    assert len(expect) == n, name
    w = orc.dequant(t, np.frombuffer(blob, dtype=np.uint8), 1, n)[0]
    assert np.array_equal(w.astype(np.float64), np.array(expect)), name


# ---- closed forms on independently packed random blocks ------------------------

@pytest.mark.parametrize("t", WEIGHT_TYPES)
def test_closed_form_random_blocks(orc, t):
    g = np.random.default_rng(100 + t)
    n = orc.BLOCK_ELEMS[t]
    for _ in range(200):
        blob, ref = P.random_block(t, g)
        w = orc.dequant(t, np.frombuffer(blob, dtype=np.uint8), 1, n)[0]
        # every format's weight is exactly representable in fp32 except Q4_K's,
        # which is the single rounding of the exact value
        assert np.array_equal(w, np.float32(np.array(ref))), t


@pytest.mark.parametrize("t", WEIGHT_TYPES)
def test_each_position_moves_one_element(orc, t):
    """Changing the code of one element changes exactly one decoded weight:
    the element order is a bijection (no two positions share bits)."""
    n = orc.BLOCK_ELEMS[t]
    g = np.random.default_rng(7)
    hit = np.zeros(n, dtype=int)
    for pos in range(n):
        if t == P.Q4_0:
            base = np.full(32, 3); alt = base.copy(); alt[pos] = 12
            a, b = P.pack_q4_0(1.0, base), P.pack_q4_0(1.0, alt)
        elif t == P.Q5_0:
            base = np.full(32, 3); alt = base.copy(); alt[pos] = 29
            a, b = P.pack_q5_0(1.0, base), P.pack_q5_0(1.0, alt)
        elif t == P.Q8_0:
            base = np.full(32, 3); alt = base.copy(); alt[pos] = -100
            a, b = P.pack_q8_0(1.0, base), P.pack_q8_0(1.0, alt)
        elif t == P.MXFP4:
            base = np.full(32, 3); alt = base.copy(); alt[pos] = 14
            a, b = P.pack_mxfp4(127, base), P.pack_mxfp4(127, alt)
        elif t == P.Q4_K:
            sc = list(range(1, 9)); m = list(range(8))
            base = np.full(256, 3); alt = base.copy(); alt[pos] = 12
            a, b = P.pack_q4_k(1.0, 0.5, sc, m, base), P.pack_q4_k(1.0, 0.5, sc, m, alt)
        else:
            sc = g.integers(1, 100, 16)
            base = np.full(256, 3); alt = base.copy(); alt[pos] = 60
            a, b = P.pack_q6_k(1.0, sc, base), P.pack_q6_k(1.0, sc, alt)
        wa = orc.dequant(t, np.frombuffer(a, dtype=np.uint8), 1, n)[0]
        wb = orc.dequant(t, np.frombuffer(b, dtype=np.uint8), 1, n)[0]
        diff = np.nonzero(wa != wb)[0]
        assert list(diff) == [pos], (t, pos, diff)
        hit[pos] += 1
    assert (hit == 1).all()


def test_q4_k_scale_field_bijection(orc):
    """The 12-byte Q4_K field carries 96 bits = 8 x (6 + 6): every pattern of
    scales/mins survives pack -> decode, and every random field decodes to
    values that re-pack to the same bytes."""
    g = np.random.default_rng(11)
    for _ in range(300):
        f = g.integers(0, 256, 12, dtype=np.uint8).tobytes()
        blob = P.f16_bytes(1.0) + P.f16_bytes(1.0) + f + bytes(128)   # all codes 0
        dec = orc.decode_block(P.Q4_K, blob)
        sc = [int(dec["sub_scale"][32 * j]) for j in range(8)]
        m = [int(dec["sub_min"][32 * j]) for j in range(8)]
        assert P.pack_q4_k_scales(sc, m) == f


def test_mxfp4_e2m1_table(orc):
    """E2M1 decoded bit by bit in the oracle against the OCP table; E8M0 scale."""
    for e in (0, 1, 118, 127, 128, 130, 254):
        for c in range(16):
            codes = np.zeros(32, dtype=int); codes[5] = c
            w = orc.dequant(P.MXFP4, np.frombuffer(P.pack_mxfp4(e, codes), dtype=np.uint8), 1, 32)[0]
            assert w[5] == np.float32(2.0 ** (e - 127) * P.e2m1(c)), (e, c)
    w = orc.dequant(P.MXFP4, np.frombuffer(P.pack_mxfp4(128, [1] + [15] * 31), dtype=np.uint8), 1, 32)[0]
    assert w[0] == 1.0 and w[1] == -12.0


# ---- activation quantiser --------------------------------------------------------

def test_q8_0_hand_example(orc):
    # amax 127 -> d = 1 exactly, id = 1; halves round away from zero
    x = np.zeros(32, dtype=np.float32)
    x[:8] = [127, -63.5, 63.5, 0.5, -0.5, 1.49, -2.5, 126.5]
    out = orc.quantize_act(P.Q8_0, x)
    assert out[:2].tobytes() == bytes([0x00, 0x3C])
    q = out[2:].view(np.int8)
    assert list(q[:8]) == [127, -64, 64, 1, -1, 1, -3, 127]
    assert (q[8:] == 0).all()


def test_q8_zero_block(orc):
    for t in (P.Q8_0, P.Q8_K):
        n = 32 if t == P.Q8_0 else 256
        out = orc.quantize_act(t, np.zeros(n, dtype=np.float32))
        assert not out.any()


@pytest.mark.parametrize("t", [P.Q8_0, P.Q8_K])
def test_quantiser_properties(orc, t):
    g = np.random.default_rng(5)
    bs = 32 if t == P.Q8_0 else 256
    x = (g.standard_normal((64, bs)) * np.exp2(g.integers(-8, 8, (64, 1)))).astype(np.float32)
    out = orc.quantize_act(t, x.reshape(-1))
    bb = orc.BLOCK_BYTES[t]
    for b in range(64):
        blk = out[b * bb:(b + 1) * bb]
        if t == P.Q8_0:
            d_st = float(blk[:2].view(np.float16)[0]); q = blk[2:34].view(np.int8).astype(int)
        else:
            d_st = float(blk[:4].view(np.float32)[0]); q = blk[4:260].view(np.int8).astype(int)
            bsums = blk[260:292].view(np.int16).astype(int)
            assert np.array_equal(bsums, q.reshape(16, 16).sum(1))
        amax = np.abs(x[b]).max()
        d32 = np.float32(amax) / np.float32(127)
        i = np.abs(x[b]).argmax()
        assert q[i] == (127 if x[b][i] > 0 else -127)
        assert np.abs(q).max() <= 127
        # round-trip against the fp32 scale the codes were taken with
        err = np.abs(x[b].astype(np.float64) - float(d32) * q)
        assert (err <= float(d32) * (0.5 + 1e-5)).all()
        # the stored scale is the fp32 scale, rounded to fp16 for Q8_0
        ref = float(np.float16(d32)) if t == P.Q8_0 else float(d32)
        assert d_st == ref


@pytest.mark.parametrize("t", [P.Q8_0, P.Q8_K])
def test_quantiser_scale_below_2_pow_minus_128(orc, t):
    """A block whose amax/127 is below 2^-128, so that 1/d overflows: the codes
    are round(x / d) of the plain definition -- zero stays 0, the extreme
    is +-127, every code a nearest integer of the exact quotient -- not the
    saturated or undefined values of x * inf."""
    bs = 32 if t == P.Q8_0 else 256
    g = np.random.default_rng(17)
    amax = np.float32(1e-37)
    x = (g.uniform(-1, 1, bs) * amax).astype(np.float32)
    x[3] = amax
    x[10] = -amax / np.float32(2)
    x[0] = 0.0
    x[7] = -0.0
    x[bs - 1] = 0.0
    out = orc.quantize_act(t, x)
    d = np.float32(amax) / np.float32(127)
    assert float(d) < 2.0 ** -128 and np.isinf(np.float32(1) / d)
    if t == P.Q8_0:
        q = out[2:34].view(np.int8).astype(int)
        assert out[:2].view(np.float16)[0] == 0      # fp16(d) underflows
    else:
        q = out[4:260].view(np.int8).astype(int)
        assert out[:4].view(np.float32)[0] == d
        assert np.array_equal(out[260:292].view(np.int16).astype(int), q.reshape(16, 16).sum(1))
    assert q[0] == 0 and q[7] == 0 and q[bs - 1] == 0
    assert q[3] == 127
    assert q[10] in (-63, -64)   # -amax/2 over the subnormal d (rounded to ~17 bits) is near -63.5
    # nearest integer of the exact quotient (fp64), up to the fp32 rounding of x/d
    exact = x.astype(np.float64) / float(d)
    assert (np.abs(exact - q) <= 0.5 + 1e-5).all()
    # halves away from zero, on the quotient the oracle is defined by (fp32 x/d)
    v = (x / d).astype(np.float64)
    assert np.array_equal(q, (np.sign(v) * np.floor(np.abs(v) + 0.5)).astype(int))


# ---- integer block dots ------------------------------------------------------------

@pytest.mark.parametrize("t", WEIGHT_TYPES)
def test_block_dots_brute_force(orc, t):
    g = np.random.default_rng(20 + t)
    rows, nblk, n_vec = 3, 3, 2
    bs = orc.BLOCK_ELEMS[t]
    cols = nblk * bs
    W, _ = P.random_matrix(t, rows, nblk, g)
    at = P.Q8_0 if bs == 32 else P.Q8_K
    x = g.standard_normal((n_vec, cols)).astype(np.float32)
    xq = orc.quantize_act(at, x)
    dots = orc.block_dots(t, W, rows, cols, xq, n_vec)
    rb = orc.row_bytes(t, cols)
    ab = orc.BLOCK_BYTES[at]
    for v in range(n_vec):
        for r in range(rows):
            for b in range(nblk):
                wb = orc.decode_block(t, W[r * rb + b * orc.BLOCK_BYTES[t]:][:orc.BLOCK_BYTES[t]].tobytes())
                blk = xq[v][b * ab:(b + 1) * ab]
                q = (blk[2:34] if at == P.Q8_0 else blk[4:260]).view(np.int8).astype(np.int64)
                S = int(np.sum(wb["sub_scale"].astype(np.int64) * wb["code"] * q))
                Mn = int(np.sum(wb["sub_min"].astype(np.int64) * q))
                assert tuple(dots[v, r, b]) == (S, Mn)


# ---- matrix-vector products ----------------------------------------------------------

@pytest.mark.parametrize("t", WEIGHT_TYPES)
def test_matvec_dense_brute_force(orc, t):
    """Tiny matrices built from independently packed blocks: the oracle's
    products equal dense fp64 products of the closed-form weights."""
    g = np.random.default_rng(40 + t)
    bs = orc.BLOCK_ELEMS[t]
    rows, nblk, n_vec = 4, 2 if bs == 256 else 5, 3
    cols = nblk * bs
    W, Wd = P.random_matrix(t, rows, nblk, g)
    if t == P.Q4_K:
        Wd = Wd.astype(np.float32).astype(np.float64)   # within 2^-24 of exact; the A32 check allows it
    x = g.standard_normal((n_vec, cols)).astype(np.float32)
    # A32
    y, ya = orc.matvec(t, P.F32, W, rows, cols, x, n_vec)
    ref = x.astype(np.float64) @ Wd.T
    scale = np.abs(x.astype(np.float64)) @ np.abs(Wd.T)
    assert (np.abs(y - ref) <= 1e-7 * scale + 1e-15).all()
    assert np.allclose(ya, scale, rtol=1e-7, atol=0)
    # A8: dense product against the dequantised activations d_x * q
    at = P.Q8_0 if bs == 32 else P.Q8_K
    xq = orc.quantize_act(at, x)
    ab = orc.BLOCK_BYTES[at]
    xh = np.zeros((n_vec, cols))
    for v in range(n_vec):
        for b in range(cols // bs):
            blk = xq[v][b * ab:(b + 1) * ab]
            if at == P.Q8_0:
                d = float(blk[:2].view(np.float16)[0]); q = blk[2:34].view(np.int8)
            else:
                d = float(blk[:4].view(np.float32)[0]); q = blk[4:260].view(np.int8)
            xh[v, b * bs:(b + 1) * bs] = d * q.astype(np.float64)
    y8, ya8 = orc.matvec(t, at, W, rows, cols, xq, n_vec)
    _, Wexact = P.random_matrix(t, rows, nblk, np.random.default_rng(40 + t))
    ref8 = xh @ Wexact.T
    assert np.allclose(y8, ref8, rtol=1e-12, atol=1e-12 * (np.abs(xh) @ np.abs(Wexact.T)).max())
    # bf16: both operands rounded to bf16, products exact in fp64
    xb = torch.from_numpy(x).to(torch.bfloat16)
    Wb = torch.from_numpy(Wd.astype(np.float32)).to(torch.bfloat16).double().numpy()
    yb, _ = orc.matvec(t, P.BF16, W, rows, cols, xb.view(torch.int16).numpy(), n_vec)
    refb = xb.double().numpy() @ Wb.T
    assert np.allclose(yb, refb, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("t", [P.Q4_0, P.Q4_K, P.MXFP4])
def test_a8_vs_a32_quantisation_bound(orc, t):
    """|y_A8 - y_A32| <= sum_i |w_i| * (d32/2 + 127*|d_stored - d32|) + fp rounding."""
    from gguf_block_quantised_gb300 import synth
    bs = orc.BLOCK_ELEMS[t]
    rows, cols = 16, 4 * bs
    W = synth.weights(t, rows, cols, seed=9, tensor_id=1)
    x = synth.activations(2, cols, seed=9)
    at = P.Q8_0 if bs == 32 else P.Q8_K
    xq = orc.quantize_act(at, x)
    y32, _ = orc.matvec(t, P.F32, W, rows, cols, x, 2)
    y8, _ = orc.matvec(t, at, W, rows, cols, xq, 2)
    Wd = np.abs(orc.dequant(t, W, rows, cols).astype(np.float64))
    xb = np.abs(x).reshape(2, -1, bs).max(-1).astype(np.float32)
    d32 = xb / np.float32(127)
    dst = d32.astype(np.float16).astype(np.float64) if at == P.Q8_0 else d32.astype(np.float64)
    per = d32 / 2 + 127 * np.abs(dst - d32)                   # [2][nblocks]
    bound = np.einsum("rbk,vb->vr", Wd.reshape(rows, -1, bs), per)
    assert (np.abs(y8 - y32) <= bound * (1 + 1e-6) + 1e-9).all()


def test_batched_equals_sequential(orc):
    """Batched prefill equals sequential decode, bit for bit."""
    from gguf_block_quantised_gb300 import synth
    t, rows, cols = P.Q5_0, 40, 96
    W = synth.weights(t, rows, cols, seed=3)
    x = synth.activations(5, cols, seed=3)
    y, _ = orc.matvec(t, P.F32, W, rows, cols, x, 5)
    for v in range(5):
        y1, _ = orc.matvec(t, P.F32, W, rows, cols, x[v:v + 1], 1)
        assert np.array_equal(y1[0], y[v])
    ids = np.array([7, 0, 39, 3])
    ys, _ = orc.matvec(t, P.F32, W, rows, cols, x, 5, row_ids=ids)
    assert np.array_equal(ys, y[:, ids])


def test_shape_and_type_errors(orc):
    W = np.zeros(1000, dtype=np.uint8)
    x = np.zeros((1, 40), dtype=np.float32)
    with pytest.raises(orc.OracleError):
        orc.matvec(P.Q4_0, P.F32, W, 1, 40, x, 1)          # 40 is not a multiple of 32
    with pytest.raises(orc.OracleError):
        orc.matvec(P.Q4_0, P.Q8_K, W, 1, 256, np.zeros(292, np.uint8), 1)   # wrong activation pairing
    with pytest.raises(orc.OracleError):
        orc.quantize_act(P.Q4_0, np.zeros(32, np.float32))


# ---- mixture of experts -----------------------------------------------------------------

def _moe_inputs(t, n_expert, rows, cols, n_tok, k, seed):
    from gguf_block_quantised_gb300 import synth
    W3 = synth.weights(t, n_expert * rows, cols, seed=seed, tensor_id=1)
    ids, gates = synth.router(n_tok, n_expert, k, seed=seed)
    b = synth.bias(n_expert, rows, seed=seed)
    return W3, ids, gates, b


def test_moe_single_expert_is_matvec_plus_bias(orc):
    from gguf_block_quantised_gb300 import synth
    t, rows, cols = P.MXFP4, 24, 64
    W3, _, _, b = _moe_inputs(t, 1, rows, cols, 3, 1, 4)
    x = synth.activations(3, cols, seed=4)
    ids = np.zeros((3, 1), np.int32)
    y, _ = orc.moe(t, P.F32, W3, 1, rows, cols, ids, None, 1, x, 3, bias=b)
    ref, _ = orc.matvec(t, P.F32, W3, rows, cols, x, 3)
    assert np.allclose(y[:, 0, :], ref + b[0], rtol=1e-14, atol=1e-14)
    g1 = np.ones((3, 1), np.float32)
    y2, _ = orc.moe(t, P.F32, W3, 1, rows, cols, ids, g1, 1, x, 3, bias=b)
    assert np.array_equal(y2, y[:, 0, :])


def test_moe_against_per_expert_matvec(orc):
    """Both MoE forms equal per-(token, slot) matvecs of the routed expert's
    slice of the stacked tensor, plus its bias, gate-weighted in slot order."""
    from gguf_block_quantised_gb300 import synth
    t, E, rows, cols, n_tok, k = P.MXFP4, 6, 16, 64, 5, 3
    W3, ids, gates, b = _moe_inputs(t, E, rows, cols, n_tok, k, 6)
    rb = orc.row_bytes(t, cols)
    x = synth.activations(n_tok, cols, seed=6)
    y, _ = orc.moe(t, P.F32, W3, E, rows, cols, ids, None, k, x, n_tok, bias=b)
    h = synth.activations(n_tok * k, cols, seed=6, tensor_id=77).reshape(n_tok, k, cols)
    yc, _ = orc.moe(t, P.F32, W3, E, rows, cols, ids, gates, k, h, n_tok, bias=b)
    for tok in range(n_tok):
        comb = np.zeros(rows)
        for s in range(k):
            e = ids[tok, s]
            We = W3[e * rows * rb:(e + 1) * rows * rb]
            ref, _ = orc.matvec(t, P.F32, We, rows, cols, x[tok:tok + 1], 1)
            assert np.allclose(y[tok, s], ref[0] + b[e], rtol=1e-14, atol=1e-14)
            r2, _ = orc.matvec(t, P.F32, We, rows, cols, h[tok, s:s + 1], 1)
            comb += float(gates[tok, s]) * (r2[0] + b[e])
        assert np.allclose(yc[tok], comb, rtol=1e-13, atol=1e-13)


def test_moe_rejects_bad_expert_id(orc):
    t, E, rows, cols = P.MXFP4, 4, 8, 32
    W3, _, _, _ = _moe_inputs(t, E, rows, cols, 1, 1, 1)
    x = np.zeros((1, cols), np.float32)
    with pytest.raises(orc.OracleError):
        orc.moe(t, P.F32, W3, E, rows, cols, np.array([[4]], np.int32), None, 1, x, 1)
