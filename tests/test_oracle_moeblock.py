"""Pins of the oracle's mixture-of-experts block, no GPU.

"Models and formats" page, "Architectures": a router picks k of n experts per
token; gpt-oss gates with a clipped SwiGLU whose linear half is offset by one
and has a bias on every expert projection.  The pages fix neither the router's
arithmetic nor the clipping constants; the readings (router logit in fp32 as
32 partial fused multiply-add sums combined by an xor butterfly, top k with
ties to the lower id, fp64 softmax over the kept logits, gate rows [0, I) and
linear rows [I, 2I)) are pinned here by integer-exact dot products, hand-worked
rounding cases, numpy's stable sort, scipy's softmax, closed forms of the
sigmoid and a dense fp64 composition over independently decoded weights."""
import math

import numpy as np
import pytest
import scipy.special

from gguf_block_quantised_gb300 import synth

Q4_0, Q8_0, F32 = 1, 3, 8


# ---- router ------------------------------------------------------------------------

def test_router_integer_inputs_are_exact(orc):
    # every partial sum of small integers is exact in fp32, so any order gives the
    # integer dot product; a dropped term, a transposed Wr or a wrong stride does not
    g = np.random.default_rng(1)
    for hidden in (1, 31, 32, 100, 257):
        x = g.integers(-8, 9, (5, hidden)).astype(np.float32)
        Wr = g.integers(-8, 9, (7, hidden)).astype(np.float32)
        br = g.integers(-50, 51, 7).astype(np.float32)
        exact = x.astype(np.int64) @ Wr.astype(np.int64).T + br.astype(np.int64)
        assert np.array_equal(orc.router(x, Wr, br), exact.astype(np.float32))
        assert np.array_equal(orc.router(x, Wr), (exact - br.astype(np.int64)).astype(np.float32))


@pytest.mark.parametrize("case", ["lane_then_tree", "tree_levels"])
def test_router_order(orc, case):
    big = np.float32(2.0 ** 24)
    if case == "lane_then_tree":
        # partial 0 holds elements 0 and 32: 2^24 then + 1 rounds back to 2^24 (ties to
        # even); partial 1 holds elements 1 and 33: 1 + 1 = 2; the tree then adds
        # 2^24 + 2 exactly.  The exact sum 2^24 + 3 is not an fp32 value; a
        # left-to-right sum loses every + 1 and gives 2^24.
        x = np.ones((1, 64), np.float32)
        w = np.zeros((1, 64), np.float32)
        w[0, 0], w[0, 32], w[0, 1], w[0, 33] = big, 1, 1, 1
        assert orc.router(x, w)[0, 0] == np.float32(2.0 ** 24 + 2)
    else:
        # partials 0 and 16 meet at the first level (o = 16): 2^24 + 1 -> 2^24; partial
        # 1 carries 3 and meets them at the last level: 2^24 + 3 -> 2^24 + 4.
        x = np.ones((1, 32), np.float32)
        w = np.zeros((1, 32), np.float32)
        w[0, 0], w[0, 16], w[0, 1] = big, 1, 3
        assert orc.router(x, w)[0, 0] == np.float32(2.0 ** 24 + 4)
        # the same values with the 1 in partial 1 and the 3 in partial 16: the first
        # level gives 2^24 + 3 -> 2^24 + 4, the last adds 1 -> 2^24 + 4 (ties to even)
        w[0, 16], w[0, 1] = 3, 1
        assert orc.router(x, w)[0, 0] == np.float32(2.0 ** 24 + 4)


def test_router_error_bound(orc):
    # fp32 with fused multiply-adds: within (hidden/32 + 5 + 1) roundings of the
    # exact sum, relative to sum |x w| + |b|
    g = np.random.default_rng(2)
    for hidden in (96, 2880):
        x = g.standard_normal((9, hidden)).astype(np.float32)
        Wr = (g.standard_normal((33, hidden)) * 0.02).astype(np.float32)
        br = (g.standard_normal(33) * 0.02).astype(np.float32)
        got = orc.router(x, Wr, br).astype(np.float64)
        X, W = x.astype(np.float64), Wr.astype(np.float64)
        exact = X @ W.T + br
        mag = np.abs(X) @ np.abs(W).T + np.abs(br)
        gam = (hidden / 32 + 7) * 2.0 ** -24
        assert np.all(np.abs(got - exact) <= gam * mag)


# ---- top k and gates -----------------------------------------------------------------

def test_topk_matches_stable_sort_and_softmax(orc):
    g = np.random.default_rng(3)
    for E, k in ((8, 1), (32, 4), (128, 4), (1024, 64), (5, 5)):
        logits = g.standard_normal((11, E)).astype(np.float32)
        logits[0, :] = 0.25                      # all tied: ids 0..k-1
        logits[1, ::3] = logits[1, 0]            # ties across a third of the experts
        ids, gates = orc.topk_softmax(logits, k)
        want = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, want)
        assert list(ids[0]) == list(range(k))
        sel = np.take_along_axis(logits, want, axis=1).astype(np.float64)
        np.testing.assert_allclose(gates, scipy.special.softmax(sel, axis=1), rtol=1e-14, atol=0)
        np.testing.assert_allclose(gates.sum(axis=1), 1.0, rtol=1e-14)
        assert np.all(np.diff(gates, axis=1) <= 0)   # descending logits, descending gates


def test_topk_k1_gate_is_one_and_two_way_closed_form(orc):
    logits = np.array([[0.0, 3.0, -1.0, 3.0]], np.float32)
    ids, gates = orc.topk_softmax(logits, 1)
    assert ids[0, 0] == 1 and gates[0, 0] == 1.0
    ids, gates = orc.topk_softmax(np.array([[1.0, math.log(3.0) + 1.0]], np.float32), 2)
    # the two gates are 3/4 and 1/4 up to the fp32 rounding of ln 3 + 1
    assert list(ids[0]) == [1, 0]
    assert abs(gates[0, 0] - 0.75) < 1e-6 and abs(gates[0, 1] - 0.25) < 1e-6


# ---- the clipped SwiGLU -----------------------------------------------------------------

def test_swiglu_closed_forms(orc):
    ln3 = math.log(3.0)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    assert orc.swiglu(1.0, 1.0, ln3, 7.0) == pytest.approx(1.5, rel=1e-15)
    assert orc.swiglu(-1.0, 0.0, ln3, 7.0) == pytest.approx(-0.25, rel=1e-15)
    # alpha = 0: sigmoid = 1/2
    assert orc.swiglu(3.0, 2.0, 0.0, 7.0) == pytest.approx(4.5, rel=1e-15)
    # the linear half is offset by one: u = -1 zeroes the output; g = 0 does too
    assert orc.swiglu(2.5, -1.0, 1.702, 7.0) == 0.0
    assert orc.swiglu(0.0, 5.0, 1.702, 7.0) == 0.0
    # clipping: g above the limit acts as the limit, u outside [-limit, limit] as its bound
    lim = 7.0
    assert orc.swiglu(100.0, 0.5, 1.702, lim) == orc.swiglu(lim, 0.5, 1.702, lim)
    assert orc.swiglu(1.0, 100.0, 1.702, lim) == orc.swiglu(1.0, lim, 1.702, lim)
    assert orc.swiglu(1.0, -100.0, 1.702, lim) == orc.swiglu(1.0, -lim, 1.702, lim)
    # g is clipped above only: a large negative g is kept (and its sigmoid vanishes)
    assert orc.swiglu(-100.0, 0.0, 1.0, lim) == pytest.approx(-100.0 / (1.0 + math.exp(100.0)), rel=1e-14)
    # large alpha * g: the sigmoid saturates, h -> g (u' + 1)
    assert orc.swiglu(2.0, 1.0, 60.0, lim) == pytest.approx(4.0, rel=1e-15)


# ---- composition ------------------------------------------------------------------------

def _experts(wt, E, rows, cols, seed):
    return synth.weights(wt, E * rows, cols, seed=seed, tensor_id=7 + rows)


def _dense(orc, wt, W, E, rows, cols):
    return orc.dequant(wt, W, E * rows, cols).astype(np.float64).reshape(E, rows, cols)


@pytest.mark.parametrize("wt,E,k,hidden,inter,n_tok", [(Q4_0, 8, 2, 64, 32, 3), (Q8_0, 6, 3, 96, 64, 2)])
def test_block_composition_dense(orc, wt, E, k, hidden, inter, n_tok):
    """F32 activations: the block equals router -> top k -> dense fp64 products of the
    decoded experts with the gate/linear halves, the clipped SwiGLU and the
    gate-weighted down sum."""
    g = np.random.default_rng(4)
    alpha, limit = 1.702, 7.0
    x = g.standard_normal((n_tok, hidden)).astype(np.float32)
    Wr = (g.standard_normal((E, hidden)) * 0.2).astype(np.float32)
    br = (g.standard_normal(E) * 0.1).astype(np.float32)
    Wgu = _experts(wt, E, 2 * inter, hidden, 5)
    Wd = _experts(wt, E, hidden, inter, 6)
    bgu = (g.standard_normal((E, 2 * inter)) * 0.02).astype(np.float32)
    bd = (g.standard_normal((E, hidden)) * 0.02).astype(np.float32)
    y, yabs, ids, gates = orc.moe_block(wt, F32, x, Wr, br, Wgu, bgu, Wd, bd, E, k, hidden, inter, alpha, limit)
    ids2, gates2 = orc.topk_softmax(orc.router(x, Wr, br), k)
    assert np.array_equal(ids, ids2) and np.array_equal(gates, gates2)
    Dgu, Dd = _dense(orc, wt, Wgu, E, 2 * inter, hidden), _dense(orc, wt, Wd, E, hidden, inter)
    want = np.zeros((n_tok, hidden))
    for t in range(n_tok):
        for s in range(k):
            e = ids[t, s]
            gu = Dgu[e] @ x[t].astype(np.float64) + bgu[e]
            h = orc.swiglu(gu[:inter], gu[inter:], alpha, limit).astype(np.float32).astype(np.float64)
            want[t] += np.float32(gates[t, s]) * (Dd[e] @ h + bd[e])
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-9 * (1 + np.abs(want).max()))
    assert np.all(yabs >= np.abs(y) - 1e-12)


def test_block_halves_are_gate_then_linear(orc):
    """Zero weights in one half: a zero gate half gives h = 0 (only the down bias
    remains); a zero linear half gives h = g' sigmoid(alpha g') (the offset of one)."""
    E, k, hidden, inter, n_tok = 4, 2, 32, 32, 2
    g = np.random.default_rng(5)
    x = g.standard_normal((n_tok, hidden)).astype(np.float32)
    Wr = g.standard_normal((E, hidden)).astype(np.float32)
    wgu = np.zeros((E, 2 * inter, hidden), np.float32)
    wgu[:, :inter] = g.standard_normal((E, inter, hidden)) * 0.1           # gate half only
    wd = (g.standard_normal((E, hidden, inter)) * 0.1).astype(np.float32)
    Wd = wd.view(np.uint8).reshape(-1)                                      # plain F32 experts throughout
    bd = g.standard_normal((E, hidden)).astype(np.float32)
    Wgu_gate = wgu.view(np.uint8).reshape(-1)
    y_gate, _, ids, gates = orc.moe_block(F32, F32, x, Wr, None, Wgu_gate, None, Wd, bd, E, k, hidden, inter,
                                          1.0, 7.0)
    Dd = wd.astype(np.float64)
    want = np.zeros((n_tok, hidden))
    for t in range(n_tok):
        for s in range(k):
            e = ids[t, s]
            gv = wgu[e, :inter].astype(np.float64) @ x[t].astype(np.float64)
            h = (gv / (1.0 + np.exp(-gv))).astype(np.float32)                 # g sigmoid(g) * (0 + 1)
            want[t] += np.float32(gates[t, s]) * (Dd[e] @ h + bd[e])
    np.testing.assert_allclose(y_gate, want, rtol=0, atol=1e-9 * np.abs(want).max())
    wlin = np.zeros_like(wgu)
    wlin[:, inter:] = wgu[:, :inter]                                        # linear half only
    y_lin, _, ids, gates = orc.moe_block(F32, F32, x, Wr, None, wlin.view(np.uint8).reshape(-1), None, Wd, bd,
                                         E, k, hidden, inter, 1.0, 7.0)
    want = (gates.astype(np.float32).astype(np.float64)[:, :, None] * bd[ids]).sum(axis=1)
    np.testing.assert_allclose(y_lin, want, rtol=0, atol=1e-12)
