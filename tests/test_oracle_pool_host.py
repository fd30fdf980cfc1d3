"""The all-cores oracle helper (tests/oracle_pool.py) splits and stacks
correctly: its outputs equal one single-threaded oracle call bit for bit,
for matvec (rows split) and both mixture-of-experts forms (tokens split).
No GPU."""
import numpy as np

import oracle_pool as OP
from gguf_block_quantised_gb300 import synth
from oracle import oracle as O


def test_pool_matvec_equals_single_call():
    rows, cols, n_vec = 37, 512, 3
    W = synth.weights(4, rows, cols, seed=1)
    xq = O.quantize_act(O.Q8_K, synth.activations(n_vec, cols, seed=1))
    y1, a1 = O.matvec(O.Q4_K, O.Q8_K, W, rows, cols, xq, n_vec)
    y2, a2 = OP.matvec(O.Q4_K, O.Q8_K, W, rows, cols, xq, n_vec, procs=3)
    assert np.array_equal(y1, y2) and np.array_equal(a1, a2)


def test_pool_moe_equals_single_call():
    E, rows, cols, k, n_tok = 5, 24, 64, 2, 7
    W3 = synth.weights(6, E * rows, cols, seed=2)
    ids, gates = synth.router(n_tok, E, k, seed=2)
    b = synth.bias(E, rows, seed=2)
    x = synth.activations(n_tok, cols, seed=3)
    y1, a1 = O.moe(O.MXFP4, O.F32, W3, E, rows, cols, ids, None, k, x, n_tok, bias=b)
    y2, a2 = OP.moe(O.MXFP4, O.F32, W3, E, rows, cols, ids, None, k, x, n_tok, bias=b, procs=3)
    assert np.array_equal(y1, y2) and np.array_equal(a1, a2)
    h = synth.activations(n_tok * k, cols, seed=4).reshape(n_tok, k, cols)
    y1, a1 = O.moe(O.MXFP4, O.F32, W3, E, rows, cols, ids, gates, k, h, n_tok, bias=b)
    y2, a2 = OP.moe(O.MXFP4, O.F32, W3, E, rows, cols, ids, gates, k, h, n_tok, bias=b, procs=3)
    assert np.array_equal(y1, y2) and np.array_equal(a1, a2)
