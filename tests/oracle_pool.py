"""The oracle on every host core, for whole-output comparisons at full size.

The C oracle is single-threaded and computes each output on its own, so its
rows (matvec) or tokens (mixture of experts) split into independent pieces.
The inputs go to .npy files that every worker maps read-only; a pool of
processes started with "spawn" (never forked from a process that has used
the GPU) computes the pieces and the parent stacks them.  Nothing here does
arithmetic of its own: each piece is one call of the oracle's matvec or moe.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

_ARR = {}


def _init(paths):
    from oracle import oracle as O
    O.lib()
    _ARR.clear()
    for k, p in paths.items():
        _ARR[k] = np.load(p, mmap_mode="r")


def _matvec_piece(args):
    from oracle import oracle as O
    wt, at, rows, cols, n_vec, r0, r1 = args
    rb = O.row_bytes(wt, cols)
    W = np.ascontiguousarray(_ARR["W"][r0 * rb:r1 * rb])
    y, ya = O.matvec(wt, at, W, r1 - r0, cols, np.asarray(_ARR["x"]), n_vec)
    return r0, y, ya


def _moe_piece(args):
    from oracle import oracle as O
    wt, at, n_expert, rows, cols, k, t0, t1, has_gates, has_bias = args
    gates = np.asarray(_ARR["gates"][t0:t1]) if has_gates else None
    bias = np.asarray(_ARR["bias"]) if has_bias else None
    y, ya = O.moe(wt, at, _ARR["W"], n_expert, rows, cols, np.asarray(_ARR["ids"][t0:t1]), gates, k,
                  np.asarray(_ARR["x"][t0:t1]), t1 - t0, bias=bias)
    return t0, y, ya


def _run(arrays, fn, tasks, procs):
    procs = procs or os.cpu_count() or 1
    with tempfile.TemporaryDirectory(prefix="orc_pool_") as d:
        paths = {}
        for k, a in arrays.items():
            paths[k] = os.path.join(d, k + ".npy")
            np.save(paths[k], np.ascontiguousarray(a))
        ctx = mp.get_context("spawn")
        with ctx.Pool(min(procs, len(tasks)), initializer=_init, initargs=(paths,)) as pool:
            return pool.map_async(fn, tasks, chunksize=1).get(timeout=1800)


def matvec(wt, at, W, rows, cols, x, n_vec, procs=None, pieces_per_proc=4):
    """(y, yabs) float64 [n_vec][rows], as oracle.matvec, rows split over processes."""
    procs = procs or os.cpu_count() or 1
    n = max(1, min(rows, procs * pieces_per_proc))
    bounds = [rows * i // n for i in range(n + 1)]
    tasks = [(wt, at, rows, cols, n_vec, bounds[i], bounds[i + 1]) for i in range(n) if bounds[i + 1] > bounds[i]]
    out = _run({"W": W, "x": x}, _matvec_piece, tasks, procs)
    y = np.empty((n_vec, rows))
    ya = np.empty((n_vec, rows))
    for r0, yp, yap in out:
        y[:, r0:r0 + yp.shape[1]] = yp
        ya[:, r0:r0 + yp.shape[1]] = yap
    return y, ya


def moe(wt, at, W3d, n_expert, rows, cols, ids, gates, k, x, n_tok, bias=None, procs=None):
    """(y, yabs) as oracle.moe, tokens split over processes."""
    procs = procs or os.cpu_count() or 1
    n = max(1, min(n_tok, procs * 2))
    bounds = [n_tok * i // n for i in range(n + 1)]
    arrays = {"W": W3d, "ids": ids, "x": x}
    if gates is not None:
        arrays["gates"] = gates
    if bias is not None:
        arrays["bias"] = bias
    tasks = [(wt, at, n_expert, rows, cols, k, bounds[i], bounds[i + 1], gates is not None, bias is not None)
             for i in range(n) if bounds[i + 1] > bounds[i]]
    out = _run(arrays, _moe_piece, tasks, procs)
    shape = (n_tok, k, rows) if gates is None else (n_tok, rows)
    y = np.empty(shape)
    ya = np.empty(shape)
    for t0, yp, yap in out:
        y[t0:t0 + yp.shape[0]] = yp
        ya[t0:t0 + yp.shape[0]] = yap
    return y, ya
