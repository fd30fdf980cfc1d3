"""Python face of the CPU oracle (test infrastructure only).

The oracle is plain C in this directory (fp.c, blocks.c, quant.c, wquant.c, mm.c),
compiled with gcc into ``oracle/_build/liboracle.so`` and loaded through
ctypes.  Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this module; the CUDA library never does, and
the two share no code.

Every function below is a thin marshalling wrapper; the arithmetic lives in the
C files, each of which cites the passage of the llamay pages it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = ["fp.c", "blocks.c", "quant.c", "wquant.c", "mm.c", "moeblock.c", "mx.c"]

# The oracle's own type numbers (oracle.h).
Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16, Q4_1, Q5_1, Q5_K, Q2_K, Q3_K, Q8_1, F16, MXFP8 = range(1, 18)
BLOCK_ELEMS = {MXFP8: 32, Q4_0: 32, Q5_0: 32, Q8_0: 32, MXFP4: 32, Q4_K: 256, Q6_K: 256, Q8_K: 256, Q4_1: 32, Q5_1: 32,
               Q5_K: 256, Q2_K: 256, Q3_K: 256, Q8_1: 32, F32: 1, F16: 1, BF16: 1}
BLOCK_BYTES = {MXFP8: 33, Q4_0: 18, Q5_0: 22, Q8_0: 34, MXFP4: 17, Q4_K: 144, Q6_K: 210, Q8_K: 292, Q4_1: 20, Q5_1: 24,
               Q5_K: 176, Q2_K: 84, Q3_K: 110, Q8_1: 36, F32: 4, F16: 2, BF16: 2}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    hdr = os.path.join(HERE, "oracle.h")
    if not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(p) for p in srcs + [hdr])
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp] + srcs + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(LIB_PATH)
            P, I64, I = C.c_void_p, C.c_int64, C.c_int
            L.orc_f16_to_f64.argtypes = [C.c_uint16]
            L.orc_f16_to_f64.restype = C.c_double
            L.orc_f32_to_f16_rn.argtypes = [C.c_float]
            L.orc_f32_to_f16_rn.restype = C.c_uint16
            L.orc_bf16_to_f64.argtypes = [C.c_uint16]
            L.orc_bf16_to_f64.restype = C.c_double
            L.orc_f32_to_bf16_rn.argtypes = [C.c_float]
            L.orc_f32_to_bf16_rn.restype = C.c_uint16
            L.orc_dequant.argtypes = [I, P, I64, I64, P]
            L.orc_quantize_act.argtypes = [I, P, I64, P]
            L.orc_quantize_weights.argtypes = [I, P, I64, P]
            L.orc_block_dots.argtypes = [I, P, I64, I64, P, I64, P]
            L.orc_matvec.argtypes = [I, I, P, I64, I64, P, I64, P, I64, P, P]
            L.orc_moe.argtypes = [I, I, P, I64, I64, I64, P, P, I64, P, I64, P, P, P]
            L.orc_decode_block.argtypes = [I, P, P]
            L.orc_router.argtypes = [P, P, P, I64, I64, I64, P]
            L.orc_router.restype = I
            L.orc_topk_softmax.argtypes = [P, I64, I64, I64, P, P]
            L.orc_topk_softmax.restype = I
            L.orc_swiglu.argtypes = [C.c_double, C.c_double, C.c_double, C.c_double]
            L.orc_swiglu.restype = C.c_double
            L.orc_e4m3_to_f64.argtypes = [C.c_uint8]
            L.orc_e4m3_to_f64.restype = C.c_double
            L.orc_f64_to_e4m3_rn_sat.argtypes = [C.c_double]
            L.orc_f64_to_e4m3_rn_sat.restype = C.c_uint8
            for f in ("orc_dequant", "orc_quantize_act", "orc_quantize_weights", "orc_block_dots", "orc_matvec",
                      "orc_moe", "orc_decode_block"):
                getattr(L, f).restype = I
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


def row_bytes(t: int, cols: int) -> int:
    return cols // BLOCK_ELEMS[t] * BLOCK_BYTES[t]


# ---- scalar conversions -------------------------------------------------------

def f16_to_f64(h: int) -> float:
    return lib().orc_f16_to_f64(int(h))


def f32_to_f16_rn(f: float) -> int:
    return lib().orc_f32_to_f16_rn(float(np.float32(f)))


def bf16_to_f64(b: int) -> float:
    return lib().orc_bf16_to_f64(int(b))


def f32_to_bf16_rn(f: float) -> int:
    return lib().orc_f32_to_bf16_rn(float(np.float32(f)))


# ---- blocks -------------------------------------------------------------------

class _Block(C.Structure):
    _fields_ = [("n", C.c_int), ("code", C.c_int32 * 256), ("sub_scale", C.c_int32 * 256),
                ("sub_min", C.c_int32 * 256), ("d", C.c_double), ("dmin", C.c_double)]


def decode_block(t: int, blk: bytes):
    """-> dict(code, sub_scale, sub_min (int arrays), d, dmin) for one block."""
    b = _Block()
    buf = np.frombuffer(bytes(blk), dtype=np.uint8).copy()
    _check(lib().orc_decode_block(t, _ptr(buf), C.byref(b)), "decode_block")
    n = b.n
    return dict(code=np.array(b.code[:n]), sub_scale=np.array(b.sub_scale[:n]),
                sub_min=np.array(b.sub_min[:n]), d=b.d, dmin=b.dmin)


def dequant(t: int, W: np.ndarray, rows: int, cols: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size >= rows * row_bytes(t, cols)
    out = np.empty((rows, cols), dtype=np.float32)
    _check(lib().orc_dequant(t, _ptr(W), rows, cols, _ptr(out)), "dequant")
    return out


def quantize_act(atype: int, x: np.ndarray) -> np.ndarray:
    """x float32 [..., cols] -> uint8 [..., cols/bs * block_bytes]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bs, bb = BLOCK_ELEMS[atype], BLOCK_BYTES[atype]
    cols = x.shape[-1]
    out = np.empty(x.shape[:-1] + (cols // bs * bb,), dtype=np.uint8)
    _check(lib().orc_quantize_act(atype, _ptr(x), x.size, _ptr(out)), "quantize_act")
    return out


def quantize_weights(wt: int, w: np.ndarray) -> np.ndarray:
    """w float32 [rows, cols] -> Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0 (cols % 32 == 0) or Q4_K / Q5_K / Q6_K
    (cols % 256 == 0) blocks, uint8 [rows * row_bytes]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(w.size // BLOCK_ELEMS[wt] * BLOCK_BYTES[wt], dtype=np.uint8)
    _check(lib().orc_quantize_weights(wt, _ptr(w), w.size, _ptr(out)), "quantize_weights")
    return out


def block_dots(wt: int, W: np.ndarray, rows: int, cols: int, xq: np.ndarray, n_vec: int) -> np.ndarray:
    """-> int64 [n_vec][rows][cols/bs][2] = (S, Mn) per block."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    nb = cols // BLOCK_ELEMS[wt]
    out = np.empty((n_vec, rows, nb, 2), dtype=np.int64)
    _check(lib().orc_block_dots(wt, _ptr(W), rows, cols, _ptr(xq), n_vec, _ptr(out)), "block_dots")
    return out


def matvec(wt: int, at: int, W: np.ndarray, rows: int, cols: int, x: np.ndarray, n_vec: int,
           row_ids=None, want_abs: bool = True):
    """-> (y, yabs) float64 [n_vec][n_rows]; x in the layout of `at` (see oracle.h)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x)
    if row_ids is not None:
        row_ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        n_rows = row_ids.size
    else:
        n_rows = rows
    y = np.empty((n_vec, n_rows), dtype=np.float64)
    ya = np.empty((n_vec, n_rows), dtype=np.float64) if want_abs else None
    _check(lib().orc_matvec(wt, at, _ptr(W), rows, cols, _ptr(x), n_vec, _ptr(row_ids),
                            n_rows, _ptr(y), _ptr(ya)), "matvec")
    return y, ya


def moe(wt: int, at: int, W3d: np.ndarray, n_expert: int, rows: int, cols: int, ids: np.ndarray,
        gates, k: int, x: np.ndarray, n_tok: int, bias=None):
    """-> (y, yabs) float64: [n_tok][k][rows] if gates is None else [n_tok][rows]."""
    W3d = np.ascontiguousarray(W3d, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    x = np.ascontiguousarray(x)
    g = None if gates is None else np.ascontiguousarray(gates, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    shape = (n_tok, k, rows) if gates is None else (n_tok, rows)
    y = np.empty(shape, dtype=np.float64)
    ya = np.empty(shape, dtype=np.float64)
    _check(lib().orc_moe(wt, at, _ptr(W3d), n_expert, rows, cols, _ptr(ids), _ptr(g), k,
                         _ptr(x), n_tok, _ptr(b), _ptr(y), _ptr(ya)), "moe")
    return y, ya


# ---- mixture-of-experts block (moeblock.c, composed with moe()) ------------------------

def router(x: np.ndarray, Wr: np.ndarray, br=None) -> np.ndarray:
    """fp32 logits [n_tok][n_expert] in the order the top-k decision is taken in."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    n_tok, hidden = x.shape
    E = Wr.shape[0]
    b = None if br is None else np.ascontiguousarray(br, dtype=np.float32)
    out = np.empty((n_tok, E), dtype=np.float32)
    _check(lib().orc_router(_ptr(x), _ptr(Wr), _ptr(b), n_tok, hidden, E, _ptr(out)), "router")
    return out


def topk_softmax(logits: np.ndarray, k: int):
    """-> (ids int32 [n_tok][k], gates float64 [n_tok][k])."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    n_tok, E = logits.shape
    ids = np.empty((n_tok, k), dtype=np.int32)
    gates = np.empty((n_tok, k), dtype=np.float64)
    _check(lib().orc_topk_softmax(_ptr(logits), n_tok, E, k, _ptr(ids), _ptr(gates)), "topk_softmax")
    return ids, gates


def swiglu(g, u, alpha: float, limit: float) -> np.ndarray:
    """The clipped, offset SwiGLU of each (g, u) pair, fp64."""
    f = lib().orc_swiglu
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    out = np.empty(np.broadcast(g, u).shape, dtype=np.float64)
    for idx in np.ndindex(out.shape):
        out[idx] = f(float(g[idx]), float(u[idx]), float(alpha), float(limit))
    return out


def moe_block(wt: int, at: int, x: np.ndarray, Wr, br, Wgu, bgu, Wdown, bdown, n_expert: int, k: int,
              hidden: int, inter: int, alpha: float, limit: float, detail: bool = False):
    """A whole expert block for fp32 hidden states x [n_tok][hidden]:
    router -> top k -> gate_up (rows [0, inter) gate, [inter, 2 inter) linear)
    -> clipped SwiGLU -> down, gate-weighted.  at: F32, BF16 or the 8-bit type
    paired with wt (the activations of both projections, quantised or rounded
    from fp32 as the library's block does).  Returns (y, yabs, ids, gates), and
    with detail=True also a dict of the gate_up outputs y1, their sums of
    magnitudes y1abs ([n_tok][k][2 inter], fp64) and the activations h
    ([n_tok][k][inter], fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n_tok = x.shape[0]
    ids, gates = topk_softmax(router(x, Wr, br), k)

    def act(v):   # fp32 values -> the activation layout of `at`
        v = np.ascontiguousarray(v, dtype=np.float32)
        if at == F32:
            return v
        if at == BF16:
            bits = np.vectorize(f32_to_bf16_rn, otypes=[np.uint16])(v)
            return bits.view(np.int16)
        return quantize_act(at, v)
    y1, y1abs = moe(wt, at, Wgu, n_expert, 2 * inter, hidden, ids, None, k, act(x), n_tok, bias=bgu)
    h = swiglu(y1[:, :, :inter], y1[:, :, inter:], alpha, limit).astype(np.float32)   # [n_tok][k][inter]
    y, yabs = moe(wt, at, Wdown, n_expert, hidden, inter, ids, gates.astype(np.float32), k, act(h), n_tok,
                  bias=bdown)
    if detail:
        return y, yabs, ids, gates, dict(y1=y1, y1abs=y1abs, h=h)
    return y, yabs, ids, gates


# ---- MXFP8 activations (mx.c) -----------------------------------------------------------

def e4m3_to_f64(b: int) -> float:
    return lib().orc_e4m3_to_f64(int(b))


def f64_to_e4m3(v: float) -> int:
    """Nearest E4M3 code (ties to even), magnitudes clamped to 448."""
    return lib().orc_f64_to_e4m3_rn_sat(float(v))


def mxfp8_values(blocks: np.ndarray) -> np.ndarray:
    """MXFP8 blocks uint8 [..., nb*33] -> the values they hold, float64 [..., nb*32]."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    lead = b.shape[:-1]
    nb = b.shape[-1] // 33
    b = b.reshape(-1, nb, 33)
    tab = np.array([e4m3_to_f64(i) for i in range(256)])
    v = tab[b[:, :, 1:]] * np.ldexp(1.0, b[:, :, :1].astype(np.int64) - 127)
    return v.reshape(lead + (nb * 32,))
