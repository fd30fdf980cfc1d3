"""gguf_block_quantised_gb300 -- GB300 (sm_103a) block-quantised matrix multiply.

A thin ctypes binding over ``libqmv.so`` (the C ABI in ``include/qmv.h``).
Functions keep the C names; arguments may be torch tensors (their
``data_ptr()`` is passed) or integer device addresses.  ``stream`` may be a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None for torch's
current stream.  Every computation runs in the library's CUDA kernels; there
is no CPU path.  If the library has not been built, :func:`load` raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libqmv.so")

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16, MXFP4_R = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
Q4_1, Q5_1, Q8_1, Q2_K, Q3_K, Q5_K, F16, MXFP8 = 11, 12, 13, 14, 15, 16, 17, 18
NAMES = {Q4_0: "Q4_0", Q5_0: "Q5_0", Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", MXFP4: "MXFP4",
         Q8_K: "Q8_K", F32: "F32", BF16: "BF16", MXFP4_R: "MXFP4_R", Q4_1: "Q4_1", Q5_1: "Q5_1",
         Q8_1: "Q8_1", Q2_K: "Q2_K", Q3_K: "Q3_K", Q5_K: "Q5_K", F16: "F16", MXFP8: "MXFP8"}
OP_MATVEC, OP_MATMUL, OP_MOE = 1, 2, 3
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_STATUS = \
    0, -1, -2, -3, -4, -5, -6, -7


FLAG_QUANTIZE_X = 1 << 16
FLAG_PDL = 1 << 17


def FMT(wtype: int, atype: int) -> int:
    return int(wtype) | (int(atype) << 8)


class QmvError(RuntimeError):
    def __init__(self, code: int, func: str, msg: str):
        super().__init__(f"{func} failed ({code}): {msg}")
        self.code = code


_lib = None
_lock = threading.Lock()

# name -> (restype, argtypes)
_P, _I, _I64, _SZ = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
_SIGS = {
    "qmv_version": (_I, []),
    "qmv_strerror": (C.c_char_p, [_I]),
    "qmv_last_error": (C.c_char_p, []),
    "qmv_block_elems": (_I, [_I]),
    "qmv_block_bytes": (_SZ, [_I]),
    "qmv_row_bytes": (_SZ, [_I, _I64]),
    "qmv_quantize_act": (_I, [_I, _P, _P, _I64, _P]),
    "qmv_quantize_weights": (_I, [_I, _P, _I64, _I64, _P, _P]),
    "qmv_repack": (_I, [_I, _P, _I64, _I64, _P, _P]),
    "qmv_dequantize": (_I, [_I, _P, _I64, _I64, _P, _P]),
    "qmv_block_dots": (_I, [_I, _P, _I64, _I64, _P, _I, _P, _P]),
    "qmv_matvec": (_I, [_I, _P, _I64, _I64, _P, _P, _I, _P]),
    "qmv_matmul": (_I, [_I, _P, _I64, _I64, _P, _P, _I64, _P]),
    "qmv_moe_matvec": (_I, [_I, _P, _I, _I64, _I64, _P, _P, _I, _P, _P, _I64, _P, _P]),
    "qmv_moe_matvec_noalloc": (_I, [_I, _P, _I, _I64, _I64, _P, _P, _I, _P, _P, _I64, _P, _P]),
    "qmv_moe_block": (_I, [_I, _I, _I, _I64, _I64, _P, _P, _P, _P, _P, _P, C.c_float, C.c_float, _P, _I64, _P,
                           _P, _P, _P]),
    "qmv_moe_block_workspace_size": (_SZ, [_I, _I, _I, _I64, _I64, _I64]),
    "qmv_set_wait_limit": (_I, [C.c_uint]),
    "qmv_workspace_size": (_SZ, [_I, _I, _I64, _I64, _I64]),
    "qmv_set_workspace": (_I, [_P, _SZ]),
    "qmv_get_status": (_I, [_P]),
}
EXPORTS = tuple(_SIGS)


def load(path: str | None = None):
    """Load libqmv.so (built by ``gguf_block_quantised_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libqmv.so is not built ({p} missing): run gguf_block_quantised_gb300.build.build()")
            L = C.CDLL(p)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    if rc != 0:
        raise QmvError(rc, name, load().qmv_last_error().decode())
    return rc


# ---- the C ABI, one wrapper per entry point ----------------------------------------

def qmv_version() -> int:
    return load().qmv_version()


def qmv_strerror(err: int) -> str:
    return load().qmv_strerror(err).decode()


def qmv_last_error() -> str:
    return load().qmv_last_error().decode()


def qmv_block_elems(t: int) -> int:
    return load().qmv_block_elems(t)


def qmv_block_bytes(t: int) -> int:
    return load().qmv_block_bytes(t)


def qmv_row_bytes(t: int, cols: int) -> int:
    return load().qmv_row_bytes(t, cols)


def qmv_quantize_act(fmt, x, xq, n, stream=None):
    return _call("qmv_quantize_act", fmt, _ptr(x), _ptr(xq), n, _stream(stream))


def qmv_quantize_weights(t, W, rows, cols, out, stream=None):
    return _call("qmv_quantize_weights", t, _ptr(W), rows, cols, _ptr(out), _stream(stream))


def qmv_repack(t, W, rows, cols, Wout, stream=None):
    return _call("qmv_repack", t, _ptr(W), rows, cols, _ptr(Wout), _stream(stream))


def qmv_dequantize(t, W, rows, cols, out, stream=None):
    return _call("qmv_dequantize", t, _ptr(W), rows, cols, _ptr(out), _stream(stream))


def qmv_block_dots(t, W, rows, cols, xq, n_vec, out, stream=None):
    return _call("qmv_block_dots", t, _ptr(W), rows, cols, _ptr(xq), n_vec, _ptr(out), _stream(stream))


def qmv_matvec(fmt, W, rows, cols, x, y, n_vec, stream=None):
    return _call("qmv_matvec", fmt, _ptr(W), rows, cols, _ptr(x), _ptr(y), n_vec, _stream(stream))


def qmv_matmul(fmt, W, rows, cols, X, Y, m, stream=None):
    return _call("qmv_matmul", fmt, _ptr(W), rows, cols, _ptr(X), _ptr(Y), m, _stream(stream))


def qmv_moe_matvec(fmt, W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias=None, stream=None):
    return _call("qmv_moe_matvec", fmt, _ptr(W3d), n_expert, rows, cols, _ptr(ids), _ptr(gates), k,
                 _ptr(x), _ptr(y), n_tok, _ptr(bias), _stream(stream))


def qmv_moe_matvec_noalloc(fmt, W3d, n_expert, rows, cols, ids, gates, k, x, y, n_tok, bias=None, stream=None):
    """qmv_moe_matvec with the library's built-in scratch (no workspace)."""
    return _call("qmv_moe_matvec_noalloc", fmt, _ptr(W3d), n_expert, rows, cols, _ptr(ids), _ptr(gates), k,
                 _ptr(x), _ptr(y), n_tok, _ptr(bias), _stream(stream))


MOE_NOALLOC_MAX_BYTES = 4 << 20


def qmv_moe_block(fmt, n_expert, k, hidden, inter, Wr, br, W_gu, b_gu, W_down, b_down, alpha, limit, x, n_tok,
                  y, ids, gates, stream=None):
    """Router -> top k -> gate_up -> clipped SwiGLU -> down for fp32 x [n_tok][hidden]."""
    return _call("qmv_moe_block", fmt, n_expert, k, hidden, inter, _ptr(Wr), _ptr(br), _ptr(W_gu), _ptr(b_gu),
                 _ptr(W_down), _ptr(b_down), float(alpha), float(limit), _ptr(x), n_tok, _ptr(y), _ptr(ids),
                 _ptr(gates), _stream(stream))


def qmv_moe_block_workspace_size(fmt, n_expert, k, hidden, inter, n_tok) -> int:
    return load().qmv_moe_block_workspace_size(fmt, n_expert, k, hidden, inter, n_tok)


def qmv_workspace_size(op, fmt, rows, cols, n) -> int:
    return load().qmv_workspace_size(op, fmt, rows, cols, n)


def qmv_set_workspace(ptr, nbytes, stream=None):
    return _call("qmv_set_workspace", _ptr(ptr), nbytes)


def qmv_set_wait_limit(ns):
    """Diagnostics: the limit of every bounded wait in nanoseconds (0: the default)."""
    return _call("qmv_set_wait_limit", int(ns))


def qmv_get_status(stream=None):
    return _call("qmv_get_status", _stream(stream))


# ---- small conveniences over the same calls (allocation stays with torch) -----------

def act_row_bytes(atype: int, cols: int) -> int:
    if atype == F32:
        return 4 * cols
    if atype == BF16:
        return 2 * cols
    return qmv_row_bytes(atype, cols)
