"""Host-side tests of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/qmv.h declares, and refuses bad arguments
with the documented codes before any CUDA work."""
import os
import re

import pytest

import gguf_block_quantised_gb300 as q
from gguf_block_quantised_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return q.load()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "qmv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qmv_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    syms = header_symbols()
    assert len(syms) >= 15
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(q.EXPORTS)


def test_geometry(lib):
    assert q.qmv_version() == 10000
    expect = {q.Q4_0: (32, 18), q.Q5_0: (32, 22), q.Q8_0: (32, 34), q.MXFP4: (32, 17),
              q.Q4_K: (256, 144), q.Q6_K: (256, 210), q.Q8_K: (256, 292)}
    for t, (bs, bb) in expect.items():
        assert q.qmv_block_elems(t) == bs and q.qmv_block_bytes(t) == bb
    assert q.qmv_row_bytes(q.Q5_0, 896) == 616
    assert q.qmv_row_bytes(q.Q4_K, 14336) == 8064
    assert q.qmv_row_bytes(q.Q4_K, 300) == 0
    assert q.qmv_block_elems(99) == 0


def rc(lib, name, *args):
    return getattr(lib, name)(*args)


def test_refusals(lib):
    F = q.FMT
    # shape: K-quant rows must be multiples of 256 (and the message says what to use)
    assert rc(lib, "qmv_matvec", F(q.Q4_K, q.F32), 4096, 8, 300, 4096, 4096, 1, None) == q.ERR_SHAPE
    assert "256" in q.qmv_last_error()
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), 4096, 8, 40, 4096, 4096, 1, None) == q.ERR_SHAPE
    # unsupported weight type / pairing
    assert rc(lib, "qmv_matvec", F(q.Q8_K, q.F32), 4096, 8, 256, 4096, 4096, 1, None) == q.ERR_UNSUPPORTED
    assert "Q4_0" in q.qmv_last_error()
    assert rc(lib, "qmv_matvec", F(q.Q4_K, q.Q8_0), 4096, 8, 256, 4096, 4096, 1, None) == q.ERR_UNSUPPORTED
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.BF16), 4096, 8, 256, 4096, 4096, 1, None) == q.ERR_UNSUPPORTED
    # null / negative / alignment
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), None, 8, 256, 4096, 4096, 1, None) == q.ERR_INVALID_ARG
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), 4096, -1, 256, 4096, 4096, 1, None) == q.ERR_INVALID_ARG
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), 4096, 8, 256, 4096, 4096, 65, None) == q.ERR_INVALID_ARG
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), 4104, 8, 256, 4096, 4096, 1, None) == q.ERR_ALIGN
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), 4096, 8, 256, 4100, 4096, 1, None) == q.ERR_ALIGN
    # empty work is a no-op, even without pointers
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.F32), None, 0, 256, None, None, 1, None) == q.OK
    assert rc(lib, "qmv_matvec", F(q.Q4_0, q.Q8_0), 4096, 8, 256, None, None, 0, None) == q.OK
    # quantiser
    assert rc(lib, "qmv_quantize_act", q.Q4_0, 4096, 4096, 32, None) == q.ERR_UNSUPPORTED
    assert rc(lib, "qmv_quantize_act", q.Q8_K, 4096, 4096, 32, None) == q.ERR_SHAPE
    assert rc(lib, "qmv_quantize_act", q.Q8_0, 4096, 4096, 0, None) == q.OK
    assert rc(lib, "qmv_quantize_act", q.Q8_0, None, 4096, 32, None) == q.ERR_INVALID_ARG
    # weight quantiser
    assert rc(lib, "qmv_quantize_weights", q.Q2_K, 4096, 2, 256, 8192, None) == q.ERR_UNSUPPORTED   # not written
    assert "Q4_0" in q.qmv_last_error() and "Q6_K" in q.qmv_last_error()
    assert rc(lib, "qmv_quantize_weights", q.Q8_K, 4096, 2, 256, 8192, None) == q.ERR_UNSUPPORTED   # activations only
    assert rc(lib, "qmv_quantize_weights", q.FMT(q.Q4_0, q.Q8_0), 4096, 2, 64, 8192, None) == q.ERR_UNSUPPORTED
    assert rc(lib, "qmv_quantize_weights", q.Q4_K, 4096, 2, 96, 8192, None) == q.ERR_SHAPE   # K-quant rows of 256
    assert "256" in q.qmv_last_error()
    assert rc(lib, "qmv_quantize_weights", q.Q4_0, 4096, 2, 48, 8192, None) == q.ERR_SHAPE
    assert rc(lib, "qmv_quantize_weights", q.Q5_0, 4100, 2, 64, 8192, None) == q.ERR_ALIGN
    assert rc(lib, "qmv_quantize_weights", q.Q8_0, 4096, 2, 64, 8193, None) == q.ERR_ALIGN
    assert rc(lib, "qmv_quantize_weights", q.Q4_0, 4096, 2, 64, 4160, None) == q.ERR_INVALID_ARG   # overlaps W
    assert rc(lib, "qmv_quantize_weights", q.Q4_0, None, 0, 64, None, None) == q.OK
    # verification calls
    assert rc(lib, "qmv_dequantize", q.Q6_K, 4096, 2, 200, 4096, None) == q.ERR_SHAPE
    assert rc(lib, "qmv_block_dots", q.Q8_0, 4096, 2, 64, 4096, -1, 4096, None) == q.ERR_INVALID_ARG
    # workspace alignment
    assert rc(lib, "qmv_set_workspace", 4100, 1024) == q.ERR_ALIGN


def test_moe_block_refusals(lib):
    F = q.FMT
    A = 4096   # any 16-byte aligned stand-in address: nothing is dereferenced before the checks

    def call(fmt, E=8, k=2, hidden=256, inter=256, n_tok=3, x=A):
        return rc(lib, "qmv_moe_block", fmt, E, k, hidden, inter, A, None, A, None, A, None, 1.702, 7.0, x, n_tok,
                  A, A, A, None)
    assert call(F(q.Q4_0, q.BF16)) == q.ERR_UNSUPPORTED            # BF16 is for MXFP4 experts only
    assert call(F(q.MXFP4_R, q.F32)) == q.ERR_UNSUPPORTED
    assert call(F(q.Q4_K, q.Q8_0)) == q.ERR_UNSUPPORTED            # K-quants pair with Q8_K
    assert call(F(q.Q8_K, q.F32)) == q.ERR_UNSUPPORTED
    assert call(F(q.Q4_0, q.Q8_0) | q.FLAG_QUANTIZE_X) == q.ERR_INVALID_ARG
    assert call(F(q.Q4_0, q.F32), E=4, k=5) == q.ERR_INVALID_ARG   # k > n_expert
    assert call(F(q.Q4_0, q.F32), E=1025, k=2) == q.ERR_INVALID_ARG
    assert call(F(q.Q4_0, q.F32), inter=40) == q.ERR_SHAPE
    assert call(F(q.Q4_K, q.F32), hidden=288) == q.ERR_SHAPE
    assert call(F(q.Q4_0, q.F32), x=4100) == q.ERR_ALIGN
    assert call(F(q.Q4_0, q.F32), n_tok=0, x=None) == q.OK
    assert call(F(q.Q4_0, q.F32)) == q.ERR_WORKSPACE               # none registered
    assert "qmv_moe_block_workspace_size" in q.qmv_last_error()
    ws = q.qmv_moe_block_workspace_size(F(q.Q4_0, q.F32), 32, 4, 2880, 2880, 1)
    assert ws >= (32 + 3 * 4 * 2880) * 4
    assert q.qmv_moe_block_workspace_size(F(q.Q4_0, q.F32), 32, 4, 2880, 2880, 0) == 0
    assert (q.qmv_moe_block_workspace_size(F(q.MXFP4, q.BF16), 32, 4, 2880, 2880, 8) >
            q.qmv_moe_block_workspace_size(F(q.MXFP4, q.F32), 32, 4, 2880, 2880, 8))


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert q.qmv_strerror(code)
    assert q.qmv_strerror(-99) == "unknown error"


def test_binding_raises_with_message(lib):
    with pytest.raises(q.QmvError) as e:
        q.qmv_matvec(q.FMT(q.Q4_K, q.F32), 4096, 8, 300, 4096, 4096, 1, stream=0)
    assert e.value.code == q.ERR_SHAPE and "multiple of 256" in str(e.value)


def test_matmul_workspace_follows_the_prefill_route(lib):
    """qmv_workspace_size(QMV_OP_MATMUL, ...) names the route qmv_matmul takes:
    none for Q4_K, for BF16 rows, and for Q4_0 / Q5_0 / Q8_0 / Q6_K rows that
    are a whole number of 16 bytes (tiles dequantised inside the GEMM); the bf16
    weight tiles (rows x cols x 2 bytes) for every other type and row length;
    the W4A8 form's codes, sums and scales for Q4_K x Q8_K."""
    F = q.FMT
    rows = 1000
    for t, cols in [(q.Q4_0, 4096), (q.Q5_0, 4096), (q.Q8_0, 4096), (q.Q6_K, 2048), (q.Q6_K, 14336),
                    (q.Q4_K, 4096), (q.BF16, 896), (q.BF16, 4096)]:
        assert q.qmv_workspace_size(q.OP_MATMUL, F(t, q.BF16), rows, cols, 512) == 0, (t, cols)
    # rows not a whole number of 16 bytes: 896 columns of Q4_0 / Q5_0 / Q8_0 (504 / 616 / 952
    # bytes), one Q6_K super-block (210 bytes)
    two_pass = [(q.Q4_0, 896), (q.Q5_0, 896), (q.Q8_0, 896), (q.Q6_K, 256)]
    two_pass += [(t, 4096) for t in (q.Q4_1, q.Q5_1, q.Q8_1, q.MXFP4, q.Q2_K, q.Q3_K, q.Q5_K, q.F32, q.F16)]
    for t, cols in two_pass:
        need = q.qmv_workspace_size(q.OP_MATMUL, F(t, q.BF16), rows, cols, 512)
        assert need >= rows * cols * 2 and need < rows * cols * 2 + 256, (t, cols, need)
    w4a8 = q.qmv_workspace_size(q.OP_MATMUL, F(q.Q4_K, q.Q8_K), rows, 4096, 512)
    assert w4a8 >= 512 * 4096 * 2    # the activation codes as fp16, at least
    assert q.qmv_workspace_size(q.OP_MATMUL, F(q.Q4_K, q.BF16), rows, 4096, 0) == 0
