"""qmv_moe_matvec_noalloc: the mixture-of-experts call for callers that
cannot allocate device memory.

A caller that owns all device memory through its own pool, that runs a
latency-critical loop where an allocation may stall the device, or that runs
before its host's allocator exists cannot hand the library a workspace.  This
call keeps its scratch in a fixed array inside the library instead.  The tests
check, through the C ABI, that two calls in a row (different routings, both
forms) give the bits qmv_moe_matvec with a registered workspace gives and
agree with the oracle within the tolerance the other tests use, on both the
8-bit matvec path and the bf16 grouped tensor-core GEMM path (which keeps its
slot list and packed activation rows in the same array); that a call needing
more than the built-in scratch is refused; and that all of this also holds in
a fresh process whose first library call on the device is this one (this
file is collected last, so a run that stops at the first failure has already
run every other test).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu

MXFP4, Q8_0, BF16 = 6, 3, 9
HERE = os.path.dirname(os.path.abspath(__file__))


def _inputs(at, n_tok, k, cols, call, down):
    if down:
        x = synth.activations(n_tok * k, cols, seed=50 + call).reshape(n_tok, k, cols)
    else:
        x = synth.activations(n_tok, cols, seed=50 + call)
    if at == BF16:
        xb = torch.from_numpy(x).to(torch.bfloat16)
        return xb.cuda(), xb.view(torch.int16).numpy()    # device copy, oracle's bf16 bits
    return dev(x), x


@pytest.mark.parametrize("at", [Q8_0, BF16], ids=["Q8_0", "BF16"])
def test_moe_noalloc_matches_workspace_call(qmv, orc, at):
    E, rows, cols, k, n_tok = 8, 256, 512, 4, 6
    W3 = synth.weights(MXFP4, E * rows, cols, seed=31, tensor_id=1)
    W3d = dev(W3)
    b = synth.bias(E, rows, seed=31)
    bd = dev(b)
    fmt = qmv.FMT(MXFP4, at) | (qmv.FLAG_QUANTIZE_X if at == Q8_0 else 0)
    need = qmv.qmv_workspace_size(qmv.OP_MOE, fmt, rows, cols, n_tok * k)
    assert 0 < need <= qmv.MOE_NOALLOC_MAX_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")   # only for the reference call
    try:
        for call, down in enumerate((False, True)):   # two calls in a row, different routings
            ids, gates = synth.router(n_tok, E, k, seed=40 + call)
            shape = (n_tok, rows) if down else (n_tok, k, rows)
            xd, x_host = _inputs(at, n_tok, k, cols, call, down)
            g = dev(gates) if down else None
            y_na = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_moe_matvec_noalloc(fmt, W3d, E, rows, cols, dev(ids), g, k, xd, y_na, n_tok, bd)
            qmv.qmv_set_workspace(ws, ws.numel())
            y_ws = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_moe_matvec(fmt, W3d, E, rows, cols, dev(ids), g, k, xd, y_ws, n_tok, bd)
            qmv.qmv_set_workspace(None, 0)
            qmv.qmv_get_status()
            a, r = host(y_na), host(y_ws)
            # the same kernels on the same inputs: only the scratch differs
            assert np.array_equal(a.view(np.uint32), r.view(np.uint32)), f"call {call}: bits differ"
            x_o = orc.quantize_act(Q8_0, x_host) if at == Q8_0 else x_host
            yref, yabs = orc.moe(MXFP4, at, W3, E, rows, cols, ids, gates if down else None, k, x_o, n_tok, bias=b)
            assert_close(a, yref, yabs, what=f"call {call} against the oracle")
    finally:
        qmv.qmv_set_workspace(None, 0)
    # beyond the built-in scratch: refused on the host, nothing launched
    big_tok = qmv.MOE_NOALLOC_MAX_BYTES // (k * rows * 4) + 1
    y = torch.empty((1,), dtype=torch.float32, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_moe_matvec_noalloc(fmt, W3d, E, rows, cols, y, None, k, y, y, big_tok, None)
    assert e.value.code == qmv.ERR_SHAPE and "built-in scratch" in str(e.value)


def test_moe_noalloc_in_a_fresh_process(qmv):
    """The same checks in a new process, where the no-allocation call is the
    first thing that asks the library for the scratch's device address."""
    if os.environ.get("QMV_NOALLOC_CHILD"):
        pytest.skip("already the child process")
    env = dict(os.environ, QMV_NOALLOC_CHILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_zz_no_alloc.py"), "-k", "matches_workspace_call"],
                       cwd=os.path.dirname(HERE), env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "2 passed" in r.stdout, r.stdout[-2000:]
