"""qmv_moe_matvec_noalloc: the mixture-of-experts call for callers that
cannot allocate device memory.

A caller that owns all device memory through its own pool, that runs a
latency-critical loop where an allocation may stall the device, or that runs
before its host's allocator exists cannot hand the library a workspace.  This
call keeps its scratch in a fixed array inside the library instead.  The test
checks, through the C ABI, that two calls in a row (different routings, both
forms) give what qmv_moe_matvec with a registered workspace gives, within the
tolerance the other tests use, and that a call needing more than the built-in
scratch is refused.  It runs alone in a fresh process as well as after the
other tests (this file is collected last).
"""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu

MXFP4, Q8_0 = 6, 3


def test_moe_noalloc_matches_workspace_call(qmv, orc):
    E, rows, cols, k, n_tok = 8, 256, 512, 4, 6
    W3 = synth.weights(MXFP4, E * rows, cols, seed=31, tensor_id=1)
    W3d = dev(W3)
    b = synth.bias(E, rows, seed=31)
    bd = dev(b)
    fmt = qmv.FMT(MXFP4, Q8_0) | qmv.FLAG_QUANTIZE_X
    need = qmv.qmv_workspace_size(qmv.OP_MOE, fmt, rows, cols, n_tok * k)
    assert 0 < need <= qmv.MOE_NOALLOC_MAX_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")   # only for the reference call
    try:
        for call, down in enumerate((False, True)):   # two calls in a row, different routings
            ids, gates = synth.router(n_tok, E, k, seed=40 + call)
            if down:
                x = synth.activations(n_tok * k, cols, seed=50 + call).reshape(n_tok, k, cols)
                shape = (n_tok, rows)
            else:
                x = synth.activations(n_tok, cols, seed=50 + call)
                shape = (n_tok, k, rows)
            g = dev(gates) if down else None
            y_na = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_moe_matvec_noalloc(fmt, W3d, E, rows, cols, dev(ids), g, k, dev(x), y_na, n_tok, bd)
            qmv.qmv_set_workspace(ws, ws.numel())
            y_ws = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_moe_matvec(fmt, W3d, E, rows, cols, dev(ids), g, k, dev(x), y_ws, n_tok, bd)
            qmv.qmv_set_workspace(None, 0)
            qmv.qmv_get_status()
            _, yabs = orc.moe(MXFP4, Q8_0, W3, E, rows, cols, ids, gates if down else None, k,
                              orc.quantize_act(Q8_0, x), n_tok, bias=b)
            assert_close(host(y_na), host(y_ws).astype(np.float64), yabs, what=f"call {call}")
    finally:
        qmv.qmv_set_workspace(None, 0)
    # beyond the built-in scratch: refused on the host, nothing launched
    big_tok = qmv.MOE_NOALLOC_MAX_BYTES // (k * rows * 4) + 1
    y = torch.empty((1,), dtype=torch.float32, device="cuda")
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_moe_matvec_noalloc(fmt, W3d, E, rows, cols, y, None, k, y, y, big_tok, None)
    assert e.value.code == qmv.ERR_SHAPE and "built-in scratch" in str(e.value)
