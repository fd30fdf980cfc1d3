"""The bounded-wait failure path, on the GPU, without a fault.

Every mbarrier wait in the library's kernels gives up after a time limit, sets
the wait-timeout bit of the device status word and lets the kernel stop early
after its own copies in flight have landed.  qmv_set_wait_limit shortens that
limit (diagnostics): with a limit of a few nanoseconds the first wait that has
to wait at all gives up.  The tests check that the host reads the fault through
qmv_get_status, and that the context stays usable: the same call, with the
default limit restored, gives the oracle's results.  Only the decode matvec and
the expert matvec run while the short limit is set."""
import numpy as np
import pytest
import torch

from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host, workspace

pytestmark = pytest.mark.gpu

Q4_0, Q8_0, MXFP4, F32 = 1, 3, 6, 8


def _timed_out(qmv):
    with pytest.raises(qmv.QmvError) as e:
        qmv.qmv_get_status()
    assert e.value.code == qmv.ERR_DEVICE_STATUS
    assert "wait gave up" in str(e.value)


def test_matvec_wait_timeout_is_reported_and_recovers(qmv, orc):
    rows, cols = 14336, 4096          # a 33 MB stream: the consumers must wait for their copies
    W = synth.weights(Q4_0, rows, cols, seed=31)
    x = synth.activations(1, cols, seed=32)
    Wd, xd = dev(W), dev(x)
    fmt = qmv.FMT(Q4_0, Q8_0) | qmv.FLAG_QUANTIZE_X
    y = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qmv.qmv_get_status()
    qmv.qmv_set_wait_limit(4)
    try:
        qmv.qmv_matvec(fmt, Wd, rows, cols, xd, y, 1)
        torch.cuda.synchronize()
    finally:
        qmv.qmv_set_wait_limit(0)
    _timed_out(qmv)
    # the default limit again: the same call completes and matches the oracle
    y.fill_(float("nan"))
    qmv.qmv_matvec(fmt, Wd, rows, cols, xd, y, 1)
    qmv.qmv_get_status()
    got = host(y)
    rids = np.arange(0, rows, 97)
    yref, yabs = orc.matvec(Q4_0, Q8_0, W, rows, cols, orc.quantize_act(Q8_0, x), 1, row_ids=rids)
    assert_close(got[:, rids], yref, yabs, what="after the timeout")
    assert not np.isnan(got).any()


def test_moe_wait_timeout_is_reported_and_recovers(qmv, orc):
    E, rows, cols, k, n_tok = 8, 2880, 2880, 4, 3
    W3 = synth.weights(MXFP4, E * rows, cols, seed=33, tensor_id=1)
    ids, gates = synth.router(n_tok, E, k, seed=34)
    x = synth.activations(n_tok, cols, seed=35)
    W3d, xd, idd = dev(W3), dev(x), dev(ids)
    fmt = qmv.FMT(MXFP4, Q8_0) | qmv.FLAG_QUANTIZE_X
    y = torch.full((n_tok, k, rows), float("nan"), dtype=torch.float32, device="cuda")
    with workspace(qmv, qmv.qmv_workspace_size(qmv.OP_MOE, fmt, rows, cols, n_tok * k)):
        qmv.qmv_get_status()
        qmv.qmv_set_wait_limit(4)
        try:
            qmv.qmv_moe_matvec(fmt, W3d, E, rows, cols, idd, None, k, xd, y, n_tok)
            torch.cuda.synchronize()
        finally:
            qmv.qmv_set_wait_limit(0)
        _timed_out(qmv)
        y.fill_(float("nan"))
        qmv.qmv_moe_matvec(fmt, W3d, E, rows, cols, idd, None, k, xd, y, n_tok)
        qmv.qmv_get_status()
        got = host(y)
    yref, yabs = orc.moe(MXFP4, Q8_0, W3, E, rows, cols, ids, None, k, orc.quantize_act(Q8_0, x), n_tok)
    assert_close(got, yref, yabs, what="after the timeout")
