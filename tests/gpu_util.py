"""Helpers for the GPU parity tests: device copies and the tolerance of the
multiply (per output |y - y_oracle| <= 1e-4 * sum_c |w * xhat|; an output
whose sum of magnitudes is 0 must be exactly 0)."""
import numpy as np
import torch

TOL = 1e-4

# The library's type numbers (include/qmv.h) and the oracle's own table
# (oracle/oracle.h) agree on the original formats; the later ones differ.
_ORC = {11: 10, 12: 11, 13: 15, 14: 13, 15: 14, 16: 12, 17: 16, 18: 17}


def orc_t(t):
    """The oracle's number for library type t."""
    return _ORC.get(t, t)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y, yref, yabs, tol=TOL, what=""):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - yref)
    bound = tol * yabs
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first at {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={yref[tuple(i)]!r} sum|wx|={yabs[tuple(i)]!r}")
    return float((err / np.maximum(yabs, 1e-300)).max()) if err.size else 0.0


class workspace:
    """Register a device workspace of at least `nbytes` for the calls inside
    the block (the mixture of experts, the W4A8 prefill); cleared on exit."""

    def __init__(self, qmv, nbytes):
        self.qmv, self.nbytes = qmv, max(int(nbytes), 256)

    def __enter__(self):
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device="cuda")
        self.qmv.qmv_set_workspace(self.buf, self.buf.numel())
        return self.buf

    def __exit__(self, *exc):
        self.qmv.qmv_set_workspace(None, 0)
