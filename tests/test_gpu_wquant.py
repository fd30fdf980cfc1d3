"""The weight quantiser (qmv_quantize_weights) against the oracle: bit-exact
blocks for Q4_0, Q5_0 and Q8_0 on adversarial inputs (magnitude ties with
opposite signs, zero and negative-zero blocks, scales over 2^-30..2^20, ragged
shapes, blocks so small that 1/d overflows) and at a full model shape;
refusals on the host."""
import numpy as np
import pytest

Q4_0, Q5_0, Q8_0, Q4_K = 1, 2, 3, 4


def weights(seed, rows, cols):
    g = np.random.default_rng(seed)
    w = g.standard_normal((rows, cols)).astype(np.float32)
    nb = rows * cols // 32
    b = w.reshape(nb, 32)
    b *= np.exp2(g.integers(-30, 20, (nb, 1))).astype(np.float32)
    b[::5] = g.uniform(-1, 1, (len(b[::5]), 32)).astype(np.float32)
    b[::7, 3] = -b[::7, 20]                 # equal magnitudes, opposite signs
    b[::13] = 0.0
    b[6::17] = -0.0
    b[::19, :8] = np.float32(2.0 ** -140)   # subnormal neighbours
    b[4::23] = g.uniform(-1, 1, (len(b[4::23]), 32)).astype(np.float32) * np.float32(2.0 ** -127)
    b[4::23, 2] = 0.0                       # a zero in a block whose 1/d overflows
    return w


@pytest.mark.gpu
@pytest.mark.parametrize("t", [Q4_0, Q5_0, Q8_0])
@pytest.mark.parametrize("rows,cols", [(1, 32), (37, 96), (300, 896), (64, 4096)])
def test_quantize_weights_bit_exact(qmv, orc, t, rows, cols):
    import torch
    w = weights(rows + cols + t, rows, cols)
    ref = orc.quantize_weights(t, w)
    out = torch.full((rows * qmv.qmv_row_bytes(t, cols),), 0xA5, dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_weights(t, torch.from_numpy(w).cuda(), rows, cols, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert got.size == ref.size and np.array_equal(got, ref), \
        f"first differing byte {int(np.flatnonzero(got != ref)[0])}"


@pytest.mark.gpu
def test_quantize_weights_full_shape(qmv, orc):
    """A 14336 x 4096 projection (58.7 M weights) to Q4_0, compared whole."""
    import torch
    rows, cols = 14336, 4096
    w = np.random.default_rng(9).standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02)
    out = torch.empty(rows * qmv.qmv_row_bytes(Q4_0, cols), dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_weights(Q4_0, torch.from_numpy(w).cuda(), rows, cols, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), orc.quantize_weights(Q4_0, w))


@pytest.mark.gpu
def test_quantized_weights_feed_the_matvec(qmv, orc):
    """Weights written by the quantiser are read by the decode matvec as GGUF blocks."""
    import torch
    rows, cols = 300, 896
    # trained-weight magnitudes (the adversarial matrix overflows fp16 scales)
    w = np.random.default_rng(3).standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02)
    wq = torch.empty(rows * qmv.qmv_row_bytes(Q5_0, cols), dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_weights(Q5_0, torch.from_numpy(w).cuda(), rows, cols, wq)
    x = np.random.default_rng(4).standard_normal((2, cols), dtype=np.float32)
    y = torch.empty((2, rows), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(Q5_0, 8), wq, rows, cols, torch.from_numpy(x).cuda(), y, 2)
    torch.cuda.synchronize()
    yref, yabs = orc.matvec(Q5_0, 8, orc.quantize_weights(Q5_0, w), rows, cols, x, 2)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - yref) <= 1e-4 * yabs)
