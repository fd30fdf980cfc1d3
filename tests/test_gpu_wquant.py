"""The weight quantiser (qmv_quantize_weights) against the oracle: bit-exact
blocks for Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K and Q6_K, from fp32 and from
bf16 weights, on adversarial inputs (magnitude ties with
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


Q4_1, Q5_1, Q5_K, Q6_K, BF16 = 11, 12, 16, 5, 9
W32_TYPES = [Q4_0, Q5_0, Q8_0, Q4_1, Q5_1]
WK_TYPES = [Q4_K, Q5_K, Q6_K]


def _check(qmv, orc, t, w_dev, w_ref, rows, cols, fmt=None):
    import torch
    from gpu_util import orc_t
    ref = orc.quantize_weights(orc_t(t), w_ref)
    out = torch.full((rows * qmv.qmv_row_bytes(t, cols),), 0xA5, dtype=torch.uint8, device="cuda")
    qmv.qmv_quantize_weights(t if fmt is None else fmt, w_dev, rows, cols, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert got.size == ref.size and np.array_equal(got, ref), \
        f"t={t}: first differing byte {int(np.flatnonzero(got != ref)[0])}"


@pytest.mark.gpu
@pytest.mark.parametrize("t", W32_TYPES + WK_TYPES)
@pytest.mark.parametrize("shape", [0, 1, 2, 3])
def test_quantize_weights_bit_exact(qmv, orc, t, shape):
    import torch
    rows, cols = ([(1, 32), (37, 96), (300, 896), (64, 4096)] if t in W32_TYPES else
                  [(1, 256), (37, 512), (300, 1024), (64, 4096)])[shape]
    w = weights(rows + cols + t, rows, cols)
    _check(qmv, orc, t, torch.from_numpy(w).cuda(), w, rows, cols)


@pytest.mark.gpu
@pytest.mark.parametrize("t", W32_TYPES + WK_TYPES)
def test_quantize_weights_bf16_input(qmv, orc, t):
    """bf16 weights: the same blocks the oracle writes from their exact fp32 values."""
    import torch
    rows, cols = 45, 1024
    w = torch.from_numpy(weights(77 + t, rows, cols)).to(torch.bfloat16)
    _check(qmv, orc, t, w.cuda(), w.float().numpy(), rows, cols, fmt=qmv.FMT(t, BF16))


@pytest.mark.gpu
@pytest.mark.parametrize("t", [Q4_0, Q4_K, Q6_K])
def test_quantize_weights_full_shape(qmv, orc, t):
    """A 14336 x 4096 projection (58.7 M weights), compared whole."""
    import torch
    rows, cols = 14336, 4096
    w = np.random.default_rng(9).standard_normal((rows, cols), dtype=np.float32) * np.float32(0.02)
    _check(qmv, orc, t, torch.from_numpy(w).cuda(), w, rows, cols)


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
