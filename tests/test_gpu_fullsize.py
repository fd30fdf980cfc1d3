"""Every output of the configurations' full-size products against the oracle.

The sampled-row tests elsewhere reach every code path on small shapes; these
compare whole outputs at the model shapes the bench runs -- the Qwen2.5-0.5B
lm_head (151936 x 896 Q8_0) and layer matrices, the Llama-3-8B K-quant
shapes at 16 vectors, the prefill GEMM at 14336 x 4096 with 512 tokens (Q4_K
with bf16 and W4A8 activations, Q8_0 and Q6_K with bf16), and the gpt-oss-20B experts at 64 tokens on both MoE paths -- so a
fault confined to one tile, K-chunk or expert deep inside a large launch
cannot pass.  The oracle runs on every host core (rows or tokens split over
spawned processes, tests/oracle_pool.py).

Bar: per output |y - y_oracle| <= 1e-4 * sum|w * xhat| (sum over slots with
the gate weights and biases for the mixture of experts)."""
import numpy as np
import pytest
import torch

import oracle_pool as OP
from gguf_block_quantised_gb300 import synth
from gpu_util import assert_close, dev, host, workspace

pytestmark = pytest.mark.gpu

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16 = 1, 2, 3, 4, 5, 6, 7, 8, 9


def _matvec_whole(qmv, orc, t, at, rows, cols, n_vec, seed, quant_in_kernel):
    W = synth.weights(t, rows, cols, seed=seed, tensor_id=rows)
    x = synth.activations(n_vec, cols, seed=seed, tensor_id=cols)
    x_o = orc.quantize_act(at, x) if at != F32 else x
    if at == F32 or quant_in_kernel:
        xin, flags = dev(x), (qmv.FLAG_QUANTIZE_X if at != F32 else 0)
    else:
        xin, flags = dev(x_o), 0
    y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
    qmv.qmv_matvec(qmv.FMT(t, at) | flags, dev(W), rows, cols, xin, y, n_vec)
    qmv.qmv_get_status()
    yref, yabs = OP.matvec(t, at, W, rows, cols, x_o, n_vec)
    return host(y), yref, yabs


@pytest.mark.parametrize("at,n_vec", [(Q8_0, 1), (Q8_0, 8), (F32, 1)], ids=["A8-1", "A8-8", "A32-1"])
def test_lm_head_whole(qmv, orc, at, n_vec):
    """Qwen2.5-0.5B lm_head 151936 x 896 in Q8_0, as the decode step runs it."""
    y, yref, yabs = _matvec_whole(qmv, orc, Q8_0, at, 151936, 896, n_vec, 11, True)
    assert_close(y, yref, yabs, what=f"lm_head at={at} n_vec={n_vec}")


@pytest.mark.parametrize("rows,cols", [(1152, 896), (896, 896), (9728, 896), (896, 4864)])
def test_qwen_layer_whole(qmv, orc, rows, cols):
    """The decode step's stacked Q5_0 layer matrices (q|k|v, o, gate|up, down), batch 1 and 8."""
    for n_vec in (1, 8):
        y, yref, yabs = _matvec_whole(qmv, orc, Q5_0, Q8_0, rows, cols, n_vec, 12, True)
        assert_close(y, yref, yabs, what=f"Q5_0 {rows}x{cols} n_vec={n_vec}")


@pytest.mark.parametrize("t,rows,cols", [(Q4_K, 14336, 4096), (Q4_K, 4096, 14336), (Q6_K, 128256, 4096)],
                         ids=["q4k_14336x4096", "q4k_4096x14336", "q6k_128256x4096"])
def test_kquant_whole_16_vectors(qmv, orc, t, rows, cols):
    """Llama-3-8B K-quant shapes with 16 vectors of Q8_K activations."""
    y, yref, yabs = _matvec_whole(qmv, orc, t, Q8_K, rows, cols, 16, 13, True)
    assert_close(y, yref, yabs, what=f"t={t} {rows}x{cols} n_vec=16")


@pytest.mark.parametrize("t,at", [(Q4_K, BF16), (Q4_K, Q8_K), (Q8_0, BF16), (Q6_K, BF16)],
                         ids=["bf16", "w4a8", "q8_0_bf16", "q6_k_bf16"])
def test_prefill_whole_14336x4096_m512(qmv, orc, t, at):
    """The prefill GEMM on 14336 x 4096 with 512 tokens, every output: Q4_K with
    bf16 and Q8_K activations, and Q8_0 / Q6_K tiles dequantised inside the GEMM."""
    rows, cols, m = 14336, 4096, 512
    W = synth.weights(t, rows, cols, seed=14, tensor_id=1)
    x = synth.activations(m, cols, seed=14)
    if at == BF16:
        xb = torch.from_numpy(x).to(torch.bfloat16)
        X, x_o = xb.cuda(), xb.view(torch.int16).numpy()
    else:
        x_o = orc.quantize_act(Q8_K, x)
        X = dev(x_o)
    Y = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    with workspace(qmv, qmv.qmv_workspace_size(qmv.OP_MATMUL, qmv.FMT(t, at), rows, cols, m)):
        qmv.qmv_matmul(qmv.FMT(t, at), dev(W), rows, cols, X, Y, m)
        qmv.qmv_get_status()
    yref, yabs = OP.matvec(t, at, W, rows, cols, x_o, m)
    assert_close(host(Y), yref, yabs, what=f"prefill t={t} at={at}")


@pytest.mark.parametrize("path", ["w4a8", "bf16", "bf16_repacked"])
def test_gpt_oss_moe_whole_64_tokens(qmv, orc, path):
    """gpt-oss-20B experts (32 MXFP4 experts, gate_up 5760 x 2880 up form, then
    down 2880 x 2880 gate-weighted), top-4 routing, 64 tokens, every output."""
    E, k, n_tok, cols = 32, 4, 64, 2880
    ids, gates = synth.router(n_tok, E, k, seed=15)
    ws_bytes = 0
    for rows, down in ((5760, False), (2880, True)):
        W3 = synth.weights(MXFP4, E * rows, cols, seed=15, tensor_id=rows)
        b = synth.bias(E, rows, seed=15, tensor_id=rows)
        x = synth.activations(n_tok * k if down else n_tok, cols, seed=16, tensor_id=rows)
        if down:
            x = x.reshape(n_tok, k, cols)
        if path == "w4a8":
            fmt, at = qmv.FMT(MXFP4, Q8_0) | qmv.FLAG_QUANTIZE_X, Q8_0
            xin, x_o = dev(x), orc.quantize_act(Q8_0, x)
        else:
            fmt, at = qmv.FMT(MXFP4, BF16), BF16
            xb = torch.from_numpy(x).to(torch.bfloat16)
            xin, x_o = xb.cuda(), xb.view(torch.int16).numpy()
        Wd = dev(W3)
        if path == "bf16_repacked":
            Wr = torch.empty(E * rows * qmv.qmv_row_bytes(qmv.MXFP4_R, cols), dtype=torch.uint8, device="cuda")
            qmv.qmv_repack(MXFP4, Wd, E * rows, cols, Wr)
            Wd, fmt = Wr, qmv.FMT(qmv.MXFP4_R, BF16)
        need = qmv.qmv_workspace_size(qmv.OP_MOE, fmt, rows, cols, n_tok * k)
        ws = torch.empty(max(need, ws_bytes), dtype=torch.uint8, device="cuda")
        qmv.qmv_set_workspace(ws, ws.numel())
        try:
            shape = (n_tok, rows) if down else (n_tok, k, rows)
            y = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            qmv.qmv_moe_matvec(fmt, Wd, E, rows, cols, dev(ids), dev(gates) if down else None, k, xin, y, n_tok,
                               dev(b))
            qmv.qmv_get_status()
        finally:
            qmv.qmv_set_workspace(None, 0)
        yref, yabs = OP.moe(MXFP4, at, W3, E, rows, cols, ids, gates if down else None, k, x_o, n_tok, bias=b)
        assert_close(host(y), yref, yabs, what=f"{path} {'down' if down else 'gate_up'}")
