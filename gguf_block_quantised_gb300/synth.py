"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and lays them into the byte fields of
the block formats; it holds none of the multiply's arithmetic (no unpacking,
no scaling, no dot products, no quantisation of activations).

Distributions (model-shaped synthetic weights; no trained weights are used):
  fp16 scale fields d, dmin : fp16(|N(0,1)| * 0.02)
  nibble / code bytes       : uniform over all byte values
  Q5_0 high-bit mask        : uniform u32
  Q8_0 codes                : uniform int8 in [-127, 127]
  Q4_K 12-byte scale field  : uniform bytes
  Q6_K int8 sub-block scales: uniform int8 in [-128, 127]
  Q4_1/Q5_1 offsets m      : fp16(N(0,1) * 0.1)
  K-quant scale/mask fields: uniform bytes (Q2_K, Q3_K, Q5_K)
  plain F32/F16/BF16       : N(0,1) * 0.05 (F16 rounded, BF16 its upper 16 bits)
  MXFP4 E8M0 exponent       : uniform in [118, 130]
  activations               : fp32 N(0,1)
  expert biases             : fp32 N(0,1) * 0.02
  router weights            : fp32 N(0,1) * 0.05 [n_expert][hidden]
  router logits             : N(0,1); top-k by logit (ties to the lower
                              expert id), gates = softmax over the k kept.
Every tensor draws from its own stream, seeded by (seed, tensor_id).
"""
from __future__ import annotations

import numpy as np

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16 = 1, 2, 3, 4, 5, 6, 7, 8, 9
Q4_1, Q5_1, Q8_1, Q2_K, Q3_K, Q5_K, F16 = 11, 12, 13, 14, 15, 16, 17
BLOCK_ELEMS = {Q4_0: 32, Q5_0: 32, Q8_0: 32, MXFP4: 32, Q4_K: 256, Q6_K: 256, Q8_K: 256,
               Q4_1: 32, Q5_1: 32, Q8_1: 32, Q2_K: 256, Q3_K: 256, Q5_K: 256, F32: 1, F16: 1, BF16: 1}
BLOCK_BYTES = {Q4_0: 18, Q5_0: 22, Q8_0: 34, MXFP4: 17, Q4_K: 144, Q6_K: 210, Q8_K: 292,
               Q4_1: 20, Q5_1: 24, Q8_1: 36, Q2_K: 84, Q3_K: 110, Q5_K: 176, F32: 4, F16: 2, BF16: 2}
NAMES = {Q4_0: "Q4_0", Q5_0: "Q5_0", Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K",
         MXFP4: "MXFP4", Q8_K: "Q8_K", F32: "F32", BF16: "BF16", Q4_1: "Q4_1", Q5_1: "Q5_1",
         Q8_1: "Q8_1", Q2_K: "Q2_K", Q3_K: "Q3_K", Q5_K: "Q5_K", F16: "F16"}

# Field layouts of one block, in storage order (little-endian).
_LAYOUT = {
    Q4_0: [("d", "<f2", ()), ("qs", "u1", (16,))],
    Q5_0: [("d", "<f2", ()), ("qh", "<u4", ()), ("qs", "u1", (16,))],
    Q8_0: [("d", "<f2", ()), ("qs", "i1", (32,))],
    MXFP4: [("e", "u1", ()), ("qs", "u1", (16,))],
    Q4_K: [("d", "<f2", ()), ("dmin", "<f2", ()), ("scales", "u1", (12,)), ("qs", "u1", (128,))],
    Q6_K: [("ql", "u1", (128,)), ("qh", "u1", (64,)), ("scales", "i1", (16,)), ("d", "<f2", ())],
    Q4_1: [("d", "<f2", ()), ("m", "<f2", ()), ("qs", "u1", (16,))],
    Q5_1: [("d", "<f2", ()), ("m", "<f2", ()), ("qh", "<u4", ()), ("qs", "u1", (16,))],
    Q8_1: [("d", "<f2", ()), ("s", "<f2", ()), ("qs", "i1", (32,))],
    Q5_K: [("d", "<f2", ()), ("dmin", "<f2", ()), ("scales", "u1", (12,)), ("qh", "u1", (32,)), ("qs", "u1", (128,))],
    Q2_K: [("scales", "u1", (16,)), ("qs", "u1", (64,)), ("d", "<f2", ()), ("dmin", "<f2", ())],
    Q3_K: [("hmask", "u1", (32,)), ("qs", "u1", (64,)), ("scales", "u1", (12,)), ("d", "<f2", ())],
}


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tensor_id)])))


def row_bytes(t: int, cols: int) -> int:
    return cols // BLOCK_ELEMS[t] * BLOCK_BYTES[t]


def block_dtype(t: int) -> np.dtype:
    dt = np.dtype(_LAYOUT[t])
    assert dt.itemsize == BLOCK_BYTES[t]
    return dt


def _fp16_scales(g: np.random.Generator, n: int) -> np.ndarray:
    return (np.abs(g.standard_normal(n, dtype=np.float32)) * np.float32(0.02)).astype(np.float16)


def weights(t: int, rows: int, cols: int, seed: int = 0, tensor_id: int = 0) -> np.ndarray:
    """rows x cols weights of block type t as a flat uint8 array (GGUF row-major blocks;
    plain F32/F16/BF16: N(0,1)*0.05 rounded to the type, row-major values)."""
    if t in (F32, F16, BF16):
        w = rng(seed, tensor_id).standard_normal((rows, cols), dtype=np.float32) * np.float32(0.05)
        if t == F32:
            return w.view(np.uint8).reshape(-1)
        if t == F16:
            return w.astype(np.float16).view(np.uint8).reshape(-1)
        # bfloat16 values: the upper 16 bits of the fp32 draws
        return (w.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8).reshape(-1)
    assert cols % BLOCK_ELEMS[t] == 0
    nblk = rows * (cols // BLOCK_ELEMS[t])
    g = rng(seed, tensor_id)
    a = np.empty(nblk, dtype=block_dtype(t))
    if t in (Q4_0, Q5_0, Q8_0, Q4_K):
        a["d"] = _fp16_scales(g, nblk)
    if t == Q4_K:
        a["dmin"] = _fp16_scales(g, nblk)
        a["scales"] = g.integers(0, 256, size=(nblk, 12), dtype=np.uint8)
        a["qs"] = g.integers(0, 256, size=(nblk, 128), dtype=np.uint8)
    elif t == Q4_0:
        a["qs"] = g.integers(0, 256, size=(nblk, 16), dtype=np.uint8)
    elif t == Q5_0:
        a["qh"] = g.integers(0, 2**32, size=nblk, dtype=np.uint32)
        a["qs"] = g.integers(0, 256, size=(nblk, 16), dtype=np.uint8)
    elif t == Q8_0:
        a["qs"] = g.integers(-127, 128, size=(nblk, 32), dtype=np.int8)
    elif t == MXFP4:
        a["e"] = g.integers(118, 131, size=nblk, dtype=np.uint8)
        a["qs"] = g.integers(0, 256, size=(nblk, 16), dtype=np.uint8)
    elif t == Q6_K:
        a["ql"] = g.integers(0, 256, size=(nblk, 128), dtype=np.uint8)
        a["qh"] = g.integers(0, 256, size=(nblk, 64), dtype=np.uint8)
        a["scales"] = g.integers(-128, 128, size=(nblk, 16), dtype=np.int8)
        a["d"] = _fp16_scales(g, nblk)
    elif t in (Q4_1, Q5_1):
        a["d"] = _fp16_scales(g, nblk)
        a["m"] = (g.standard_normal(nblk, dtype=np.float32) * np.float32(0.1)).astype(np.float16)
        if t == Q5_1:
            a["qh"] = g.integers(0, 2**32, size=nblk, dtype=np.uint32)
        a["qs"] = g.integers(0, 256, size=(nblk, 16), dtype=np.uint8)
    elif t == Q8_1:
        a["d"] = _fp16_scales(g, nblk)
        a["s"] = (g.standard_normal(nblk, dtype=np.float32)).astype(np.float16)   # not read as a weight
        a["qs"] = g.integers(-127, 128, size=(nblk, 32), dtype=np.int8)
    elif t == Q5_K:
        a["d"] = _fp16_scales(g, nblk)
        a["dmin"] = _fp16_scales(g, nblk)
        a["scales"] = g.integers(0, 256, size=(nblk, 12), dtype=np.uint8)
        a["qh"] = g.integers(0, 256, size=(nblk, 32), dtype=np.uint8)
        a["qs"] = g.integers(0, 256, size=(nblk, 128), dtype=np.uint8)
    elif t == Q2_K:
        a["scales"] = g.integers(0, 256, size=(nblk, 16), dtype=np.uint8)
        a["qs"] = g.integers(0, 256, size=(nblk, 64), dtype=np.uint8)
        a["d"] = _fp16_scales(g, nblk)
        a["dmin"] = _fp16_scales(g, nblk)
    elif t == Q3_K:
        a["hmask"] = g.integers(0, 256, size=(nblk, 32), dtype=np.uint8)
        a["qs"] = g.integers(0, 256, size=(nblk, 64), dtype=np.uint8)
        a["scales"] = g.integers(0, 256, size=(nblk, 12), dtype=np.uint8)
        a["d"] = _fp16_scales(g, nblk)
    else:
        raise ValueError(f"not a weight block type: {t}")
    return a.view(np.uint8).reshape(-1)


def activations(n_vec: int, cols: int, seed: int = 0, tensor_id: int = 1000) -> np.ndarray:
    return rng(seed, tensor_id).standard_normal((n_vec, cols), dtype=np.float32)


def bias(n_expert: int, rows: int, seed: int = 0, tensor_id: int = 2000) -> np.ndarray:
    return rng(seed, tensor_id).standard_normal((n_expert, rows), dtype=np.float32) * np.float32(0.02)


def router_weights(n_expert: int, hidden: int, seed: int = 0, tensor_id: int = 4000) -> np.ndarray:
    return rng(seed, tensor_id).standard_normal((n_expert, hidden), dtype=np.float32) * np.float32(0.05)


def router(n_tok: int, n_expert: int, k: int, seed: int = 0, tensor_id: int = 3000):
    """Top-k routing over N(0,1) logits -> (ids int32 [n_tok][k], gates fp32 [n_tok][k])."""
    logits = rng(seed, tensor_id).standard_normal((n_tok, n_expert), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]     # stable: ties keep the lower id
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    gates = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return order.astype(np.int32), gates
