#!/usr/bin/env python
"""Benchmark of the block-quantised decode path on GB300.

Workload (one step): a Qwen2.5-0.5B-shaped decode step through the W4A8 path
-- for each of 24 layers, the fp32 activations are quantised to Q8_0 blocks
and multiplied by q 896x896, k 128x896, v 128x896, o 896x896, gate 4864x896,
up 4864x896 and down 896x4864 weights in Q5_0; then the lm_head 151936x896 in
Q8_0.  Matrices that read the same activations are stored stacked (q|k|v,
gate|up), so a step is 97 matvec launches (4 per layer + lm_head), each
quantising its own input, chained with programmatic dependent launch;
390,648,832 weight bytes per step
(372.55 MiB), synthetic weights and N(0,1) activations, batch 1.
The weights (> 3x the 129 MB L2) are streamed cold every step.

Metric: weight GB/s = weight bytes of the step / step time (higher is
better), reported against the HBM roofline.  The step is captured once in a
CUDA graph and replayed; timing uses CUDA events on the replay stream.

Also reported: the dominant kernel for the roofline (the step's 96 Q5_0
layer matvecs, launched as in the step, ~95% of its launch time) and each of
their four shapes alone; the lm_head matvec alone; batch-8 and fp32-activation
(A32) forms of the step; end to end through host buffers; a single Q4_0
896x896 matvec (cold stream and single-call latency); the K-quant decode
shapes, the prefill GEMMs, the gpt-oss MoE layer and the weight quantiser;
and the CPU oracle on bounded samples of each (cpu_baseline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gguf_block_quantised_gb300 import synth  # noqa: E402

Q4_0, Q5_0, Q8_0, Q4_K, Q6_K, MXFP4, Q8_K, F32, BF16, MXFP4_R = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
NAMES = {Q4_0: "Q4_0", Q5_0: "Q5_0", Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", MXFP4: "MXFP4"}
LAYERS = 24
HID, FFN, KV, VOCAB = 896, 4864, 128, 151936
# (name, rows, cols, input index) per layer; inputs: 0 attn-in, 1 o-in, 2 ffn-in, 3 down-in
LAYER_MATS = [("q", HID, HID, 0), ("k", KV, HID, 0), ("v", KV, HID, 0), ("o", HID, HID, 1),
              ("gate", FFN, HID, 2), ("up", FFN, HID, 2), ("down", HID, FFN, 3)]
IN_COLS = [HID, HID, HID, FFN]
# Matrices that read the same input are stored stacked (rows concatenated) and
# multiplied by one launch: q|k|v, o, gate|up, down.  Same weights and bytes as
# the seven matrices; four dependent launches per layer.
LAYER_GROUPS = [[0, 1, 2], [3], [4, 5], [6]]


def row_bytes(t, cols):
    return synth.row_bytes(t, cols)


STEP_WEIGHT_BYTES = LAYERS * sum(r * row_bytes(Q5_0, c) for _, r, c, _ in LAYER_MATS) + VOCAB * row_bytes(Q8_0, HID)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            if hbm:
                return float(hbm), "measured"
        except Exception:
            pass
    return 6800.0, "fallback"


def load_tflops_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d.get("bf16_tflops") or 1900.0)
    except Exception:
        return 1900.0


# ---- clocks sampled during the timed region -----------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- the decode step ---------------------------------------------------------------------
class DecodeStep:
    """Weights and buffers of the Qwen2.5-0.5B-shaped decode step on one device.

    The seven matrices of a layer are held as four stacked groups (q|k|v,
    o, gate|up, down: the matrices of a group read the same activations), so
    a step is 24 x 4 + 1 = 97 matvecs.  fused=True: each matvec quantises
    its fp32 activations itself (QMV_FLAG_QUANTIZE_X) and is launched as a
    programmatic dependent of the one before (QMV_FLAG_PDL): 97 launches per
    step.  fused=False: separate qmv_quantize_act launches, plain stream
    order: 194 launches per step."""

    def __init__(self, q, torch, n_vec, seed=1, fused=True, a32=False):
        self.q, self.torch, self.n_vec, self.fused, self.a32 = q, torch, n_vec, fused, a32
        dev = torch.device("cuda")
        self.W = []
        tid = 0
        for layer in range(LAYERS):
            mats = [synth.weights(Q5_0, rows, cols, seed=seed, tensor_id=tid + m)
                    for m, (name, rows, cols, inp) in enumerate(LAYER_MATS)]
            tid += len(LAYER_MATS)
            groups = []
            for g in LAYER_GROUPS:
                rows = sum(LAYER_MATS[m][1] for m in g)
                cols, inp = LAYER_MATS[g[0]][2], LAYER_MATS[g[0]][3]
                W = np.concatenate([mats[m] for m in g])   # rows are contiguous: stacking = concatenation
                groups.append((torch.from_numpy(W).to(dev), rows, cols, inp))
            self.W.append(groups)
        self.lm = torch.from_numpy(synth.weights(Q8_0, VOCAB, HID, seed=seed, tensor_id=tid)).to(dev)
        # activations: 4 inputs per layer + the final hidden state
        self.x_host = [synth.activations(n_vec, IN_COLS[i], seed=seed, tensor_id=10000 + 4 * l + i)
                       for l in range(LAYERS) for i in range(4)] + [synth.activations(n_vec, HID, seed=seed,
                                                                                       tensor_id=20000)]
        # all activations of a step in one device buffer (views per input), so
        # that a step's inputs arrive from the host in one copy
        self.x_host_all = np.concatenate([a.reshape(-1) for a in self.x_host])
        self.x_all = torch.from_numpy(self.x_host_all).to(dev)
        self.x, o = [], 0
        for a in self.x_host:
            self.x.append(self.x_all[o:o + a.size].view(a.shape))
            o += a.size
        self.xq = [torch.empty(n_vec * q.qmv_row_bytes(Q8_0, a.shape[1]), dtype=torch.uint8, device=dev)
                   for a in self.x_host]
        self.y = [[torch.empty((n_vec, r), dtype=torch.float32, device=dev) for _, r, _, _ in self.W[0]]
                  for _ in range(LAYERS)]
        self.logits = torch.empty((n_vec, VOCAB), dtype=torch.float32, device=dev)
        per_layer = len(LAYER_GROUPS)
        self.launches = LAYERS * per_layer + 1 if fused else LAYERS * (4 + per_layer) + 2

    def run_layers(self, stream):
        """The step's 96 layer matvecs alone (no lm_head), launched as in run()."""
        q, n, s = self.q, self.n_vec, stream.cuda_stream
        fl = q.FLAG_QUANTIZE_X | q.FLAG_PDL
        for l in range(LAYERS):
            for m, (W, rows, cols, inp) in enumerate(self.W[l]):
                q.qmv_matvec(q.FMT(Q5_0, Q8_0) | fl, W, rows, cols, self.x[4 * l + inp], self.y[l][m], n, s)

    def run(self, stream):
        q, n = self.q, self.n_vec
        s = stream.cuda_stream
        if self.a32:
            # fp32 activations straight into the matvec (no quantisation), PDL chain
            for l in range(LAYERS):
                for m, (W, rows, cols, inp) in enumerate(self.W[l]):
                    q.qmv_matvec(q.FMT(Q5_0, F32) | q.FLAG_PDL, W, rows, cols, self.x[4 * l + inp], self.y[l][m],
                                 n, s)
            q.qmv_matvec(q.FMT(Q8_0, F32) | q.FLAG_PDL, self.lm, VOCAB, HID, self.x[-1], self.logits, n, s)
            return
        if self.fused:
            fl = q.FLAG_QUANTIZE_X | q.FLAG_PDL
            for l in range(LAYERS):
                for m, (W, rows, cols, inp) in enumerate(self.W[l]):
                    q.qmv_matvec(q.FMT(Q5_0, Q8_0) | fl, W, rows, cols, self.x[4 * l + inp], self.y[l][m], n, s)
            q.qmv_matvec(q.FMT(Q8_0, Q8_0) | fl, self.lm, VOCAB, HID, self.x[-1], self.logits, n, s)
            return
        for l in range(LAYERS):
            for i in range(4):
                j = 4 * l + i
                q.qmv_quantize_act(Q8_0, self.x[j], self.xq[j], n * IN_COLS[i], s)
            for m, (W, rows, cols, inp) in enumerate(self.W[l]):
                q.qmv_matvec(q.FMT(Q5_0, Q8_0), W, rows, cols, self.xq[4 * l + inp], self.y[l][m], n, s)
        q.qmv_quantize_act(Q8_0, self.x[-1], self.xq[-1], n * HID, s)
        q.qmv_matvec(q.FMT(Q8_0, Q8_0), self.lm, VOCAB, HID, self.xq[-1], self.logits, n, s)


def time_graph(torch, fn, stream, steps, warmup, sampler_index=None):
    """Capture fn(stream) once, replay warmup + steps times; returns (ms/step, clocks)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn(stream)                      # build-time set-up outside the capture
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn(stream)
    for _ in range(warmup):
        g.replay()
    stream.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = None
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    if sampler:
        sampler.__enter__()
        time.sleep(0.3)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            g.replay()
        end.record(stream)
    end.synchronize()
    if sampler:
        sampler.__exit__(None, None, None)
        clocks = sampler.summary()
    return start.elapsed_time(end) / steps, clocks


def cpu_baseline(n_steps=4):
    """The oracle (single thread) on a bounded sample: n_steps full decode steps."""
    from oracle import oracle as O
    rng_w = []
    tid = 0
    for layer in range(LAYERS):
        for name, rows, cols, inp in LAYER_MATS:
            rng_w.append((synth.weights(Q5_0, rows, cols, seed=1, tensor_id=tid), rows, cols, inp, Q5_0))
            tid += 1
    lm = synth.weights(Q8_0, VOCAB, HID, seed=1, tensor_id=tid)
    xs = [synth.activations(1, IN_COLS[i], seed=1, tensor_id=10000 + 4 * l + i) for l in range(LAYERS)
          for i in range(4)]
    xf = synth.activations(1, HID, seed=1, tensor_id=20000)
    t0 = time.perf_counter()
    for _ in range(n_steps):
        xq = [O.quantize_act(O.Q8_0, a) for a in xs]
        for k, (W, rows, cols, inp, t) in enumerate(rng_w):
            O.matvec(t, O.Q8_0, W, rows, cols, xq[4 * (k // 7) + inp], 1, want_abs=False)
        O.matvec(O.Q8_0, O.Q8_0, lm, VOCAB, HID, O.quantize_act(O.Q8_0, xf), 1, want_abs=False)
    dt = time.perf_counter() - t0
    return {"value": STEP_WEIGHT_BYTES * n_steps / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n_steps} full decode steps (batch 1, W4A8), single-threaded C oracle, {dt:.1f} s"}


def lm_roofline(q, torch, stream, step, dev_index, pdl=True):
    """The dominant kernel alone: the lm_head matvec (144.6 MB per launch),
    launched as in the decode step (quantising its fp32 input; with pdl, as a
    programmatic dependent of the launch before it).  Four copies of the
    weights rotate (578 MB > 4x L2), so every launch reads its weights from
    HBM; 200 launches replay from one CUDA graph.  Returns (ms per launch,
    clocks)."""
    lm_copies = [step.lm] + [step.lm.clone() for _ in range(3)]
    fl = q.FLAG_QUANTIZE_X | (q.FLAG_PDL if pdl else 0)

    def lm_only(s, Wl):
        q.qmv_matvec(q.FMT(Q8_0, Q8_0) | fl, Wl, VOCAB, HID, step.x[-1], step.logits, 1, s.cuda_stream)
    lm_reps = 200
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        lm_only(stream, lm_copies[0])
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(lm_reps):
                lm_only(stream, lm_copies[i % 4])
    for _ in range(3):
        g.replay()
    stream.synchronize()
    sampler = ClockSampler(dev_index)
    sampler.__enter__()
    time.sleep(0.2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(5):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    sampler.__exit__(None, None, None)
    del g, lm_copies
    return e0.elapsed_time(e1) / (5 * lm_reps), sampler.summary()


LAYER_BYTES_PER_STEP = LAYERS * sum(r * row_bytes(Q5_0, c) for _, r, c, _ in LAYER_MATS)
LAYER_LAUNCHES_PER_STEP = LAYERS * len(LAYER_GROUPS)


def layer_roofline(torch, stream, step, dev_index, reps=200):
    """The dominant kernel: the Q5_0 layer matvecs, which take ~95% of the
    step's launch time.  The step's 96 layer launches (q|k|v 1152x896, o
    896x896, gate|up 9728x896, down 896x4864 per layer; each quantising its
    fp32 input, a programmatic dependent of the one before) are replayed alone
    from one CUDA graph and timed with CUDA events on the replay stream.
    Their 246 MB of weights exceed L2, so every pass streams them from HBM.
    Returns (ms per launch on average, clocks)."""
    ms, clocks = time_graph(torch, step.run_layers, stream, reps, 10, sampler_index=dev_index)
    return ms / LAYER_LAUNCHES_PER_STEP, clocks


def layer_shapes_leg(q, torch, stream, step, hbm):
    """Each of the four stacked Q5_0 layer shapes alone, launched as in the step
    (fp32 input quantised in the kernel, PDL chain), round robin over enough
    weight copies (> 300 MB) that every launch reads its weights from HBM."""
    out = {}
    for m, (W0, rows, cols, inp) in enumerate(step.W[0]):
        x, y = step.x[inp], step.y[0][m]
        copies = [step.W[l][m][0] for l in range(LAYERS)]
        while sum(c.numel() for c in copies) < 300_000_000:
            copies.append(W0.clone())
        fmt = q.FMT(Q5_0, Q8_0) | q.FLAG_QUANTIZE_X | q.FLAG_PDL
        calls = [lambda s, W=W: q.qmv_matvec(fmt, W, rows, cols, x, y, 1, s.cuda_stream) for W in copies]
        ms = time_rotating(torch, stream, calls, max(len(copies), 100))
        nbytes = W0.numel()
        gbs = nbytes / (ms / 1e3) / 1e9
        out[f"{rows}x{cols}"] = {"us": ms * 1e3, "bytes": nbytes, "weight_gbs": gbs, "frac_of_hbm": gbs / hbm}
        del copies
    return out


def config1_leg(q, torch, stream, hbm):
    """A single Q4_0 896x896 matvec (451,584 weight bytes), fp32 activations
    (A32) and the W4A8 path (x quantised to Q8_0, in the kernel or by a
    separate qmv_quantize_act).  The matrix fits in L2 many times over, so
    (1) the cold-stream rate is taken round robin over 640 weight copies (289 MB,
    over twice L2), as plain launches and as a PDL chain, and (2) the latency
    of one call is the event-timed span of a single launch between idle
    periods, median of 50."""
    rows = cols = 896
    W0 = torch.from_numpy(synth.weights(Q4_0, rows, cols, seed=0)).cuda()
    copies = [W0] + [W0.clone() for _ in range(639)]
    x = torch.from_numpy(synth.activations(1, cols, seed=0)).cuda()
    xq = torch.empty(q.qmv_row_bytes(Q8_0, cols), dtype=torch.uint8, device="cuda")
    q.qmv_quantize_act(Q8_0, x, xq, cols)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    modes = {"A32": (q.FMT(Q4_0, F32), x), "A8_in_kernel": (q.FMT(Q4_0, Q8_0) | q.FLAG_QUANTIZE_X, x),
             "A8_prequantised": (q.FMT(Q4_0, Q8_0), xq)}
    res = {}
    for name, (fmt, xin) in modes.items():
        r = {}
        for pdl in (False, True):
            f = fmt | (q.FLAG_PDL if pdl else 0)
            calls = [lambda s, W=W, f=f: q.qmv_matvec(f, W, rows, cols, xin, y, 1, s.cuda_stream) for W in copies]
            ms = time_rotating(torch, stream, calls, len(copies))
            gbs = W0.numel() / (ms / 1e3) / 1e9
            r["pdl_chain" if pdl else "plain"] = {"us": ms * 1e3, "weight_gbs": gbs, "frac_of_hbm": gbs / hbm}
        lat = []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(60):
            with torch.cuda.stream(stream):
                e0.record(stream)
                q.qmv_matvec(fmt, copies[i % len(copies)], rows, cols, xin, y, 1, stream.cuda_stream)
                e1.record(stream)
            e1.synchronize()
            if i >= 10:
                lat.append(e0.elapsed_time(e1) * 1e3)
        r["single_call_latency_us"] = statistics.median(lat)
        res[name] = r
    q.qmv_get_status(stream)
    del copies
    return {"workload": "Q4_0 896x896, batch 1", "weight_bytes": W0.numel(), "by_mode": res}


def oracle_rate(fn, nbytes, min_s=2.0):
    """Single-threaded oracle rate on a bounded sample: fn() repeated for at
    least min_s seconds; returns (GB/s of weight bytes, seconds, calls)."""
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_s:
            return nbytes * n / dt / 1e9, dt, n


def time_rotating(torch, stream, calls, reps, warmup=3, timed=3):
    """Time `calls` (closures taking a stream, each on its own input copy so
    consecutive launches do not hit in L2) replayed round robin from one CUDA
    graph of `reps` calls: at least `warmup` replays and 20 ms of warm-up (so
    the clocks have ramped after the idle capture), then `timed` replays
    between CUDA events.  Returns ms per call."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in calls:
            c(stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                calls[i % len(calls)](stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    spent, n = 0.0, 0
    while n < warmup or spent < 20.0:
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        spent += e0.elapsed_time(e1)
        n += 1
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(timed):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / (timed * reps)


def kquant_decode_leg(q, torch, stream, hbm):
    """Llama-3-8B-shaped decode matvecs in K-quants (Q4_K 4096x4096,
    1024x4096, 14336x4096, 4096x14336; Q6_K lm_head 128256x4096) with Q8_K
    activations quantised in the kernel, at 1, 4 and 16 vectors.  Each shape
    is launched as in a decode step (a programmatic dependent of the launch
    before it), round robin over enough weight copies to exceed L2 twice, so
    every launch reads its weights from HBM.  Metric: weight GB/s."""
    shapes = [(Q4_K, 4096, 4096), (Q4_K, 1024, 4096), (Q4_K, 14336, 4096), (Q4_K, 4096, 14336),
              (Q6_K, 128256, 4096), (16, 14336, 4096)]
    res = {}
    for t, rows, cols in shapes:
        W0 = torch.from_numpy(synth.weights(t, rows, cols, seed=7)).cuda()
        copies = [W0] + [W0.clone() for _ in range(max(1, -(-300_000_000 // W0.numel())) - 1)]
        for nv in (1, 4, 16):
            x = torch.from_numpy(synth.activations(nv, cols, seed=8)).cuda()
            y = torch.empty((nv, rows), dtype=torch.float32, device="cuda")
            fmt = q.FMT(t, Q8_K) | q.FLAG_QUANTIZE_X | q.FLAG_PDL
            calls = [lambda s, W=W: q.qmv_matvec(fmt, W, rows, cols, x, y, nv, s.cuda_stream) for W in copies]
            reps = max(len(copies), 40)
            ms = time_rotating(torch, stream, calls, reps)
            gbs = W0.numel() / (ms / 1e3) / 1e9
            res[f"{NAMES.get(t, 'Q5_K')}_{rows}x{cols}_nv{nv}"] = {"us": ms * 1e3, "weight_gbs": gbs,
                                                                 "frac_of_hbm": gbs / hbm}
        del copies, W0
    q.qmv_get_status(stream)
    return {"metric": "decode matvec weight GB/s (K-quants, Q8_K activations quantised in-kernel, PDL chain)",
            "unit": "GB/s", "by_shape": res}


ALL_FORMATS = [(Q4_0, "Q4_0"), (11, "Q4_1"), (Q5_0, "Q5_0"), (12, "Q5_1"), (Q8_0, "Q8_0"), (13, "Q8_1"),
               (MXFP4, "MXFP4"), (14, "Q2_K"), (15, "Q3_K"), (Q4_K, "Q4_K"), (16, "Q5_K"), (Q6_K, "Q6_K"),
               (F32, "F32"), (17, "F16"), (BF16, "BF16")]


def formats_leg(q, torch, stream, hbm, rows=14336, cols=4096):
    """Every weight format on one Llama-3-8B-shaped matrix (14336x4096), batch
    1, launched as in a decode step (PDL chain; 8-bit activations quantised in
    the kernel for the block formats, fp32 for the plain ones), round robin
    over enough weight copies (> 300 MB) that every launch reads from HBM.
    Metric: weight bytes of the format / kernel time."""
    res = {}
    x = torch.from_numpy(synth.activations(1, cols, seed=8)).cuda()
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    for t, name in ALL_FORMATS:
        W0 = torch.from_numpy(synth.weights(t, rows, cols, seed=7)).cuda()
        copies = [W0] + [W0.clone() for _ in range(max(1, -(-300_000_000 // W0.numel())) - 1)]
        plain = t in (F32, 17, BF16)
        at = F32 if plain else (Q8_K if t in (Q4_K, Q6_K, 14, 15, 16) else Q8_0)
        fmt = q.FMT(t, at) | q.FLAG_PDL | (0 if plain else q.FLAG_QUANTIZE_X)
        calls = [lambda s, W=W: q.qmv_matvec(fmt, W, rows, cols, x, y, 1, s.cuda_stream) for W in copies]
        ms = time_rotating(torch, stream, calls, max(len(copies), 40))
        gbs = W0.numel() / (ms / 1e3) / 1e9
        res[name] = {"us": ms * 1e3, "bytes": W0.numel(), "bytes_per_weight": W0.numel() / (rows * cols),
                     "weight_gbs": gbs, "frac_of_hbm": gbs / hbm}
        del copies, W0
    q.qmv_get_status(stream)
    return {"metric": "decode matvec weight GB/s per format (14336x4096, batch 1, PDL chain)", "unit": "GB/s",
            "by_format": res}


def prefill_leg(q, torch, stream, tflops_peak):
    """Q4_K prefill GEMMs on the tensor cores (tcgen05): 14336x4096 and
    4096x14336 at M = 512 and 2048, with bf16 activations (weights dequantised
    to bf16) and with Q8_K activations (W4A8: exact integer block dots on fp16
    operands, plus its activation pre-pass).  Four (W, X) copies rotate so that
    every launch reads its operands from HBM (> L2 in total).  Both report
    2*M*rows*cols flops over the kernel time against the measured dense bf16
    peak (fp16 runs at the bf16 rate)."""
    out = {"bf16": {}, "w4a8": {}}
    tot = {"bf16": [0.0, 0.0], "w4a8": [0.0, 0.0]}
    ws = None
    for rows, cols in ((14336, 4096), (4096, 14336)):
        Ws = [torch.from_numpy(synth.weights(Q4_K, rows, cols, seed=4, tensor_id=rows + i)).cuda() for i in range(4)]
        for m in (512, 2048):
            flop = 2.0 * m * rows * cols
            Xs = [torch.randn(m, cols, device="cuda").to(torch.bfloat16) for _ in range(4)]
            Y = torch.empty(m, rows, device="cuda")
            calls = [(lambda s, W=W, X=X: q.qmv_matmul(q.FMT(Q4_K, BF16), W, rows, cols, X, Y, m, s.cuda_stream))
                     for W, X in zip(Ws, Xs)]
            ms = time_rotating(torch, stream, calls, 40)
            out["bf16"][f"{rows}x{cols}_m{m}"] = {"ms": ms, "tflops": flop / (ms / 1e3) / 1e12,
                                                 "frac_of_peak": flop / (ms / 1e3) / 1e12 / tflops_peak}
            tot["bf16"][0] += flop
            tot["bf16"][1] += ms
            del Xs
            Xq = []
            for _ in range(4):
                xq = torch.empty(m * q.qmv_row_bytes(Q8_K, cols), dtype=torch.uint8, device="cuda")
                q.qmv_quantize_act(Q8_K, torch.randn(m, cols, device="cuda"), xq, m * cols)
                Xq.append(xq)
            need = q.qmv_workspace_size(q.OP_MATMUL, q.FMT(Q4_K, Q8_K), rows, cols, m)
            if ws is None or ws.numel() < need:
                ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            q.qmv_set_workspace(ws, ws.numel())
            calls = [(lambda s, W=W, X=X: q.qmv_matmul(q.FMT(Q4_K, Q8_K), W, rows, cols, X, Y, m, s.cuda_stream))
                     for W, X in zip(Ws, Xq)]
            ms = time_rotating(torch, stream, calls, 40)
            q.qmv_set_workspace(None, 0)
            out["w4a8"][f"{rows}x{cols}_m{m}"] = {"ms": ms, "tflops": flop / (ms / 1e3) / 1e12,
                                                 "frac_of_peak": flop / (ms / 1e3) / 1e12 / tflops_peak}
            tot["w4a8"][0] += flop
            tot["w4a8"][1] += ms
            del Xq, Y
        del Ws
    q.qmv_get_status(stream)
    agg = {k: tot[k][0] / (tot[k][1] / 1e3) / 1e12 for k in tot}
    formats = prefill_formats(q, torch, stream, tflops_peak)
    return {"metric": "prefill GEMM TFLOP/s (Q4_K weights; bf16 and W4A8 activations, fp32 accumulate)",
            "unit": "TFLOP/s", "value": agg["bf16"], "frac": agg["bf16"] / tflops_peak,
            "w4a8_value": agg["w4a8"], "w4a8_frac": agg["w4a8"] / tflops_peak, "peak": tflops_peak,
            "shapes": out["bf16"], "w4a8": out["w4a8"], "formats": formats,
            "kernels": {"bf16": "k_gemm_q4k_bf16 (tcgen05.mma kind::f16 bf16, M=128 rows x N=256 tokens, A in TMEM)",
                        "w4a8": "k_w4a8_prep + k_gemm_q4k_w4a8 (tcgen05.mma kind::f16 on fp16 integer operands, "
                                "M=128 x N=128, S and Mn drained per super-block)"}}


def moe_leg(q, torch, stream, hbm, tflops_peak=None):
    """gpt-oss-20B-shaped MoE layer: 32 MXFP4 experts, gate_up 5760x2880 (up
    form, x shared by the 4 slots) then down 2880x2880 (per-slot inputs,
    gate-weighted), fp32 biases, top-4 of N(0,1) router logits.  Two paths:
    W4A8 (fp32 activations quantised to Q8_0 inside the grouped matvec) and
    bf16 activations through the grouped tensor-core GEMM.  Metric: distinct
    expert weight bytes read per layer / time, and useful TFLOP/s."""
    E, k = 32, 4
    Wgu = torch.from_numpy(synth.weights(MXFP4, E * 5760, 2880, seed=5, tensor_id=1)).cuda()
    Wd = torch.from_numpy(synth.weights(MXFP4, E * 2880, 2880, seed=5, tensor_id=2)).cuda()
    bgu = torch.from_numpy(synth.bias(E, 5760, seed=5)).cuda()
    bd = torch.from_numpy(synth.bias(E, 2880, seed=5, tensor_id=2001)).cuda()
    # the same experts repacked once (qmv_repack, MXFP4 -> MXFP4_R rows)
    Wgu_r = torch.empty(E * 5760 * q.qmv_row_bytes(MXFP4_R, 2880), dtype=torch.uint8, device="cuda")
    Wd_r = torch.empty(E * 2880 * q.qmv_row_bytes(MXFP4_R, 2880), dtype=torch.uint8, device="cuda")
    q.qmv_repack(MXFP4, Wgu, E * 5760, 2880, Wgu_r)
    q.qmv_repack(MXFP4, Wd, E * 2880, 2880, Wd_r)
    Wr = torch.from_numpy(synth.router_weights(E, 2880, seed=5)).cuda()
    br = torch.from_numpy(synth.bias(1, E, seed=5, tensor_id=4001)[0]).cuda()
    paths = {"w4a8": (q.FMT(MXFP4, Q8_0) | q.FLAG_QUANTIZE_X, torch.float32, Wgu, Wd),
             "bf16_gemm": (q.FMT(MXFP4, BF16), torch.bfloat16, Wgu, Wd),
             "bf16_gemm_repacked": (q.FMT(MXFP4_R, BF16), torch.bfloat16, Wgu_r, Wd_r),
             "mx_gemm": (q.FMT(MXFP4, q.MXFP8), torch.float32, Wgu, Wd),
             "mx_gemm_repacked": (q.FMT(MXFP4_R, q.MXFP8), torch.float32, Wgu_r, Wd_r)}
    # the tensor peak of each path's MMA: bf16 (kind::f16) measured; fp8 (the
    # block-scaled kind) as twice the bf16 figure, the nominal dense ratio
    peak_of = {"bf16_gemm": tflops_peak, "bf16_gemm_repacked": tflops_peak,
               "mx_gemm": 2 * tflops_peak if tflops_peak else None,
               "mx_gemm_repacked": 2 * tflops_peak if tflops_peak else None}
    out = {}
    ws = None
    for name, (fmt, xdt, Wgu_p, Wd_p) in paths.items():
        res = {}
        for n_tok in (1, 64, 1024):
            # four routings rotate, so the experts one launch reads were not just read
            routes = [synth.router(n_tok, E, k, seed=6 + r) for r in range(4)]
            x = torch.randn(n_tok, 2880, device="cuda").to(xdt)
            h = torch.randn(n_tok, k, 2880, device="cuda").to(xdt)
            y1 = torch.empty(n_tok, k, 5760, device="cuda")
            y2 = torch.empty(n_tok, 2880, device="cuda")
            need = q.qmv_workspace_size(q.OP_MOE, fmt, 5760, 2880, n_tok * k)
            if ws is None or ws.numel() < need:
                ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            q.qmv_set_workspace(ws, ws.numel())
            calls = []
            for ids_np, gates_np in routes:
                ids, gates = torch.from_numpy(ids_np).cuda(), torch.from_numpy(gates_np).cuda()

                def layer(s, ids=ids, gates=gates, fmt=fmt, x=x, h=h, y1=y1, y2=y2, n_tok=n_tok, A=Wgu_p, B=Wd_p):
                    q.qmv_moe_matvec(fmt, A, E, 5760, 2880, ids, None, k, x, y1, n_tok, bgu, s.cuda_stream)
                    q.qmv_moe_matvec(fmt, B, E, 2880, 2880, ids, gates, k, h, y2, n_tok, bd, s.cuda_stream)
                calls.append(layer)
            reps = 20 if n_tok >= 1024 else 100
            ms = time_rotating(torch, stream, calls, reps)
            used = float(np.mean([len(np.unique(r[0])) for r in routes]))
            wbytes = used * (5760 + 2880) * synth.row_bytes(MXFP4, 2880)
            flop = 2.0 * n_tok * k * (5760 + 2880) * 2880
            res[f"tok{n_tok}"] = {"ms": ms, "experts_used": used, "weight_bytes": int(wbytes),
                                  "weight_gbs": wbytes / (ms / 1e3) / 1e9,
                                  "frac_of_hbm": wbytes / (ms / 1e3) / 1e9 / hbm,
                                  "tflops": flop / (ms / 1e3) / 1e12}
            if peak_of.get(name):
                res[f"tok{n_tok}"]["frac_of_tensor_peak"] = flop / (ms / 1e3) / 1e12 / peak_of[name]
            res[f"block_tok{n_tok}"] = block_time(q, torch, stream, fmt, Wgu_p, Wd_p, bgu, bd, Wr, br, n_tok, hbm)
        out[name] = res
    q.qmv_set_workspace(None, 0)
    q.qmv_get_status(stream)
    return {"metric": "MoE layer (gate_up + down) expert weight GB/s", "unit": "GB/s", "by_path": out,
            "block": "block_tok*: qmv_moe_block, the whole block from fp32 hidden states (router 32x2880 fp32, "
                     "top 4, gate_up, clipped SwiGLU, down): k_router + k_topk + the path's expert kernels + "
                     "k_swiglu; four hidden-state batches rotate (each routes its own way)",
            "paths": {"w4a8": "k_moe_group + k_moe_gemv (dp4a, grouped per expert) + k_moe_combine",
                      "bf16_gemm": "k_moe_group + k_moe_tiles + k_moe_gather + k_moe_gemm_mxfp4_bf16 (tcgen05) "
                                   "+ k_moe_combine",
                      "bf16_gemm_repacked": "the same on MXFP4_R experts (qmv_repack once; TMA tensor copies of "
                                            "the codes and exponents)",
                      "mx_gemm": "k_moe_group + k_moe_tiles + k_moe_gather_mxfp8 (fp32 -> MXFP8) + "
                                 "k_moe_gemm_mxfp4<MX> (tcgen05 kind::mxf8f6f4.block_scale) + k_moe_combine",
                      "mx_gemm_repacked": "the same on MXFP4_R experts"},
            "tensor_peaks_tflops": {"bf16": tflops_peak, "fp8": 2 * tflops_peak if tflops_peak else None,
                                    "fp8_kind": "twice the measured bf16 burst (nominal dense fp8/bf16 ratio)"}}


def block_time(q, torch, stream, fmt, Wgu, Wd, bgu, bd, Wr, br, n_tok, hbm, E=32, k=4, hidden=2880, inter=2880):
    """qmv_moe_block on gpt-oss-shaped experts; fmt's flags are dropped (the block
    always quantises 8-bit activations itself)."""
    fmt &= 0xffff
    xs = [torch.from_numpy(synth.activations(n_tok, hidden, seed=40 + r)).cuda() for r in range(4)]
    y = torch.empty(n_tok, hidden, device="cuda")
    ids = torch.empty(n_tok, k, dtype=torch.int32, device="cuda")
    gates = torch.empty(n_tok, k, device="cuda")
    ws = torch.empty(q.qmv_moe_block_workspace_size(fmt, E, k, hidden, inter, n_tok), dtype=torch.uint8,
                     device="cuda")
    used = []
    for x in xs:
        q.qmv_set_workspace(ws, ws.numel())
        q.qmv_moe_block(fmt, E, k, hidden, inter, Wr, br, Wgu, bgu, Wd, bd, 1.702, 7.0, x, n_tok, y, ids, gates,
                        stream.cuda_stream)
        torch.cuda.synchronize()
        used.append(len(np.unique(ids.cpu().numpy())))
    calls = [lambda s, x=x: q.qmv_moe_block(fmt, E, k, hidden, inter, Wr, br, Wgu, bgu, Wd, bd, 1.702, 7.0, x,
                                            n_tok, y, ids, gates, s.cuda_stream) for x in xs]
    ms = time_rotating(torch, stream, calls, 20 if n_tok >= 1024 else 100)
    wbytes = float(np.mean(used)) * (2 * inter + hidden) * synth.row_bytes(MXFP4, hidden)
    return {"ms": ms, "experts_used": float(np.mean(used)), "weight_gbs": wbytes / (ms / 1e3) / 1e9,
            "frac_of_hbm": wbytes / (ms / 1e3) / 1e9 / hbm}


def prefill_formats(q, torch, stream, tflops_peak):
    """The prefill product for the other formats of the pages' prefill mix (and
    Q4_0) on the same shapes, bf16 activations: Q4_0 / Q5_0 / Q8_0 / Q6_K rows of
    whole 16 bytes dequantise tiles into TMEM inside the GEMM (k_gemm_deq_bf16);
    the Qwen2-0.5B layer shapes whose rows are not (896 columns: 616-byte Q5_0
    rows) convert to bf16 in the workspace first (k_dequant_bf16 + k_gemm_bf16),
    timed whole.  BF16 rows go straight into the plain bf16 GEMM (k_gemm_bf16),
    and MXFP4 rows (no tile dequantiser) take the two passes.  Four (W, X)
    copies rotate, as for Q4_K."""
    out = {}
    cases = [(t, rows, cols, m) for t in (Q8_0, Q5_0, Q6_K, Q4_0) for rows, cols in ((14336, 4096), (4096, 14336))
             for m in (512, 2048)] + [(Q5_0, 4864, 896, 512), (Q5_0, 896, 4864, 512)]
    cases += [(t, 14336, 4096, m) for t in (BF16, MXFP4) for m in (512, 2048)]
    names = {Q4_0: "Q4_0", Q5_0: "Q5_0", Q8_0: "Q8_0", Q6_K: "Q6_K", BF16: "BF16", MXFP4: "MXFP4"}
    ws = None
    for t, rows, cols, m in cases:
        flop = 2.0 * m * rows * cols
        Ws = [torch.from_numpy(synth.weights(t, rows, cols, seed=4, tensor_id=rows + i)).cuda() for i in range(4)]
        Xs = [torch.randn(m, cols, device="cuda").to(torch.bfloat16) for _ in range(4)]
        Y = torch.empty(m, rows, device="cuda")
        need = q.qmv_workspace_size(q.OP_MATMUL, q.FMT(t, BF16), rows, cols, m)
        if need and (ws is None or ws.numel() < need):
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        if need:
            q.qmv_set_workspace(ws, ws.numel())
        calls = [(lambda s, W=W, X=X: q.qmv_matmul(q.FMT(t, BF16), W, rows, cols, X, Y, m, s.cuda_stream))
                 for W, X in zip(Ws, Xs)]
        ms = time_rotating(torch, stream, calls, 40)
        q.qmv_set_workspace(None, 0)
        out[f"{names[t]}_{rows}x{cols}_m{m}"] = {
            "ms": ms, "tflops": flop / (ms / 1e3) / 1e12, "frac_of_peak": flop / (ms / 1e3) / 1e12 / tflops_peak,
            "path": "two passes (bf16 in the workspace)" if need else
                    ("bf16 rows as they are" if t == BF16 else "tiles dequantised inside the GEMM")}
        del Ws, Xs, Y
    q.qmv_get_status(stream)
    return out


def run_probe(spec):
    """Single-kernel runs for profiling (ncu captures).  Specs:
      gemv:T:rows:cols:atype:n_vec   qmv_matvec on synthetic weights (atype 8 = fp32)
      gemm:rows:cols:m[:T]           qmv_matmul, weight type T (default Q4_K) x bf16; other types than
                                     Q4_K run the two-pass product (bf16 dequantisation, then the GEMM)
      gemm8:rows:cols:m              qmv_matmul, Q4_K x Q8_K (W4A8, with its activation pre-pass)
      step[:n_vec]                   one fused decode step of the Qwen2.5-0.5B shape (97 matvecs)
      block:n_tok[:atype]            qmv_moe_block on the gpt-oss MoE shapes (atype 3 = Q8_0, 8 = fp32, 9 = bf16)
      moe:n_tok[:atype[:repacked]]   one gpt-oss-shaped MoE layer (gate_up + down); atype 3 = Q8_0
                                     quantised in-kernel (default), 9 = bf16 (grouped tensor-core GEMM),
                                     18 = MXFP8 (block-scaled tensor-core GEMM); repacked 1: experts
                                     repacked to MXFP4_R first (bf16 and MXFP8 only)
    Each runs its call five times and prints the event-timed mean of the last three."""
    import torch
    import gguf_block_quantised_gb300 as q
    from gguf_block_quantised_gb300 import build as B
    B.build()
    q.load()
    parts = spec.split(":")
    kind, a = parts[0], [int(v) for v in parts[1:]]
    if kind == "gemv":
        t, rows, cols, at, nv = a
        W = torch.from_numpy(synth.weights(t, rows, cols, seed=1)).cuda()
        x = torch.from_numpy(synth.activations(nv, cols)).cuda()
        if at != F32:
            xq = torch.empty(nv * q.qmv_row_bytes(at, cols), dtype=torch.uint8, device="cuda")
            q.qmv_quantize_act(at, x, xq, nv * cols)
            x = xq
        y = torch.empty((nv, rows), dtype=torch.float32, device="cuda")
        call = lambda: q.qmv_matvec(q.FMT(t, at), W, rows, cols, x, y, nv)
        nbytes, what = W.numel(), "weight GB/s"
    elif kind == "gemm":
        rows, cols, m, t = (a + [Q4_K])[:4]
        W = torch.from_numpy(synth.weights(t, rows, cols, seed=1)).cuda()
        X = torch.randn(m, cols, device="cuda").to(torch.bfloat16)
        Y = torch.empty(m, rows, device="cuda")
        need = q.qmv_workspace_size(q.OP_MATMUL, q.FMT(t, BF16), rows, cols, m)
        if need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            q.qmv_set_workspace(ws, ws.numel())
        call = lambda: q.qmv_matmul(q.FMT(t, BF16), W, rows, cols, X, Y, m)
        nbytes, what = 2 * m * rows * cols / 1e3, "TFLOP/s"
    elif kind == "gemm8":
        rows, cols, m = a
        W = torch.from_numpy(synth.weights(Q4_K, rows, cols, seed=1)).cuda()
        X = torch.empty(m * q.qmv_row_bytes(Q8_K, cols), dtype=torch.uint8, device="cuda")
        q.qmv_quantize_act(Q8_K, torch.randn(m, cols, device="cuda"), X, m * cols)
        Y = torch.empty(m, rows, device="cuda")
        ws = torch.empty(q.qmv_workspace_size(q.OP_MATMUL, q.FMT(Q4_K, Q8_K), rows, cols, m), dtype=torch.uint8,
                         device="cuda")
        q.qmv_set_workspace(ws, ws.numel())
        call = lambda: q.qmv_matmul(q.FMT(Q4_K, Q8_K), W, rows, cols, X, Y, m)
        nbytes, what = 2 * m * rows * cols / 1e3, "TFLOP/s"
    elif kind == "step":
        (n_vec,) = (a + [1])[:1]
        step = DecodeStep(q, torch, n_vec)
        stream = torch.cuda.current_stream()
        call = lambda: step.run(stream)
        nbytes, what = STEP_WEIGHT_BYTES, "weight GB/s"
    elif kind == "block":
        n_tok, at = (a + [Q8_0][len(a) - 1:])[:2]
        E, k, hid, inter = 32, 4, 2880, 2880
        Wgu = torch.from_numpy(synth.weights(MXFP4, E * 2 * inter, hid, seed=5, tensor_id=1)).cuda()
        Wd = torch.from_numpy(synth.weights(MXFP4, E * hid, inter, seed=5, tensor_id=2)).cuda()
        bgu = torch.from_numpy(synth.bias(E, 2 * inter, seed=5)).cuda()
        bd = torch.from_numpy(synth.bias(E, hid, seed=5, tensor_id=2001)).cuda()
        Wr = torch.from_numpy(synth.router_weights(E, hid, seed=5)).cuda()
        br = torch.from_numpy(synth.bias(1, E, seed=5, tensor_id=4001)[0]).cuda()
        x = torch.from_numpy(synth.activations(n_tok, hid, seed=40)).cuda()
        y = torch.empty(n_tok, hid, device="cuda")
        ids = torch.empty(n_tok, k, dtype=torch.int32, device="cuda")
        gates = torch.empty(n_tok, k, device="cuda")
        fmt = q.FMT(MXFP4, at)
        ws = torch.empty(q.qmv_moe_block_workspace_size(fmt, E, k, hid, inter, n_tok), dtype=torch.uint8,
                         device="cuda")
        q.qmv_set_workspace(ws, ws.numel())
        call = lambda: q.qmv_moe_block(fmt, E, k, hid, inter, Wr, br, Wgu, bgu, Wd, bd, 1.702, 7.0, x, n_tok, y, ids,
                                       gates)
        call()
        torch.cuda.synchronize()
        nbytes = len(np.unique(ids.cpu().numpy())) * (2 * inter + hid) * synth.row_bytes(MXFP4, hid)
        what = "expert weight GB/s"
    elif kind == "moe":
        n_tok, at, repacked = (a + [Q8_0, 0][len(a) - 1:])[:3]
        E, k = 32, 4
        Wgu = torch.from_numpy(synth.weights(MXFP4, E * 5760, 2880, seed=5, tensor_id=1)).cuda()
        Wd = torch.from_numpy(synth.weights(MXFP4, E * 2880, 2880, seed=5, tensor_id=2)).cuda()
        bgu = torch.from_numpy(synth.bias(E, 5760, seed=5)).cuda()
        bd = torch.from_numpy(synth.bias(E, 2880, seed=5, tensor_id=2001)).cuda()
        ids_np, gates_np = synth.router(n_tok, E, k, seed=6)
        ids, gates = torch.from_numpy(ids_np).cuda(), torch.from_numpy(gates_np).cuda()
        xdt = torch.bfloat16 if at == BF16 else torch.float32
        x = torch.randn(n_tok, 2880, device="cuda").to(xdt)
        h = torch.randn(n_tok, k, 2880, device="cuda").to(xdt)
        y1 = torch.empty(n_tok, k, 5760, device="cuda")
        y2 = torch.empty(n_tok, 2880, device="cuda")
        fmt = q.FMT(MXFP4, at) if at in (BF16, q.MXFP8) else q.FMT(MXFP4, Q8_0) | q.FLAG_QUANTIZE_X
        if repacked and at in (BF16, q.MXFP8):
            Wgu_r = torch.empty(E * 5760 * q.qmv_row_bytes(MXFP4_R, 2880), dtype=torch.uint8, device="cuda")
            Wd_r = torch.empty(E * 2880 * q.qmv_row_bytes(MXFP4_R, 2880), dtype=torch.uint8, device="cuda")
            q.qmv_repack(MXFP4, Wgu, E * 5760, 2880, Wgu_r)
            q.qmv_repack(MXFP4, Wd, E * 2880, 2880, Wd_r)
            Wgu, Wd, fmt = Wgu_r, Wd_r, q.FMT(MXFP4_R, at)
        ws = torch.empty(q.qmv_workspace_size(q.OP_MOE, fmt, 5760, 2880, n_tok * k), dtype=torch.uint8, device="cuda")
        q.qmv_set_workspace(ws, ws.numel())

        def call():
            q.qmv_moe_matvec(fmt, Wgu, E, 5760, 2880, ids, None, k, x, y1, n_tok, bgu)
            q.qmv_moe_matvec(fmt, Wd, E, 2880, 2880, ids, gates, k, h, y2, n_tok, bd)
        nbytes = len(np.unique(ids_np)) * (5760 + 2880) * synth.row_bytes(MXFP4, 2880)
        what = "expert weight GB/s"
    else:
        raise SystemExit(f"unknown probe {spec}")
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        call()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / 3
    q.qmv_get_status()
    print(json.dumps({"probe": spec, "ms": ms, what: nbytes / (ms / 1e3) / 1e9}))
    return 0


def traffic_for(kernel):
    """DRAM bytes per launch from the committed ncu record, if the kernel's
    source is unchanged since that capture; else None."""
    import hashlib
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kernel]
        src = os.path.join(ROOT, "gguf_block_quantised_gb300", "csrc")
        h = hashlib.sha1(b"".join(open(os.path.join(src, f), "rb").read()
                                  for f in ["common.cuh", "formats.cuh", "gemv.cuh", "gemv_launch.cuh"])).hexdigest()
        return rec["dram_bytes"] if h == rec["source_sha1"] else None
    except Exception:
        return None


def max_over_ranks(torch, values, device):
    """The element-wise maximum of `values` over the ranks of the process group
    (a copy of `values` for a single process): replicas report the slowest
    rank's time, so value = all ranks' units / that time."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def wquant_leg(q, torch, stream, hbm):
    """The weight quantiser (qmv_quantize_weights): a 14336x4096 matrix (fp32
    235 MB, or bf16 117 MB; two copies alternating so each launch reads from
    HBM) to every block type it writes.  Bytes = the weights read plus the
    blocks written."""
    rows, cols = 14336, 4096
    n = rows * cols
    g = torch.Generator(device="cuda").manual_seed(7)
    src = [torch.randn(rows, cols, device="cuda", generator=g) * 0.02 for _ in range(2)]
    srcb = [w.to(torch.bfloat16) for w in src]
    res = {}
    cases = [(Q4_0, "Q4_0", False), (11, "Q4_1", False), (Q5_0, "Q5_0", False), (12, "Q5_1", False),
             (Q8_0, "Q8_0", False), (Q4_K, "Q4_K", False), (16, "Q5_K", False), (Q6_K, "Q6_K", False),
             (Q4_0, "Q4_0_from_bf16", True), (Q4_K, "Q4_K_from_bf16", True)]
    for t, name, bf in cases:
        out = torch.empty(rows * q.qmv_row_bytes(t, cols), dtype=torch.uint8, device="cuda")
        fmt = q.FMT(t, BF16) if bf else t
        ins = srcb if bf else src
        nbytes = (2 if bf else 4) * n + out.numel()
        with torch.cuda.stream(stream):
            for i in range(4):
                q.qmv_quantize_weights(fmt, ins[i % 2], rows, cols, out, stream.cuda_stream)
            reps = 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(reps):
                q.qmv_quantize_weights(fmt, ins[i % 2], rows, cols, out, stream.cuda_stream)
            e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms / 1e3) / 1e9
        res[name] = {"us": 1e3 * ms, "gbs": gbs, "frac_of_hbm": gbs / hbm, "bytes": nbytes}
        del out
    q.qmv_get_status(stream)
    del src, srcb
    torch.cuda.empty_cache()
    return {"metric": "weight quantiser GB/s (weights read + blocks written)", "unit": "GB/s",
            "shape": f"{rows}x{cols}", "by_type": res,
            "kernels": "k_quant_w32 (32-element formats: eight threads per block), k_quant_wk (K-quants: one warp "
                       "per super-block)"}


def _oracle_step_workload():
    """The decode step's matrices and activations for the oracle (single thread)."""
    mats, tid = [], 0
    for layer in range(LAYERS):
        for name, rows, cols, inp in LAYER_MATS:
            mats.append((synth.weights(Q5_0, rows, cols, seed=1, tensor_id=tid), rows, cols, 4 * layer + inp, Q5_0))
            tid += 1
    mats.append((synth.weights(Q8_0, VOCAB, HID, seed=1, tensor_id=tid), VOCAB, HID, 4 * LAYERS, Q8_0))
    xs = [synth.activations(1, IN_COLS[i], seed=1, tensor_id=10000 + 4 * l + i) for l in range(LAYERS)
          for i in range(4)] + [synth.activations(1, HID, seed=1, tensor_id=20000)]
    return mats, xs


def _oracle_work_items(mats, slice_bytes=8 << 20):
    """The step's matrices as work items in step order; matrices larger than
    slice_bytes (the lm_head) are cut into row slices of about that size."""
    items = []
    for k, (W, rows, cols, xi, t) in enumerate(mats):
        rb = row_bytes(t, cols)
        step = max(1, slice_bytes // rb)
        for r0 in range(0, rows, step):
            items.append((k, r0, min(rows, r0 + step)))
    return items


def _oracle_items(O, mats, xs, items):
    """The oracle on some work items (their activations quantised first).
    Returns (seconds, weight bytes)."""
    t0 = time.perf_counter()
    xq = {}
    nbytes = 0
    for k, r0, r1 in items:
        W, rows, cols, xi, t = mats[k]
        if xi not in xq:
            xq[xi] = O.quantize_act(O.Q8_0, xs[xi])
        rb = row_bytes(t, cols)
        O.matvec(t, O.Q8_0, W[r0 * rb:r1 * rb], r1 - r0, cols, xq[xi], 1, want_abs=False)
        nbytes += (r1 - r0) * rb
    return time.perf_counter() - t0, nbytes


# ---- the oracle on every host core: a pool of spawned processes ----------------------
# Each worker builds a workload once (from the same seeds as the GPU legs) and
# then computes its static share of it per step: rows of every matrix (decode
# step, prefill slice) or tokens (mixture of experts).
_PW = {}

PREFILL_CPU = (14336, 4096, 64)          # the 14336x4096 prefill on a 64-token slice
MOE_CPU_TOKENS = 64


def _prefill_workload(O):
    rows, cols, m = PREFILL_CPU
    import torch
    W = synth.weights(Q4_K, rows, cols, seed=4, tensor_id=rows)
    x = synth.activations(m, cols, seed=9)
    xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    return W, xb, O.quantize_act(O.Q8_K, x)


def _moe_workload(O, n_tok):
    E, k = 32, 4
    Wgu = synth.weights(MXFP4, E * 5760, 2880, seed=5, tensor_id=1)
    Wd = synth.weights(MXFP4, E * 2880, 2880, seed=5, tensor_id=2)
    bgu, bd = synth.bias(E, 5760, seed=5), synth.bias(E, 2880, seed=5, tensor_id=2001)
    ids, gates = synth.router(n_tok, E, k, seed=6)
    x = O.quantize_act(O.Q8_0, synth.activations(n_tok, 2880, seed=10))
    h = O.quantize_act(O.Q8_0, synth.activations(n_tok * k, 2880, seed=11).reshape(n_tok, k, 2880))
    return Wgu, Wd, bgu, bd, ids, gates, x, h


def _moe_tokens(O, wl, t0, t1):
    """The oracle's W4A8 MoE layer (gate_up up form, then down gate-weighted) on tokens t0..t1."""
    Wgu, Wd, bgu, bd, ids, gates, x, h = wl
    E, k = 32, 4
    O.moe(O.MXFP4, O.Q8_0, Wgu, E, 5760, 2880, ids[t0:t1], None, k, x[t0:t1], t1 - t0, bias=bgu)
    O.moe(O.MXFP4, O.Q8_0, Wd, E, 2880, 2880, ids[t0:t1], gates[t0:t1], k, h[t0:t1], t1 - t0, bias=bd)


def _pw_init(kind):
    from oracle import oracle as O
    _PW["O"] = O
    if kind == "decode":
        _PW[kind] = _oracle_step_workload()
    elif kind.startswith("prefill"):
        _PW[kind] = _prefill_workload(O)
    elif kind == "moe":
        _PW[kind] = _moe_workload(O, MOE_CPU_TOKENS)


def _pw_task(args):
    """One worker's share of one step of workload `kind`."""
    kind, w, nw = args
    O = _PW["O"]
    if kind == "decode":
        mats, xs = _PW[kind]
        xq = [O.quantize_act(O.Q8_0, a) for a in xs]
        for W, rows, cols, xi, t in mats:
            r0, r1 = rows * w // nw, rows * (w + 1) // nw
            if r1 > r0:
                rb = row_bytes(t, cols)
                O.matvec(t, O.Q8_0, W[r0 * rb:r1 * rb], r1 - r0, cols, xq[xi], 1, want_abs=False)
    elif kind.startswith("prefill"):
        W, xb, xq = _PW[kind]
        rows, cols, m = PREFILL_CPU
        r0, r1 = rows * w // nw, rows * (w + 1) // nw
        rb = row_bytes(Q4_K, cols)
        at, xin = (O.BF16, xb) if kind == "prefill_bf16" else (O.Q8_K, xq)
        if r1 > r0:
            O.matvec(O.Q4_K, at, W[r0 * rb:r1 * rb], r1 - r0, cols, xin, m, want_abs=False)
    elif kind == "moe":
        t0, t1 = MOE_CPU_TOKENS * w // nw, MOE_CPU_TOKENS * (w + 1) // nw
        if t1 > t0:
            _moe_tokens(O, _PW[kind], t0, t1)
    return w


def pool_time(kind, n_steps):
    """Seconds per step of workload `kind` on every host core (a warm step first)."""
    import multiprocessing as mp
    nw = os.cpu_count() or 1
    tasks = [(kind, w, nw) for w in range(nw)]
    # map_async with a time limit: a worker that dies would leave a plain map waiting forever
    with mp.get_context("spawn").Pool(nw, initializer=_pw_init, initargs=(kind,)) as pool:
        pool.map_async(_pw_task, tasks, chunksize=1).get(timeout=600)   # set-up and a warm step
        t0 = time.perf_counter()
        for _ in range(n_steps):
            pool.map_async(_pw_task, tasks, chunksize=1).get(timeout=300)
        dt = time.perf_counter() - t0
    return dt / n_steps, nw


def cpu_baseline_all_cores(n_steps=8):
    """The oracle on every host core: a pool of processes (spawned, never forked
    from a process that has used the GPU), each owning a static share of the
    rows of every matrix of the step; a step ends when every share is done."""
    sec, nw = pool_time("decode", n_steps)
    return {"value": STEP_WEIGHT_BYTES / sec / 1e9, "unit": "GB/s", "cores": nw, "kind": "oracle",
            "sample": f"{n_steps} full decode steps (batch 1, W4A8), the rows of every matrix split statically "
                      f"over {nw} processes, {sec * n_steps:.1f} s"}


def cpu_baseline_kquant():
    """The oracle, single-threaded, on each K-quant decode shape (a row slice of
    about 8 MB of each matrix, one vector of Q8_K activations)."""
    from oracle import oracle as O
    shapes = [(Q4_K, 4096, 4096), (Q4_K, 1024, 4096), (Q4_K, 14336, 4096), (Q4_K, 4096, 14336),
              (Q6_K, 128256, 4096)]
    tot_b = tot_s = 0.0
    for t, rows, cols in shapes:
        rb = row_bytes(t, cols)
        nr = min(rows, max(1, 8_000_000 // rb))
        W = synth.weights(t, nr, cols, seed=7)
        xq = O.quantize_act(O.Q8_K, synth.activations(1, cols, seed=8))
        gbs, dt, n = oracle_rate(lambda: O.matvec(t, O.Q8_K, W, nr, cols, xq, 1, want_abs=False), nr * rb, 0.5)
        tot_b += nr * rb * n
        tot_s += dt
    return {"value": tot_b / tot_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"a ~8 MB row slice of each of the five shapes, 1 vector, single-threaded C oracle, "
                      f"{tot_s:.1f} s"}


def cpu_baseline_prefill():
    """The oracle on the 14336x4096 prefill restricted to a 64-token slice:
    single-threaded on 256 rows of it, and on every host core over all rows.
    TFLOP/s counts 2 flops per multiply-add of the definition."""
    from oracle import oracle as O
    rows, cols, m = PREFILL_CPU
    W, xb, xq = _prefill_workload(O)
    rb = row_bytes(Q4_K, cols)
    out = {}
    for name, at, xin in (("bf16", O.BF16, xb), ("w4a8", O.Q8_K, xq)):
        nr = 256
        Ws = W[:nr * rb]
        _, dt, n = oracle_rate(lambda: O.matvec(O.Q4_K, at, Ws, nr, cols, xin, m, want_abs=False), 1, 1.0)
        one = {"value": 2.0 * m * nr * cols * n / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": f"{m} tokens x {nr} rows of 14336x4096 Q4_K ({name}), {n} calls, {dt:.1f} s"}
        try:
            sec, nw = pool_time("prefill_" + name, 1)
            allc = {"value": 2.0 * m * rows * cols / sec / 1e12, "unit": "TFLOP/s", "cores": nw, "kind": "oracle",
                    "sample": f"{m} tokens x all 14336 rows ({name}), rows split over {nw} processes, "
                              f"{sec:.2f} s per pass"}
        except Exception as e:   # an auxiliary measurement: report it, keep the line
            allc = {"error": f"{type(e).__name__}: {e}"}
        out[name] = {"single_core": one, "all_cores": allc}
    return out


def cpu_baseline_moe():
    """The oracle's W4A8 MoE layer (gate_up + down, gpt-oss shapes): one token
    single-threaded, and 64 tokens on every host core (tokens split)."""
    from oracle import oracle as O
    wl = _moe_workload(O, MOE_CPU_TOKENS)
    ids = wl[4]
    per_tok_bytes = (5760 + 2880) * synth.row_bytes(MXFP4, 2880) * 4   # four routed experts per token
    _, dt, n = oracle_rate(lambda: _moe_tokens(O, wl, 0, 1), 1, 1.0)
    one = {"value": per_tok_bytes * n / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "ms_per_layer": 1e3 * dt / n,
           "sample": f"1 token (4 experts, {per_tok_bytes / 1e6:.1f} MB of expert weights), {n} calls, {dt:.1f} s"}
    try:
        sec, nw = pool_time("moe", 1)
        used = len(np.unique(ids)) * (5760 + 2880) * synth.row_bytes(MXFP4, 2880)
        allc = {"value": used / sec / 1e9, "unit": "GB/s (distinct expert bytes)", "cores": nw, "kind": "oracle",
                "ms_per_layer": 1e3 * sec,
                "sample": f"{MOE_CPU_TOKENS} tokens split over {nw} processes, {sec:.2f} s per layer"}
    except Exception as e:
        allc = {"error": f"{type(e).__name__}: {e}"}
    return {"tok1_single_core": one, "tok64_all_cores": allc}


def run_reference(args):
    """The oracle on the bench's workload, on the host cores, single-threaded.
    The decode step is a list of work items (every matrix in step order, the
    lm_head in row slices of ~8 MB); each timed step takes whole items from a
    cursor that runs round the list, as many as fit the step's time share,
    so that warm-up and timed steps take about 150 s together and, over the
    run, the items cover the step's mix of formats and shapes.  The rate is
    the weight bytes done over the time taken."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import oracle as O
    mats, xs = _oracle_step_workload()
    items = _oracle_work_items(mats)
    per_step = 150.0 / (args.steps + args.warmup)
    t_cal, b_cal = _oracle_items(O, mats, xs, items[:8])
    # bytes per step: 70% of the time share, since a step ends on a whole item
    budget = max(1, int(0.7 * per_step * b_cal / max(t_cal, 1e-9)))
    cursor = 0

    def take():
        nonlocal cursor
        out, nb = [], 0
        while True:
            k, r0, r1 = items[cursor % len(items)]
            out.append(items[cursor % len(items)])
            cursor += 1
            nb += (r1 - r0) * row_bytes(mats[k][4], mats[k][2])
            if nb >= budget or len(out) >= len(items):
                return out
    for _ in range(args.warmup):
        _oracle_items(O, mats, xs, take())
    secs = nbytes = 0.0
    for _ in range(args.steps):
        dt, nb = _oracle_items(O, mats, xs, take())
        secs += dt
        nbytes += nb
    value = nbytes / secs / 1e9
    ms = 1e3 * STEP_WEIGHT_BYTES / (value * 1e9)   # the time of a whole step at that rate
    sample = (f"{nbytes / args.steps / 1e6:.1f} MB of the decode step's weights per timed step "
              f"({1e3 * secs / args.steps:.1f} ms): whole matrices in step order from a rotating cursor, "
              f"the lm_head in ~8 MB row slices; single-threaded C oracle")
    line = {"impl": "reference", "metric": "quant GEMV weight GB/s (decode step, W4A8)", "value": value,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "q5_0/q8_0 weights x int8 activations (dp4a int32, fp32 accumulate)",
            "data": "synthetic",
            "config": {"workload": "qwen2.5-0.5b-shaped decode step (24 layers Q5_0 + lm_head Q8_0), batch 1",
                       "l2": "weights 390.6 MB, streamed from host memory"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the prefill and MoE legs")
    ap.add_argument("--probe", default=None, help="run one kernel for profiling (see run_probe)")
    args = ap.parse_args()
    if args.probe:
        return run_probe(args.probe)
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import gguf_block_quantised_gb300 as q
    from gguf_block_quantised_gb300 import build as B

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or ws == 1:
        B.build()
    if ws > 1:
        torch.distributed.barrier()
    q.load()
    stream = torch.cuda.Stream()

    # --- the step at batch 1 (the headline) and batch 8; the two-launch form and A32 for comparison
    step1 = DecodeStep(q, torch, 1)
    lm_ms_first, _ = lm_roofline(q, torch, stream, step1, local)
    step8 = DecodeStep(q, torch, 8)
    step1u = DecodeStep(q, torch, 1, fused=False)
    step1f = DecodeStep(q, torch, 1, a32=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms1, clocks = time_graph(torch, step1.run, stream, args.steps, args.warmup, sampler_index=local)
    ms8, _ = time_graph(torch, step8.run, stream, max(args.steps // 4, 10), args.warmup)
    ms1u, _ = time_graph(torch, step1u.run, stream, max(args.steps // 4, 10), args.warmup)
    ms1f, _ = time_graph(torch, step1f.run, stream, max(args.steps // 4, 10), args.warmup)
    q.qmv_get_status(stream)
    ms1, ms8 = max_over_ranks(torch, [ms1, ms8], "cuda")
    del step1u, step1f

    # --- the dominant kernel (the Q5_0 layer matvecs, as launched in the step) and the lm_head
    hbm, peak_kind = load_peaks()
    layer_ms, layer_clocks = layer_roofline(torch, stream, step1, local)
    layer_bytes = LAYER_BYTES_PER_STEP / LAYER_LAUNCHES_PER_STEP
    layer_gbs = layer_bytes / (layer_ms / 1e3) / 1e9
    shapes = layer_shapes_leg(q, torch, stream, step1, hbm)
    lm_ms, lm_clocks = lm_roofline(q, torch, stream, step1, local)
    lm_ms_nopdl, _ = lm_roofline(q, torch, stream, step1, local, pdl=False)
    lm_bytes = VOCAB * row_bytes(Q8_0, HID)
    lm_gbs = lm_bytes / (lm_ms / 1e3) / 1e9

    # --- end to end through host buffers: pinned activations in, logits out, per step
    host_x = torch.from_numpy(step1.x_host_all).pin_memory()   # the step's 97 activation vectors, contiguous
    host_logits = torch.empty((1, VOCAB), dtype=torch.float32).pin_memory()
    h2d = host_x.numel() * 4
    d2h = host_logits.numel() * 4

    def e2e_step(s):
        with torch.cuda.stream(s):
            step1.x_all.copy_(host_x, non_blocking=True)
            step1.run(s)
            host_logits.copy_(step1.logits, non_blocking=True)
    e2e_steps = max(args.steps // 4, 10)
    e2e_ms, _ = time_graph(torch, e2e_step, stream, e2e_steps, args.warmup)

    tflops_peak = 1900.0 if peak_kind == "fallback" else load_tflops_peak()
    cfg1 = None if args.no_extra else config1_leg(q, torch, stream, hbm)
    kquant = None if args.no_extra else kquant_decode_leg(q, torch, stream, hbm)
    formats = None if args.no_extra else formats_leg(q, torch, stream, hbm)
    prefill = None if args.no_extra else prefill_leg(q, torch, stream, tflops_peak)
    moe = None if args.no_extra else moe_leg(q, torch, stream, hbm, tflops_peak)
    wquant = None if args.no_extra else wquant_leg(q, torch, stream, hbm)
    value = ws * STEP_WEIGHT_BYTES / (ms1 / 1e3) / 1e9
    if rank != 0:
        if ws > 1:
            torch.distributed.barrier()
        return 0
    cpu = cpu_all = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(4)
        try:
            cpu_all = cpu_baseline_all_cores()
        except Exception as e:   # an auxiliary measurement: report it, keep the line
            cpu_all = {"error": f"{type(e).__name__}: {e}"}
        if kquant is not None:
            kquant["cpu_baseline"] = cpu_baseline_kquant()
        if prefill is not None:
            prefill["cpu_baseline"] = cpu_baseline_prefill()
        if moe is not None:
            moe["cpu_baseline"] = cpu_baseline_moe()
    line = {
        "metric": "quant GEMV weight GB/s (decode step, W4A8)",
        "value": value,
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms1,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q5_0/q8_0 weights x int8 activations (dp4a int32, fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": "qwen2.5-0.5b-shaped decode step (24 layers q/k/v/o/gate/up/down Q5_0, stored as "
                               "q|k|v, o, gate|up, down stacks, + lm_head 151936x896 Q8_0; fp32 activations "
                               "quantised to Q8_0 inside each matvec), batch 1",
                   "launches_per_step": step1.launches,
                   "weight_bytes_per_step": STEP_WEIGHT_BYTES, "parallelism": f"replicas x{ws}",
                   "l2": "weights 390.6 MB > 129 MB L2, streamed cold every step (no flush needed)",
                   "graph": "step captured once as a CUDA graph and replayed"},
        "frac_of_hbm": value / ws / hbm,
        "batch8": {"ms_per_step": ms8, "value": ws * STEP_WEIGHT_BYTES / (ms8 / 1e3) / 1e9, "unit": "GB/s",
                   "vector_rate_tok_s": ws * 8 / (ms8 / 1e3)},
        "a32_batch1": {"ms_per_step": ms1f, "value": ws * STEP_WEIGHT_BYTES / (ms1f / 1e3) / 1e9, "unit": "GB/s",
                       "how": "fp32 activations straight into every matvec (QMV_FMT(Q5_0|Q8_0, F32)), PDL chain"},
        "unfused_batch1": {"ms_per_step": ms1u, "value": ws * STEP_WEIGHT_BYTES / (ms1u / 1e3) / 1e9,
                           "unit": "GB/s", "launches_per_step": step1.launches * 2,
                           "how": "qmv_quantize_act + qmv_matvec as separate launches, no PDL"},
        "roofline": {"bound": "hbm",
                     "kernel": "k_gemv<Q5_0,A8,NV=1> -- the step's 96 layer matvecs (q|k|v 1152x896, o 896x896, "
                               "gate|up 9728x896, down 896x4864 per layer), launched as in the step (each quantising "
                               "its fp32 input, a programmatic dependent of the one before); ~95% of the step's "
                               "launch time",
                     "achieved": layer_gbs, "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": layer_gbs / hbm, "traffic": traffic_for("k_gemv<Q5_0,A8,NV=1> qwen layer matvecs"),
                     "algorithmic_bytes_per_launch": layer_bytes, "launch_ms": layer_ms,
                     "units": "weight bytes of the block format (Q5_0: 0.6875 B per weight) x rows x cols, "
                              "averaged over the 96 launches (246,005,760 B per step)",
                     "clocks": layer_clocks, "by_shape": shapes,
                     "l2": "the 246 MB of layer weights exceed L2; every pass streams them"},
        "lm_head": {"kernel": "k_gemv<Q8_0,A8,NV=1> lm_head 151936x896 (quantising its fp32 input; PDL)",
                    "achieved": lm_gbs, "unit": "GB/s", "frac": lm_gbs / hbm, "launch_ms": lm_ms,
                    "algorithmic_bytes_per_launch": lm_bytes,
                    "traffic": traffic_for("k_gemv<Q8_0,A8,NV=1> lm_head 151936x896"),
                    "launch_ms_plain_launches": lm_ms_nopdl,
                    "achieved_plain_launches": lm_bytes / (lm_ms_nopdl / 1e3) / 1e9,
                    "launch_ms_before_step_graphs": lm_ms_first, "clocks": lm_clocks,
                    "l2": "4 weight copies rotated, each launch reads cold"},
        "clocks": clocks,
        "e2e": {"value": ws * STEP_WEIGHT_BYTES / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "the step's pinned host activations copied in (one copy) and the logits copied out every "
                       "step, all in one replayed CUDA graph on the caller's stream"},
        "gpu_launches": step1.launches * args.steps,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "config1_q4_0_896": cfg1,
        "kquant_decode": kquant,
        "formats": formats,
        "prefill": prefill,
        "moe": moe,
        "weight_quantiser": wquant,
    }
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.barrier()
    return 0


if __name__ == "__main__":
    sys.exit(main())
