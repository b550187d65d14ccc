#!/usr/bin/env python3
"""Benchmark of the IHA attention-layer hot path on GB300.

One step = one pass of every hot-path operation over one batch of seeded
synthetic inputs, each at its workload's shape:
  premix     LLaMA-2.4B layer shape B=1, N=8192, H=20, P=4, d=128: forward
             for Q and K (fused RoPE, base 10000) and V in one launch; backward (input
             gradient, inverse RoPE for Q and K, and weight gradient from the
             same pass over dY) for Q, K, V;
  attention  80 pseudo-heads, N=4096, d=128, causal window W=1024, fp32 LSE,
             and its backward (dQ, dK, dV for an upstream gradient dO);
  Hiera      MAE stage 1, B=128, 56x56 tokens, 8x8 units, 20 kept, C=d=96:
             gather, attention inside each unit, scatter;
  long ctx   the long-context IHA layer forward, B=2, N=16384, H=20, P=4,
             d=128: premix Q and K with RoPE and V (one launch), then causal attention over
             the 80 pseudo-heads on those premix outputs (fp32 LSE).
The step's working set (~5 GB) is far larger than L2 (129 MB), so no L2
flush is needed between steps: every op's inputs were evicted by the others.
The tiny fp32 layer (B=1, N=128, H=4, P=2, d=32: premix Q, K, V and unmasked
attention) is latency-bound; its time per layer is reported separately.

Metric: every op has an algorithmic roofline time, max(bytes / HBM peak,
flops / bf16 peak) with the measured peaks (burst: the timed region lasts
well under a second); the step's efficiency is the sum of those times over
the measured step time.  `value` is that efficiency in % summed over GPUs (it
adds up across replicas; at N=1 it is the efficiency).  Per-op GB/s, TFLOP/s
and roofline fractions are in `ops`.

--impl reference times the oracle (CPU) on a bounded random sample of the
same step and scales it to the whole step; it is a deliberately slow
baseline, not a target.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as S  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
METRIC = "premix+gather GB/s and attention TFLOP/s at 1 GB300, as % of roofline"
UNIT = "% of 1-GPU roofline, summed over GPUs"
# Fraction of every op the oracle runs per CPU sample (same in both CPU legs).
CPU_FRAC = 1 / 256

# DRAM bytes (read + write) per launch of the dominant kernel, from a one-pass
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of the full-size
# launch; removed whenever that kernel changes, until it is captured again.
NCU_TRAFFIC: dict = {}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- workload
def _attn_pairs(N: int, mask: str, W: int = 0) -> int:
    """Visible (query, key) pairs of one head."""
    if mask == "causal":
        return N * (N + 1) // 2
    return sum(min(i + 1, W) for i in range(N))


def max_over_ranks(x: float, world: int, device) -> float:
    """The job's time: the largest x over the ranks (x itself at world 1).
    Every rank runs the same replica of the step, so the job processed
    world x one step's work in that time."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(ideal_step_s: float, step_ms: float, world: int) -> float:
    """`value`: % of the 1-GPU roofline summed over the replicas."""
    return round(100.0 * ideal_step_s / (step_ms * 1e-3) * world, 3)


def op_table():
    """(name, bytes, flops) per op of one step, algorithmic (inputs read once,
    outputs written once)."""
    ops = []
    pm = S.LLAMA_PREMIX
    tok = pm.B * pm.N
    x_b, y_b, w_b = tok * pm.H * pm.d * 2, tok * pm.HP * pm.d * 2, pm.HP * pm.H * 4
    pf = 2 * tok * pm.HP * pm.H * pm.d
    ops.append(("premix_fwd_qkv", 3 * (x_b + y_b + w_b), 3 * pf))
    # dX and dW of Q, K and V in one launch, each from one read of dY and X
    ops.append(("premix_bwd_qkv", 3 * (y_b + 2 * x_b + 2 * w_b), 3 * 2 * pf))
    aw = S.LLAMA_WINDOW
    attn_fl = 4 * aw.d * _attn_pairs(aw.N, "window", S.WINDOW_KEYS) * aw.HP * aw.B
    tens = aw.B * aw.N * aw.HP * aw.d * 2
    ops.append(("attention_window", 4 * tens + aw.B * aw.HP * aw.N * 4, attn_fl))
    # backward: Q, K, V, O, dO and lse in, dQ, dK, dV out; five GEMMs to two
    ops.append(("attention_window_bwd", 8 * tens + aw.B * aw.HP * aw.N * 4, attn_fl * 5 // 2))
    mu = S.HIERA_MU
    kept = mu.B * mu.n_keep * mu.unit_tokens * mu.C * 2
    ops.append(("mu_gather", 2 * kept + mu.B * mu.n_keep * 4, 0))
    ops.append(("mu_attention", 4 * kept,
                4 * mu.C * mu.unit_tokens * mu.unit_tokens * mu.B * mu.n_keep))
    ops.append(("mu_scatter", 2 * kept + mu.B * mu.n_keep * 4, 0))
    lc = S.LONG_CTX
    tok = lc.B * lc.N
    x_b, y_b = tok * lc.H * lc.d * 2, tok * lc.HP * lc.d * 2
    pf = 2 * tok * lc.HP * lc.H * lc.d
    ops.append(("long_premix_fwd_qkv", 3 * (x_b + y_b + w_b), 3 * pf))
    ops.append(("long_attention_causal", 4 * y_b + lc.B * lc.HP * lc.N * 4,
                4 * lc.d * _attn_pairs(lc.N, "causal") * lc.HP * lc.B))
    return ops


def launches_per_step() -> int:
    # premix fwd (Q, K, V in one launch); premix bwd (zero the three dW + one
    # kernel for Q, K, V); window attention; its backward (preprocess, kernel,
    # postprocess); gather, MU attention, scatter; long-context premix (one
    # launch) + attention
    return 1 + 2 + 1 + 3 + 3 + 1 + 1


def _input_recipes(seed: int):
    """Generator of every synthetic input of the step, by name."""
    pm, aw, mu, lc = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU, S.LONG_CTX
    r = {}
    for c, t in enumerate("qkv"):
        r[f"x_{t}"] = lambda c=c: S.normal((pm.B, pm.N, pm.H, pm.d), seed, 10 + c)
        r[f"w_{t}"] = lambda c=c: S.premix_weight(pm.H, pm.P, seed, 20 + c)
        r[f"dy_{t}"] = lambda c=c: S.normal((pm.B, pm.N, pm.HP, pm.d), seed, 30 + c)
        r[f"a_{t}"] = lambda c=c: S.normal((aw.B, aw.N, aw.HP, aw.d), seed, 40 + c)
        r[f"lx_{t}"] = lambda c=c: S.normal((lc.B, lc.N, lc.H, lc.d), seed, 60 + c)
        r[f"lw_{t}"] = lambda c=c: S.premix_weight(lc.H, lc.P, seed, 70 + c)
    r["a_do"] = lambda: S.normal((aw.B, aw.N, aw.HP, aw.d), seed, 43)
    r["mu_x"] = lambda: S.normal((mu.B, mu.grid_h * mu.grid_w, mu.C), seed, 50)
    r["mu_keep"] = lambda: S.keep_units(mu.B, mu.n_units, mu.n_keep, seed)
    return r


def host_inputs(seed: int, keys=None):
    rec = _input_recipes(seed)
    return {k: rec[k]() for k in (keys if keys is not None else rec)}


# inputs each op of the step reads (directly or through the op that feeds it)
OP_INPUTS = {
    "premix_fwd_qkv": [f"{a}_{t}" for t in "qkv" for a in "xw"],
    "premix_bwd_qkv": [f"{a}_{t}" for t in "qkv" for a in ("dy", "x", "w")],
    "attention_window": ["a_q", "a_k", "a_v"],
    "attention_window_bwd": ["a_q", "a_k", "a_v", "a_do"],
    "mu_gather": ["mu_x", "mu_keep"],
    "mu_attention": ["mu_x", "mu_keep"],
    "mu_scatter": ["mu_x", "mu_keep"],
    "mu_attention_fused": ["mu_x", "mu_keep"],
    "long_premix_fwd_qkv": [f"l{a}_{t}" for t in "qkv" for a in "xw"],
    "long_attention_causal": [f"l{a}_{t}" for t in "qkv" for a in "xw"],
    "mu_attention_qpool": [],   # generated on the device (see qpool_case)
}


# --------------------------------------------------------------------------- GPU arm
def host_tensor(a: np.ndarray, torch):
    """CPU torch tensor of a synthetic array (uint16 arrays are bf16 bit patterns)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def gpu_id(torch, device) -> str:
    """nvidia-smi id of the device (its UUID when torch exposes it)."""
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device.index or 0)


class Step:
    """Device buffers and the launch sequence of one step (every op through the
    package's public calls)."""

    def __init__(self, T, torch, dev_inputs, device):
        pm, aw, mu, lc = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU, S.LONG_CTX
        self.T, self.torch = T, torch
        self.i = dev_inputs
        e = lambda shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt, device=device)
        self.y = {t: e((pm.B, pm.N, pm.HP, pm.d)) for t in "qkv"}
        self.dx = {t: e((pm.B, pm.N, pm.H, pm.d)) for t in "qkv"}
        self.dw = {t: e((pm.H, pm.P, pm.H), torch.float32) for t in "qkv"}
        self.o = e((aw.B, aw.N, aw.HP, aw.d))
        self.lse = e((aw.B, 1, aw.HP, aw.N), torch.float32)
        self.agrad = {t: e((aw.B, aw.N, aw.HP, aw.d)) for t in "qkv"}
        self.ws = torch.empty(T.mha_bwd_workspace_bytes(aw.B, aw.HP, aw.N, aw.d),
                              dtype=torch.uint8, device=device)
        self.g = e((mu.B, mu.n_keep, mu.unit_tokens, mu.C))
        self.ou = e((mu.B, mu.n_keep, mu.unit_tokens, mu.C))
        self.dec = torch.zeros((mu.B, mu.grid_h * mu.grid_w, mu.C), dtype=torch.bfloat16,
                               device=device)
        self.ly = {t: e((lc.B, lc.N, lc.HP, lc.d)) for t in "qkv"}
        self.lo = e((lc.B, lc.N, lc.HP, lc.d))
        self.llse = e((lc.B, 1, lc.HP, lc.N), torch.float32)

    def results(self):
        """What a caller reads back: every op's final output (the long-context
        premix outputs are intermediates consumed by its attention)."""
        return ([self.y[t] for t in "qkv"] + [self.dx[t] for t in "qkv"] +
                [self.dw[t] for t in "qkv"] + [self.o, self.lse] +
                [self.agrad[t] for t in "qkv"] + [self.dec, self.lo, self.llse])

    def run(self, marks=None):
        """Enqueue the step; `marks(k)` records an event before op 0 and after op k-1."""
        T, i = self.T, self.i
        pm, aw, mu, lc = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU, S.LONG_CTX
        mark = marks or (lambda k: None)
        k = 0
        mark(k)

        def done():
            nonlocal k
            k += 1
            mark(k)

        T.premix_fwd_qkv([i[f"x_{t}"] for t in "qkv"], [i[f"w_{t}"] for t in "qkv"], pm.P,
                         rope=True, rope_base=S.ROPE_BASE, out=tuple(self.y[t] for t in "qkv"))
        done()
        T.premix_bwd_qkv([i[f"dy_{t}"] for t in "qkv"], [i[f"x_{t}"] for t in "qkv"],
                         [i[f"w_{t}"] for t in "qkv"], rope=True, rope_base=S.ROPE_BASE,
                         dxs=tuple(self.dx[t] for t in "qkv"), dws=tuple(self.dw[t] for t in "qkv"))
        done()
        T.mha_fwd(i["a_q"], i["a_k"], i["a_v"], mask=T.MASK_CAUSAL_WINDOW, window=S.WINDOW_KEYS,
                  out=self.o, lse=self.lse)
        done()
        T.mha_bwd(i["a_q"], i["a_k"], i["a_v"], self.o, i["a_do"], self.lse,
                  mask=T.MASK_CAUSAL_WINDOW, window=S.WINDOW_KEYS, dq=self.agrad["q"],
                  dk=self.agrad["k"], dv=self.agrad["v"], workspace=self.ws)
        done()
        T.mu_gather(i["mu_x"], i["mu_keep"], mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w, out=self.g)
        done()
        u = self.g.view(mu.B * mu.n_keep, 1, mu.unit_tokens, 1, mu.C)
        T.mha_fwd(u, u, u, out=self.ou.view(mu.B * mu.n_keep, 1, mu.unit_tokens, 1, mu.C))
        done()
        T.mu_scatter(self.ou, i["mu_keep"], self.dec, mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w)
        done()
        T.premix_fwd_qkv([i[f"lx_{t}"] for t in "qkv"], [i[f"lw_{t}"] for t in "qkv"], lc.P,
                         rope=True, rope_base=S.ROPE_BASE, out=tuple(self.ly[t] for t in "qkv"))
        done()
        T.mha_fwd(self.ly["q"], self.ly["k"], self.ly["v"], mask=T.MASK_CAUSAL, out=self.lo,
                  lse=self.llse)
        done()


def qpool_case(T, torch, device):
    """The Hiera stage-2 pooling block: (enqueue function, algorithmic bytes,
    flops).  qkv (seeded, on the device) is read in place in Hiera's
    [B, T, units, 3, heads, head_dim] layout and O written in its
    [B, Tq, units, heads, head_dim] layout; the queries are max-pooled 4:1
    inside the kernel."""
    hq = S.HIERA_QPOOL
    gen = torch.Generator(device=device)
    gen.manual_seed(7)
    qkv = torch.randn((hq.B, hq.T, hq.n_units, 3, hq.heads, hq.head_dim), generator=gen,
                      device=device).to(torch.bfloat16)
    qv, kv, vv = (qkv[:, :, :, c].permute(0, 2, 1, 3, 4) for c in range(3))
    dst = torch.empty((hq.B, hq.Tq, hq.n_units, hq.heads, hq.head_dim), dtype=torch.bfloat16,
                      device=device)
    run = lambda: T.mha_fwd_qpool(qv, kv, vv, hq.q_stride, out=dst.permute(0, 2, 1, 3, 4))
    units = hq.B * hq.n_units * hq.heads
    nbytes = units * (3 * hq.T + hq.Tq) * hq.head_dim * 2
    flops = 4 * hq.head_dim * hq.Tq * hq.T * units
    return run, nbytes, flops


def extra_ops(T, torch, dev, step, device, iters: int, hbm: float, tc: float):
    """Ops beyond the step's rows, timed alone after it (not part of `value`):
    the fused gather -> mask-unit attention -> scatter of the Hiera stage-1
    step, against its own algorithmic bytes (kept tokens read once from x and
    written once to the canvas)."""
    mu = S.HIERA_MU
    kept = mu.B * mu.n_keep * mu.unit_tokens * mu.C * 2
    nbytes = 2 * kept + mu.B * mu.n_keep * 4
    flops = 4 * mu.C * mu.unit_tokens * mu.unit_tokens * mu.B * mu.n_keep
    canvas = torch.zeros_like(dev["mu_x"])
    run = lambda: T.mu_attention_fused(dev["mu_x"], dev["mu_keep"], canvas, mu.grid_h, mu.grid_w,
                                       mu.mu_h, mu.mu_w)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # > L2 between launches
    for _ in range(3):
        run()
    ts = []
    for _ in range(max(iters, 3)):
        flush.fill_(0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize(device)
        ts.append(e0.elapsed_time(e1))
    ms = statistics.median(ts)
    ideal = max(nbytes / hbm, flops / tc)
    out = {"mu_attention_fused": {
        "ms": round(ms, 5), "roofline_ms": round(ideal * 1e3, 5),
        "frac": round(ideal / (ms * 1e-3), 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "bound": "hbm", "l2": "256 MB written between launches",
        "replaces": "mu_gather + mu_attention + mu_scatter (one pass, no gathered copy in HBM)"}}
    # Hiera stage-2 pooling block: mask-unit attention with the queries
    # max-pooled 4:1 inside the kernel, on qkv read in place in Hiera's
    # [B, T, units, 3, heads, head_dim] layout and O written in its
    # [B, Tq, units, heads, head_dim] layout
    hq = S.HIERA_QPOOL
    runq, qbytes, qflops = qpool_case(T, torch, device)
    for _ in range(3):
        runq()
    ts = []
    for _ in range(max(iters, 3)):
        flush.fill_(0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        runq()
        e1.record()
        torch.cuda.synchronize(device)
        ts.append(e0.elapsed_time(e1))
    ms = statistics.median(ts)
    ideal = max(qbytes / hbm, qflops / tc)
    out["mu_attention_qpool"] = {
        "config": f"Hiera stage-2 pooling block: B={hq.B}, {hq.n_units} units, T={hq.T} -> "
                  f"Tq={hq.Tq} (q_stride {hq.q_stride}), {hq.heads} heads of {hq.head_dim}",
        "ms": round(ms, 5), "roofline_ms": round(ideal * 1e3, 5),
        "frac": round(ideal / (ms * 1e-3), 4), "GB/s": round(qbytes / (ms * 1e-3) / 1e9, 1),
        "bound": "hbm", "l2": "256 MB written between launches"}
    del canvas, flush, runq
    # joint-softmax variant of the layer forward at the LLaMA shape: premix Q,
    # K (RoPE), V into the interleaved layout, then causal attention of the 20
    # heads over the N*P = 32768 pseudo-tokens
    pm = S.LLAMA_PREMIX
    ys = tuple(torch.empty((pm.B, pm.N, pm.P, pm.H, pm.d), dtype=torch.bfloat16, device=device)
               for _ in range(3))
    o = torch.empty((pm.B, pm.N * pm.P, pm.H, pm.d), dtype=torch.bfloat16, device=device)
    M = pm.N * pm.P
    pre = lambda: T.premix_fwd_qkv_interleaved([dev[f"x_{t}"] for t in "qkv"],
                                               [dev[f"w_{t}"] for t in "qkv"], pm.P, rope=True,
                                               rope_base=S.ROPE_BASE, out=ys)
    att = lambda: T.mha_fwd(*(y.view(pm.B, M, pm.H, pm.d) for y in ys), mask=T.MASK_CAUSAL,
                            out=o)
    for _ in range(2):
        pre()
        att()
    tp, ta = [], []
    for _ in range(max(iters // 2, 3)):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        pre()
        e[1].record()
        att()
        e[2].record()
        torch.cuda.synchronize(device)
        tp.append(e[0].elapsed_time(e[1]))
        ta.append(e[1].elapsed_time(e[2]))
    mp, ma = statistics.median(tp), statistics.median(ta)
    tok = pm.B * pm.N
    pbytes = 3 * (tok * pm.H * pm.d * 2 + tok * pm.HP * pm.d * 2 + pm.HP * pm.H * 4)
    aflops = 4 * pm.d * (M * (M + 1) // 2) * pm.H * pm.B
    out["iha_joint_softmax_layer"] = {
        "config": "B=1, N=8192, H=20, P=4, d=128: premix Q,K(+RoPE),V -> [B,N,P,H,d]; causal "
                  "attention of 20 heads over N*P=32768 pseudo-tokens",
        "premix_ms": round(mp, 5), "premix_GB/s": round(pbytes / (mp * 1e-3) / 1e9, 1),
        "premix_frac": round(pbytes / hbm / (mp * 1e-3), 4),
        "attention_ms": round(ma, 5), "attention_TFLOP/s": round(aflops / (ma * 1e-3) / 1e12, 1),
        "attention_frac": round(aflops / tc / (ma * 1e-3), 4)}
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def tiny_layer_latency(T, torch, device, iters: int = 50):
    """Tiny fp32 IHA layer forward (premix Q, K, V into 8 pseudo-heads in one
    launch, then unmasked attention): microseconds per layer, CUDA events.
    Its two kernels take a few microseconds each, so issued one call at a time the
    layer waits on the host; the layer is captured once in a CUDA graph and
    replayed (`us_per_layer`), and the eager time is reported beside it."""
    sh = S.TINY
    xs = [host_tensor(S.normal((sh.B, sh.N, sh.H, sh.d), 0, c, dtype="f32"), torch).to(device)
          for c in range(3)]
    ws = [host_tensor(S.premix_weight(sh.H, sh.P, 0, 10 + c), torch).to(device) for c in range(3)]
    ys = tuple(torch.empty((sh.B, sh.N, sh.HP, sh.d), dtype=torch.float32, device=device)
               for _ in range(3))
    o = torch.empty_like(ys[0])

    def layer():
        T.premix_fwd_qkv(xs, ws, sh.P, out=ys)
        T.mha_fwd(*ys, out=o)

    def timed(run):
        stream = torch.cuda.current_stream(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(stream)
        for _ in range(iters):
            run()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / iters

    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for _ in range(5):
            layer()
    torch.cuda.current_stream(device).wait_stream(side)
    eager = timed(layer)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()
    graph.replay()
    torch.cuda.synchronize(device)
    replay = timed(graph.replay)
    return {"us_per_layer": round(replay, 2), "us_per_layer_eager": round(eager, 2),
            "launches": 2, "how": "CUDA graph of the layer replayed (eager: one call at a time)",
            "config": "B=1, N=128, H=4, P=2, d=32, fp32, unmasked"}


def gpu_arm(args, rank, world, local_rank):
    import torch
    import transformer_attention_iha_gb300 as T
    T.build()
    T.lib()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12   # burst: the timed region is well under a second

    host = host_inputs(seed=rank)
    hostt = {k: host_tensor(v, torch) for k, v in host.items()}
    del host
    dev = {k: v.to(device) for k, v in hostt.items()}
    step = Step(T, torch, dev, device)
    stream = torch.cuda.current_stream(device)
    ops = op_table()
    nops = len(ops)

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize(device)
    if T.device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)]
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id(torch, device))
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    start.record(stream)
    for s in range(args.steps):
        step.run(lambda k, s=s: evs[s][k].record(stream))
    end.record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(start.elapsed_time(end), world, device)
    ms_step = total_ms / args.steps
    op_ms = [statistics.mean(evs[s][k].elapsed_time(evs[s][k + 1]) for s in range(args.steps))
             for k in range(nops)]
    derr = T.device_error()

    op_out, ideal_total = {}, 0.0
    for (name, nbytes, flops), ms in zip(ops, op_ms):
        t_hbm, t_tc = nbytes / hbm, (flops / tc if flops else 0.0)
        ideal = max(t_hbm, t_tc)
        ideal_total += ideal
        rec = {"ms": round(ms, 5), "roofline_ms": round(ideal * 1e3, 5),
               "frac": round(ideal / (ms * 1e-3), 4),
               "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
               "bound": "tensor" if t_tc > t_hbm else "hbm"}
        if flops:
            rec["TFLOP/s"] = round(flops / (ms * 1e-3) / 1e12, 1)
        op_out[name] = rec

    # dominant kernel by time share
    dom = max(range(nops), key=lambda k: op_ms[k])
    dname, dbytes, dflops = ops[dom]
    dsec = op_ms[dom] * 1e-3
    if op_out[dname]["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": round(dflops / dsec / 1e12, 1),
                "peak": round(tc / 1e12, 1), "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(dbytes / dsec / 1e9, 1),
                "peak": round(hbm / 1e9, 1), "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = NCU_TRAFFIC.get(dname)
    roof["kernel"] = dname
    roof["share"] = round(op_ms[dom] / ms_step, 4)
    roof["peak_source"] = f"{peak_src} ({'bf16 burst' if roof['bound'] == 'tensor' else 'copy'})"

    tiny = tiny_layer_latency(T, torch, device)
    extras = extra_ops(T, torch, dev, step, device, args.steps, hbm, tc)

    # end to end: host buffers; every input copied in and every result read back per step
    e2e = None
    if args.e2e_steps > 0:
        # Every step copies its inputs in from pinned host memory and its
        # results back out.  Copies and compute run on their own streams over
        # two sets of device buffers, so step i + 1's inputs arrive (and step
        # i - 1's results leave) while step i computes, as a training loop
        # with prefetching would run it.
        pinned = {k: v.pin_memory() for k, v in hostt.items()}
        dev2 = {k: torch.empty_like(v) for k, v in dev.items()}
        steps2 = [step, Step(T, torch, dev2, device)]
        devs = [dev, dev2]
        res_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in step.results()]
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        d2h = sum(o.numel() * o.element_size() for o in res_host)
        s_in, s_run, s_out = (torch.cuda.Stream(device) for _ in range(3))
        ev = lambda: torch.cuda.Event()
        in_done, run_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(run_done[b])       # step i - 2 has read these inputs
                for k, v in pinned.items():
                    devs[b][k].copy_(v, non_blocking=True)
                in_done[b].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(in_done[b])
                if used[b]:
                    s_run.wait_event(out_done[b])      # step i - 2's results have left
                steps2[b].run()
                run_done[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(run_done[b])
                for o, h in zip(steps2[b].results(), res_host):
                    h.copy_(o, non_blocking=True)
                out_done[b].record(s_out)
            used[b] = True

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        e0.record(s_in)
        s_run.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(args.e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize(device)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, device)
        e2e = {"value": job_value(ideal_total, e2e_ms, world), "unit": UNIT,
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h)}

    line = {
        "metric": METRIC,
        "value": job_value(ideal_total, ms_step, world),
        "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, W ~ N(0,1/H) fp32)",
        "config": {"workload": "IHA hot-path step: premix fwd(+RoPE) and fused dX+dW for Q,K,V at "
                               "B=1,N=8192,H=20,P=4,d=128; causal-window attention 80 heads "
                               "N=4096 d=128 W=1024; Hiera-Base MAE stage-1 gather + mask-unit "
                               "attention (2560 units x 64 tokens, d=96) + scatter; long-context "
                               "layer B=2,N=16384: premix Q,K(+RoPE),V and causal attention over "
                               "80 pseudo-heads",
                   "l2": "no flush: step working set ~5 GB > 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "ops": op_out,
        "roofline": roof,
        "tiny_layer_fp32": tiny,
        "extras": extras,
        "e2e": e2e,
        "gpu_launches": launches_per_step() * args.steps,
        "clocks": clk,
        "device_error": derr,
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                  "source": peak_src},
    }
    return line


# --------------------------------------------------------------------------- CPU (oracle) arm
def oracle_sample(host, frac: float, seed: int = 0):
    """Time the oracle on a random `frac` of every op of one step and scale each
    op's time by its sampled share.  Returns (seconds per full step, measured
    seconds, sample description, threads)."""
    import oracle as O
    pm, aw, mu, lc = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU, S.LONG_CTX
    g = np.random.default_rng(seed)
    t_full = t_meas = 0.0

    def timed(fn, scale):
        nonlocal t_full, t_meas
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        t_meas += dt
        t_full += dt * scale

    def attn_rows(q, k, v, heads, N, B, mask, window, nrows):
        rows = np.stack([g.integers(0, B, nrows), np.zeros(nrows, np.int64),
                         g.integers(0, heads, nrows), g.integers(0, N, nrows)], axis=1)
        O.attention_rows(q[:, None], k[:, None], v[:, None], rows.astype(np.int64), mask, window)

    ntok = max(1, int(pm.N * frac))
    for t in "qkv":
        rope = t != "v"
        x, w, dy = host[f"x_{t}"][:, :ntok], host[f"w_{t}"], host[f"dy_{t}"][:, :ntok]
        timed(lambda: O.premix_fwd(x, w, pm.P, rope=rope, rope_base=S.ROPE_BASE), pm.N / ntok)
        timed(lambda: (O.premix_bwd_dx(dy, w, rope=rope, rope_base=S.ROPE_BASE),
                       O.premix_bwd_dw(dy, x, pm.P, rope=rope, rope_base=S.ROPE_BASE)),
              pm.N / ntok)
    n_all = aw.B * aw.N * aw.HP
    n = max(1, int(n_all * frac))
    timed(lambda: attn_rows(host["a_q"], host["a_k"], host["a_v"], aw.HP, aw.N, aw.B,
                            O.MASK_CAUSAL_WINDOW, S.WINDOW_KEYS, n), n_all / n)
    # backward: whole heads only (every key gathers over all its queries); one
    # head stands in for the HP heads of every batch
    h1 = [np.ascontiguousarray(host[nm][:1, :, :1]) for nm in ("a_q", "a_k", "a_v", "a_do")]
    timed(lambda: O.attention_bwd(*h1, O.MASK_CAUSAL_WINDOW, S.WINDOW_KEYS), aw.HP * aw.B)
    nb = max(1, int(mu.B * frac))
    x, keep = host["mu_x"][:nb], host["mu_keep"][:nb]

    def hiera():
        gg = O.mu_gather(x, keep, mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w)
        u = gg.reshape(nb * mu.n_keep, 1, mu.unit_tokens, 1, mu.C)
        ou, _ = O.attention(u, u, u)
        ob = S.f32_to_bf16_bits(ou.astype(np.float32)).reshape(nb, mu.n_keep, mu.unit_tokens,
                                                               mu.C)
        O.mu_scatter(ob, keep, np.zeros_like(x), mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w)

    timed(hiera, mu.B / nb)
    ntok = max(1, int(lc.N * frac))
    ys = {}
    for t in "qkv":
        x, w = host[f"lx_{t}"][:, :ntok], host[f"lw_{t}"]

        def fwd(t=t, x=x, w=w):
            ys[t] = O.premix_fwd(x, w, lc.P, rope=(t != "v"), rope_base=S.ROPE_BASE)

        timed(fwd, lc.N / ntok)
    # causal attention rows (independent; a row's cost depends only on its
    # position, so one head of full-length inputs stands in for all 80)
    n_all = lc.B * lc.N * lc.HP
    n = max(1, int(n_all * frac))
    qa, ka, va = (np.ascontiguousarray(host[f"lx_{t}"][:, :, :1]) for t in "qkv")
    timed(lambda: attn_rows(qa, ka, va, 1, lc.N, lc.B, O.MASK_CAUSAL, 0, n), n_all / n)
    desc = (f"random {frac:.5f} of every op: tokens of each premix, query rows of each attention "
            f"forward (uniform over batch, head, position), Hiera samples; one whole head of "
            f"the attention backward; each op's time scaled by its sampled share")
    return t_full, t_meas, desc, O.num_threads()


def ideal_step_seconds():
    peaks, _ = load_peaks()
    hbm, tc = peaks["hbm_gbs"] * 1e9, peaks["bf16_tflops"] * 1e12
    return sum(max(b / hbm, (f / tc) if f else 0.0) for _, b, f in op_table())


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    host = host_inputs(seed=0)
    ideal = ideal_step_seconds()
    for w in range(args.warmup):
        oracle_sample(host, args.cpu_frac, seed=1000 + w)
    full, meas = [], []
    for s in range(args.steps):
        f, m, desc, cores = oracle_sample(host, args.cpu_frac, seed=s)
        full.append(f)
        meas.append(m)
    sec = statistics.mean(full)
    val = round(100.0 * ideal / sec, 8)
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
            "ms_per_step_kind": "scaled from the sample (see cpu_baseline.sample)",
            "sample_ms_per_step_measured": round(statistics.mean(meas) * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "same step as the GPU arm (oracle, CPU)"},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# --------------------------------------------------------------------------- one op
def single_op(T, torch, name, dev, device):
    """Enqueue function of one op of the step, on its full-size inputs only;
    what feeds it (the forward before a backward, the gather before the MU
    attention, the premix before the long-context attention) runs once here."""
    pm, aw, mu, lc = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU, S.LONG_CTX
    e = lambda shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt, device=device)
    i = dev
    kind, t = name.rsplit("_", 1) if name[-2:] in ("_q", "_k", "_v") else (name, None)
    ly = {u: e((lc.B, lc.N, lc.HP, lc.d)) for u in "qkv"} if kind.startswith("long") else None
    long_premix = (lambda: T.premix_fwd_qkv([i[f"lx_{u}"] for u in "qkv"],
                                            [i[f"lw_{u}"] for u in "qkv"], lc.P, rope=True,
                                            rope_base=S.ROPE_BASE,
                                            out=tuple(ly[u] for u in "qkv"))
                   if ly is not None else None)
    if kind == "premix_fwd_qkv":
        y = tuple(e((pm.B, pm.N, pm.HP, pm.d)) for _ in range(3))
        return lambda: T.premix_fwd_qkv([i[f"x_{u}"] for u in "qkv"], [i[f"w_{u}"] for u in "qkv"],
                                        pm.P, rope=True, rope_base=S.ROPE_BASE, out=y)
    if kind == "premix_bwd_qkv":
        dx = tuple(e((pm.B, pm.N, pm.H, pm.d)) for _ in range(3))
        dw = tuple(e((pm.H, pm.P, pm.H), torch.float32) for _ in range(3))
        return lambda: T.premix_bwd_qkv([i[f"dy_{u}"] for u in "qkv"], [i[f"x_{u}"] for u in "qkv"],
                                        [i[f"w_{u}"] for u in "qkv"], rope=True,
                                        rope_base=S.ROPE_BASE, dxs=dx, dws=dw)
    if kind in ("attention_window", "attention_window_bwd"):
        o, lse = e((aw.B, aw.N, aw.HP, aw.d)), e((aw.B, 1, aw.HP, aw.N), torch.float32)
        fwd = lambda: T.mha_fwd(i["a_q"], i["a_k"], i["a_v"], mask=T.MASK_CAUSAL_WINDOW,
                                window=S.WINDOW_KEYS, out=o, lse=lse)
        if kind == "attention_window":
            return fwd
        fwd()
        g = [e((aw.B, aw.N, aw.HP, aw.d)) for _ in range(3)]
        ws = torch.empty(T.mha_bwd_workspace_bytes(aw.B, aw.HP, aw.N, aw.d), dtype=torch.uint8,
                         device=device)
        return lambda: T.mha_bwd(i["a_q"], i["a_k"], i["a_v"], o, i["a_do"], lse,
                                 mask=T.MASK_CAUSAL_WINDOW, window=S.WINDOW_KEYS, dq=g[0],
                                 dk=g[1], dv=g[2], workspace=ws)
    if kind == "mu_attention_fused":
        canvas = torch.zeros_like(i["mu_x"])
        return lambda: T.mu_attention_fused(i["mu_x"], i["mu_keep"], canvas, mu.grid_h, mu.grid_w,
                                            mu.mu_h, mu.mu_w)
    if kind == "mu_attention_qpool":
        return qpool_case(T, torch, device)[0]
    if kind.startswith("mu_"):
        g, ou = e((mu.B, mu.n_keep, mu.unit_tokens, mu.C)), e((mu.B, mu.n_keep, mu.unit_tokens, mu.C))
        dec = torch.zeros((mu.B, mu.grid_h * mu.grid_w, mu.C), dtype=torch.bfloat16, device=device)
        gather = lambda: T.mu_gather(i["mu_x"], i["mu_keep"], mu.grid_h, mu.grid_w, mu.mu_h,
                                     mu.mu_w, out=g)
        u = g.view(mu.B * mu.n_keep, 1, mu.unit_tokens, 1, mu.C)
        attn = lambda: T.mha_fwd(u, u, u, out=ou.view(mu.B * mu.n_keep, 1, mu.unit_tokens, 1, mu.C))
        scatter = lambda: T.mu_scatter(ou, i["mu_keep"], dec, mu.grid_h, mu.grid_w, mu.mu_h,
                                       mu.mu_w)
        if kind == "mu_gather":
            return gather
        gather()
        if kind == "mu_attention":
            return attn
        attn()
        return scatter
    if kind == "long_premix_fwd_qkv":
        return long_premix
    if kind == "long_attention_causal":
        long_premix()
        lo, llse = e((lc.B, lc.N, lc.HP, lc.d)), e((lc.B, 1, lc.HP, lc.N), torch.float32)
        return lambda: T.mha_fwd(ly["q"], ly["k"], ly["v"], mask=T.MASK_CAUSAL, out=lo, lse=llse)
    raise ValueError(f"unknown op {name}")


def single_op_arm(args):
    """Time one op of the step alone (the case `ncu -k` captures): warm-up,
    then `steps` launches between CUDA events on the launching stream."""
    import torch
    import transformer_attention_iha_gb300 as T
    T.build()
    T.lib()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    host = host_inputs(0, OP_INPUTS[args.only])
    dev = {k: host_tensor(v, torch).to(device) for k, v in host.items()}
    run = single_op(T, torch, args.only, dev, device)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize(device)
    if T.device_error() != 0:
        raise RuntimeError("device error word set")
    table = {n: (b, f) for n, b, f in op_table()}
    mu = S.HIERA_MU
    table["mu_attention_fused"] = (2 * mu.B * mu.n_keep * mu.unit_tokens * mu.C * 2 +
                                   mu.B * mu.n_keep * 4,
                                   4 * mu.C * mu.unit_tokens ** 2 * mu.B * mu.n_keep)
    hq = S.HIERA_QPOOL
    units = hq.B * hq.n_units * hq.heads
    table["mu_attention_qpool"] = (units * (3 * hq.T + hq.Tq) * hq.head_dim * 2,
                                   4 * hq.head_dim * hq.Tq * hq.T * units)
    nbytes, flops = table[args.only]
    ms = e0.elapsed_time(e1) / args.steps
    out = {"op": args.only, "ms": round(ms, 5), "GB/s": round(nbytes / ms / 1e6, 1),
           "bytes": nbytes, "flops": flops, "steps": args.steps, "warmup": args.warmup,
           "note": "back-to-back launches of one op (inputs may stay in L2); not the step metric"}
    if flops:
        out["TFLOP/s"] = round(flops / ms / 1e9, 1)
    return out


# --------------------------------------------------------------------------- main
def make_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of the run; must equal WORLD_SIZE (torchrun) when > 1")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--cpu-frac", type=float, default=CPU_FRAC,
                    help="fraction of every op each oracle sample runs")
    ap.add_argument("--cpu-samples", type=int, default=2,
                    help="oracle samples behind the cpu_baseline of the GPU arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=sorted(OP_INPUTS),
                    help="time one op of the step alone on one GPU (profiling case)")
    return ap


def main():
    ap = make_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N>1 with "
                 f"torch.distributed.run --nproc-per-node N")

    if args.only:
        if world != 1 or args.impl != "native":
            ap.error("--only runs the native arm on one GPU")
        print(json.dumps(single_op_arm(args)), flush=True)
        return

    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    # oracle CPU baseline first, before any CUDA call in this process
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = host_inputs(seed=0)
        full, meas = [], []
        for s in range(args.cpu_samples):
            f, m, desc, cores = oracle_sample(host, args.cpu_frac, seed=s)
            full.append(f)
            meas.append(m)
        sec = statistics.mean(full)
        cpu = {"value": round(100.0 * ideal_step_seconds() / sec, 8), "unit": UNIT,
               "cores": cores, "kind": "oracle", "sample": desc,
               "ms_per_step_scaled": round(sec * 1e3, 1),
               "sample_ms_measured": round(statistics.mean(meas) * 1e3, 1),
               "samples": args.cpu_samples}
        del host

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = gpu_arm(args, rank, world, local_rank)
    line["cpu_baseline"] = cpu
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
