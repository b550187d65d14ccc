#!/usr/bin/env python3
"""Benchmark of the IHA attention-layer hot path on GB300.

One step = one pass of every hot-path operation over one batch of seeded
synthetic inputs, each at its workload's shape:
  premix   LLaMA-2.4B layer shape B=1, N=8192, H=20, P=4, d=128:
           forward for Q and K (fused RoPE, base 10000) and V; backward (input
           gradient with inverse RoPE for Q, K, and weight gradient) for Q, K, V,
           both gradients from one pass over dY;
  attention 80 pseudo-heads, N=4096, d=128, causal window W=1024, fp32 LSE;
  Hiera    MAE stage 1, B=128, 56x56 tokens, 8x8 units, 20 kept, C=d=96:
           gather, attention inside each unit, scatter.
The step's working set (~1.7 GB) is far larger than L2 (129 MB), so no L2
flush is needed between steps: every op's inputs were evicted by the others.

Metric: every op has an algorithmic roofline time, max(bytes / HBM peak,
flops / bf16 peak) with the measured peaks; the step's efficiency is the sum
of those times over the measured step time.  `value` is that efficiency in %
summed over GPUs (so it adds up across replicas; at N=1 it is the
efficiency).  Per-op GB/s and TFLOP/s are in `ops`.

--impl reference times the oracle (CPU) on a bounded sample of the same step
and extrapolates; it is a deliberately slow baseline, not a target.
"""
from __future__ import annotations

import argparse
import json
import math
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

# dram bytes (read + write) per launch from ncu captures of the current kernels
# (see profiles/); None where no capture of the current kernel exists.
NCU_TRAFFIC = {}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- workload
def op_table():
    """(name, kind, algorithmic bytes, algorithmic flops) per op of one step."""
    pm = S.LLAMA_PREMIX
    tok = pm.B * pm.N
    x_b = tok * pm.H * pm.d * 2
    y_b = tok * pm.HP * pm.d * 2
    w_b = pm.HP * pm.H * 4
    premix_flops = 2 * tok * pm.HP * pm.H * pm.d
    ops = []
    for t in ("q", "k", "v"):
        ops.append((f"premix_fwd_{t}", "premix", x_b + y_b + w_b, premix_flops))
    for t in ("q", "k", "v"):   # dX and dW from one read of dY and X
        ops.append((f"premix_bwd_{t}", "premix", y_b + 2 * x_b + 2 * w_b, 2 * premix_flops))
    aw = S.LLAMA_WINDOW
    W = S.WINDOW_KEYS
    pairs = sum(min(i + 1, W) for i in range(aw.N))
    attn_flops = 4 * aw.d * pairs * aw.HP
    attn_bytes = 4 * aw.B * aw.N * aw.HP * aw.d * 2 + aw.B * aw.HP * aw.N * 4
    ops.append(("attention_window", "attention", attn_bytes, attn_flops))
    mu = S.HIERA_MU
    kept = mu.B * mu.n_keep * mu.unit_tokens * mu.C * 2
    ops.append(("mu_gather", "gather", 2 * kept + mu.B * mu.n_keep * 4, 0))
    mu_flops = 4 * mu.C * mu.unit_tokens * mu.unit_tokens * mu.B * mu.n_keep
    ops.append(("mu_attention", "attention", 4 * kept, mu_flops))
    ops.append(("mu_scatter", "gather", 2 * kept + mu.B * mu.n_keep * 4, 0))
    return ops


LAUNCHES_PER_STEP = 3 + 3 * 2 + 1 + 3   # premix fwd, bwd (zero dW + kernel), attention, MU x3


def host_inputs(seed: int):
    pm, aw, mu = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU
    d = {}
    for c, t in enumerate("qkv"):
        d[f"x_{t}"] = S.normal((pm.B, pm.N, pm.H, pm.d), seed, 10 + c)
        d[f"w_{t}"] = S.premix_weight(pm.H, pm.P, seed, 20 + c)
        d[f"dy_{t}"] = S.normal((pm.B, pm.N, pm.HP, pm.d), seed, 30 + c)
    for c, t in enumerate("qkv"):
        d[f"a_{t}"] = S.normal((aw.B, aw.N, aw.HP, aw.d), seed, 40 + c)
    d["mu_x"] = S.normal((mu.B, mu.grid_h * mu.grid_w, mu.C), seed, 50)
    d["mu_keep"] = S.keep_units(mu.B, mu.n_units, mu.n_keep, seed)
    return d


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
    """Device buffers and the launch sequence of one step."""

    def __init__(self, T, torch, dev_inputs, device):
        pm, aw, mu = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU
        self.T, self.torch = T, torch
        self.i = dev_inputs
        e = lambda shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt, device=device)
        self.y = {t: e((pm.B, pm.N, pm.HP, pm.d)) for t in "qkv"}
        self.dx = {t: e((pm.B, pm.N, pm.H, pm.d)) for t in "qkv"}
        self.dw = {t: e((pm.H, pm.P, pm.H), torch.float32) for t in "qkv"}
        self.o = e((aw.B, aw.N, aw.HP, aw.d))
        self.lse = e((aw.B, 1, aw.HP, aw.N), torch.float32)
        self.g = e((mu.B, mu.n_keep, mu.unit_tokens, mu.C))
        self.ou = e((mu.B, mu.n_keep, mu.unit_tokens, mu.C))
        self.dec = torch.zeros((mu.B, mu.grid_h * mu.grid_w, mu.C), dtype=torch.bfloat16,
                               device=device)

    def outputs(self):
        return ([self.y[t] for t in "qkv"] + [self.dx[t] for t in "qkv"] +
                [self.dw[t] for t in "qkv"] + [self.o, self.lse, self.dec])

    def run(self, marks=None):
        """Enqueue the step; `marks(i)` records an event after op i (and before op 0)."""
        T, i = self.T, self.i
        pm, aw, mu = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU
        mark = marks or (lambda k: None)
        k = 0
        mark(k)
        for t in "qkv":
            T.premix_fwd(i[f"x_{t}"], i[f"w_{t}"], pm.P, rope=(t != "v"), rope_base=S.ROPE_BASE,
                         out=self.y[t])
            k += 1
            mark(k)
        for t in "qkv":
            T.premix_bwd(i[f"dy_{t}"], i[f"x_{t}"], i[f"w_{t}"], rope=(t != "v"),
                         rope_base=S.ROPE_BASE, dx=self.dx[t], dw=self.dw[t])
            k += 1
            mark(k)
        T.mha_fwd(i["a_q"], i["a_k"], i["a_v"], mask=T.MASK_CAUSAL_WINDOW, window=S.WINDOW_KEYS,
                  out=self.o, lse=self.lse)
        k += 1
        mark(k)
        T.mu_gather(i["mu_x"], i["mu_keep"], mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w, out=self.g)
        k += 1
        mark(k)
        u = self.g.view(mu.B * mu.n_keep, 1, mu.unit_tokens, 1, mu.C)
        T.mha_fwd(u, u, u, out=self.ou.view(mu.B * mu.n_keep, 1, mu.unit_tokens, 1, mu.C))
        k += 1
        mark(k)
        T.mu_scatter(self.ou, i["mu_keep"], self.dec, mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w)
        k += 1
        mark(k)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.lines = []

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


def gpu_arm(args, rank, world, local_rank):
    import torch
    import transformer_attention_iha_gb300 as T
    T.build()
    T.lib()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 1e12

    host = host_inputs(seed=rank)
    hostt = {k: host_tensor(v, torch) for k, v in host.items()}
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

    # per-op events: K x (nops + 1)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)] for _ in range(args.steps)]
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
    total_ms = start.elapsed_time(end)
    if world > 1:
        t = torch.tensor([total_ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_step = total_ms / args.steps
    op_ms = [statistics.mean(evs[s][k].elapsed_time(evs[s][k + 1]) for s in range(args.steps))
             for k in range(nops)]
    derr = T.device_error()

    # roofline per op and for the step
    op_out = {}
    ideal_total = 0.0
    for (name, kind, nbytes, flops), ms in zip(ops, op_ms):
        t_hbm = nbytes / hbm
        t_tc = flops / tc if flops else 0.0
        ideal = max(t_hbm, t_tc)
        ideal_total += ideal
        rec = {"ms": round(ms, 5), "roofline_ms": round(ideal * 1e3, 5),
               "frac": round(ideal / (ms * 1e-3), 4)}
        rec["GB/s"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
        if flops:
            rec["TFLOP/s"] = round(flops / (ms * 1e-3) / 1e12, 1)
        rec["bound"] = "tensor" if t_tc > t_hbm else "hbm"
        op_out[name] = rec
    eff = ideal_total / (ms_step * 1e-3)

    # dominant kernel by time share
    dom = max(range(nops), key=lambda k: op_ms[k])
    dname, dkind, dbytes, dflops = ops[dom]
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
    roof["peak_source"] = peak_src + (" sustained" if roof["bound"] == "tensor" else "")

    # end to end: host buffers, H2D of every input and D2H of every output per step
    e2e = None
    if args.e2e_steps > 0:
        pinned = {k: v.pin_memory() for k, v in hostt.items()}
        outs_host = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in step.outputs()]
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        d2h = sum(o.numel() * o.element_size() for o in outs_host)

        def e2e_step():
            for k, v in pinned.items():
                dev[k].copy_(v, non_blocking=True)
            step.run()
            for o, h in zip(step.outputs(), outs_host):
                h.copy_(o, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        if world > 1:
            t = torch.tensor([e2e_ms], device=device)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(t.item())
        e2e = {"value": round(100.0 * ideal_total / (e2e_ms * 1e-3) * world, 3),
               "unit": "% of 1-GPU roofline, summed over GPUs", "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    line = {
        "metric": METRIC,
        "value": round(100.0 * eff * world, 3),
        "unit": "% of 1-GPU roofline, summed over GPUs",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, W ~ N(0,1/H) fp32)",
        "config": {"workload": "IHA hot-path step: premix fwd(+RoPE) and fused dX+dW for Q,K,V at "
                               "B=1,N=8192,H=20,P=4,d=128; causal-window attention 80 heads "
                               "N=4096 d=128 W=1024; Hiera-Base MAE stage-1 gather + mask-unit "
                               "attention (2560 units x 64 tokens, d=96) + scatter",
                   "l2": "no flush: step working set ~1.7 GB > 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "ops": op_out,
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clk,
        "device_error": derr,
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops_sustained": tc / 1e12,
                  "source": peak_src},
    }
    return line, step


# --------------------------------------------------------------------------- CPU (oracle) arm
def oracle_sample(host, frac: float):
    """Time the oracle on a bounded sample of one step and extrapolate.

    Returns (extrapolated seconds per full step, sample description, threads)."""
    import oracle as O
    pm, aw, mu = S.LLAMA_PREMIX, S.LLAMA_WINDOW, S.HIERA_MU
    ntok = max(1, int(pm.N * frac))
    t_total = 0.0
    for t in "qkv":
        rope = t != "v"
        x, w, dy = host[f"x_{t}"][:, :ntok], host[f"w_{t}"], host[f"dy_{t}"][:, :ntok]
        t0 = time.perf_counter()
        O.premix_fwd(x, w, pm.P, rope=rope, rope_base=S.ROPE_BASE)
        O.premix_bwd_dx(dy, w, rope=rope, rope_base=S.ROPE_BASE)
        O.premix_bwd_dw(dy, x, pm.P, rope=rope, rope_base=S.ROPE_BASE)
        t_total += (time.perf_counter() - t0) * (pm.N / ntok)
    nrows_all = aw.N * aw.HP
    nrows = max(1, int(nrows_all * frac))
    g = np.random.default_rng(0)
    rows = np.stack([np.zeros(nrows, np.int64), np.zeros(nrows, np.int64),
                     g.integers(0, aw.HP, nrows), g.integers(0, aw.N, nrows)], axis=1)
    qa, ka, va = (host[f"a_{t}"][:, None] for t in "qkv")
    t0 = time.perf_counter()
    O.attention_rows(qa, ka, va, rows, O.MASK_CAUSAL_WINDOW, S.WINDOW_KEYS)
    t_total += (time.perf_counter() - t0) * (nrows_all / nrows)
    nb = max(1, int(mu.B * frac))
    x, keep = host["mu_x"][:nb], host["mu_keep"][:nb]
    t0 = time.perf_counter()
    gg = O.mu_gather(x, keep, mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w)
    u = gg.reshape(nb * mu.n_keep, 1, mu.unit_tokens, 1, mu.C)
    ou, _ = O.attention(u, u, u)
    ob = S.f32_to_bf16_bits(ou.astype(np.float32)).reshape(nb, mu.n_keep, mu.unit_tokens, mu.C)
    O.mu_scatter(ob, keep, np.zeros_like(x), mu.grid_h, mu.grid_w, mu.mu_h, mu.mu_w)
    t_total += (time.perf_counter() - t0) * (mu.B / nb)
    desc = (f"{ntok}/{pm.N} tokens per premix op, {nrows}/{nrows_all} attention rows, "
            f"{nb}/{mu.B} Hiera samples; times scaled to the full step")
    return t_total, desc, O.num_threads()


def ideal_step_seconds():
    peaks, _ = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 1e12
    return sum(max(b / hbm, (f / tc) if f else 0.0) for _, _, b, f in op_table())


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    host = host_inputs(seed=0)
    ideal = ideal_step_seconds()
    for _ in range(args.warmup):
        oracle_sample(host, args.ref_frac)
    times = []
    for _ in range(args.steps):
        t, desc, cores = oracle_sample(host, args.ref_frac)
        times.append(t)
    sec = statistics.mean(times)
    val = round(100.0 * ideal / sec, 8)
    unit = "% of 1-GPU roofline, summed over GPUs"
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": "same step as the GPU arm (oracle, CPU)"},
            "cpu_baseline": {"value": val, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-frac", type=float, default=1 / 4,
                    help="fraction of the step the CPU baseline samples")
    ap.add_argument("--ref-frac", type=float, default=1 / 64,
                    help="fraction of the step each reference-arm step samples")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    # oracle CPU baseline first (spawned-free: before any CUDA call in this process)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = host_inputs(seed=0)
        sec, desc, cores = oracle_sample(host, args.cpu_frac)
        cpu = {"value": round(100.0 * ideal_step_seconds() / sec, 8),
               "unit": "% of 1-GPU roofline, summed over GPUs", "cores": cores, "kind": "oracle",
               "sample": desc, "ms_per_step": round(sec * 1e3, 1)}
        del host

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line, _ = gpu_arm(args, rank, world, local_rank)
    line["cpu_baseline"] = cpu
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
