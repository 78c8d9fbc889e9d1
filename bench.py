#!/usr/bin/env python3
"""Benchmark of the GB300 attention forward (one JSON line on rank 0).

Workload ("S=4K/8K/16K sweep"): the headline shapes S=4K (B=4, H=16), S=8K
(B=2, H=16), S=16K (B=1, H=16); D=128, dense, non-causal, BF16, scale
1/sqrt(128), inputs N(0,1).  One step is a batch of --reps independent problems
of each shape (default 24, each with its own Q/K/V/O buffers, all resident in
HBM), run as one attention forward per problem, shape after shape; with the
default 20 steps the timed region is about a second.  metric: TFLOPS =
4*B*H*Sq*Sk*D summed over the step's problems / the step's device time, and its
fraction of the measured GB300 dense BF16 peak; the line also gives the median
step's figure (value_p50).  Every problem's inputs (Q+K+V = 192 MiB) are larger
than the 129 MB L2, and consecutive launches read different problems' inputs,
so no explicit flush is needed between timed iterations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--reps R]
                  [--impl ours|reference]
                  [--row dense|causal|bshd|soft-exp2|backward|backward-causal]

--row (default dense, the headline above) times the same sweep on one of the
other built rows instead: the causal forward (half of 4*B*H*S^2*D counted),
the [B,S,H,D] forward, or the backward (dQ, dK, dV; 2.5x the forward FLOPs
counted, the convention of the FlashAttention papers).

--impl reference times the fp64 CPU oracle (the only reference this path has)
on bounded samples of the same workload, on the host cores.
Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (replicas, weak scaling); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS (4·B·H·S²·D) at S=4K/8K/16K, % of GB300 BF16 peak"
UNIT = "TFLOP/s"
WORKLOAD = "S=4K/8K/16K sweep (B=4/2/1, H=16, D=128, BF16, non-causal)"
FALLBACK_BF16_TFLOPS = 1900.0
# MUFU exp2 rate per SM: 4 sub-partitions x one 32-lane ex2 warp instruction per 4 clocks, as
# measured on GB300 with back-to-back ex2.approx.ftz; the co-roofline's peak is this x SMs x the
# SM clock sampled during the timed region.
MUFU_EX2_PER_CLK_PER_SM = 32

# --row: (metric, workload, FLOP factor on 4*B*H*S^2*D)
ROWS = {
    "dense": (METRIC, WORKLOAD, 1.0),
    "causal": ("attention fwd TFLOPS, causal (half of 4·B·H·S²·D counted) at S=4K/8K/16K",
               "S=4K/8K/16K sweep (B=4/2/1, H=16, D=128, BF16, causal top-left)", 0.5),
    "bshd": ("attention fwd TFLOPS (4·B·H·S²·D), [B,S,H,D] tensors, at S=4K/8K/16K",
             "S=4K/8K/16K sweep (B=4/2/1, H=16, D=128, BF16, non-causal, BSHD layout)", 1.0),
    "soft-exp2": ("attention fwd TFLOPS (4·B·H·S²·D), 4/16 of P by software exp2, at S=4K/8K/16K",
                  "S=4K/8K/16K sweep (B=4/2/1, H=16, D=128, BF16, non-causal, ATTN_FLAG_SOFT_EXP2)",
                  1.0),
    "backward": ("attention bwd TFLOPS (2.5 × 4·B·H·S²·D) at S=4K/8K/16K",
                 "S=4K/8K/16K sweep (B=4/2/1, H=16, D=128, BF16, non-causal), dQ/dK/dV", 2.5),
    "backward-causal": ("attention bwd TFLOPS, causal (1.25 × 4·B·H·S²·D) at S=4K/8K/16K",
                        "S=4K/8K/16K sweep (B=4/2/1, H=16, D=128, BF16, causal), dQ/dK/dV", 1.25),
}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in a background process."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the timing rule: a step takes as long as its slowest
    replica); the value itself when no process group is initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _source_sha() -> str:
    """Hash of the forward kernel's device source (the files its code is compiled from), with
    comments and blank lines removed, so that only code changes make a recorded profile stale."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_attention_forward_attn_gb300", "csrc")
    for name in ("attn_fwd_kernel.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(name.encode() + code.encode())
    return h.hexdigest()[:16]


def _traffic_for(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on this exact source."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_kernel_dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha") != _source_sha():
            return None
        return d["per_launch_bytes"].get(workload_name)
    except Exception:
        return None


def oracle_sample_tflops(shapes, seconds: float, seed: int = 0):
    """Time the fp64 CPU oracle on random rows of each shape for about `seconds` in total."""
    import numpy as np
    import oracle
    from dense_attention_forward_attn_gb300 import workloads as wl

    total_flops, total_t, rows_done = 0.0, 0.0, []
    per = seconds / len(shapes)
    threads = oracle.max_threads()
    for w, (qb, kb, vb) in shapes:
        # calibrate with a small batch, then run a batch sized to `per` seconds
        rng = np.random.Generator(np.random.PCG64(seed))
        n = max(threads, 16)
        bh = rng.integers(0, w.B * w.H, n)
        rows = rng.integers(0, w.Sq, n)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(qb, kb, vb, w.scale, bh, rows)
        dt = time.perf_counter() - t0
        n2 = max(threads, int(n * per / max(dt, 1e-6)))
        bh = rng.integers(0, w.B * w.H, n2)
        rows = rng.integers(0, w.Sq, n2)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(qb, kb, vb, w.scale, bh, rows)
        dt = time.perf_counter() - t0
        total_flops += 4.0 * w.Sk * w.D * n2
        total_t += dt
        rows_done.append(f"{n2} rows of {w.name}")
    return total_flops / total_t / 1e12, threads, ", ".join(rows_done), total_t


def bench_config(workload, shapes, reps, ws, causal=False, layout="bhsd"):
    """The `config` object of the JSON line, the same for both arms."""
    described = []
    for w in shapes:
        d = w.describe()
        d["causal"] = bool(causal)
        if layout == "bshd":
            d["layout"] = "BSHD contiguous"
        described.append(d)
    return {"workload": workload, "shapes": described,
            "problems_per_shape_per_step": reps,
            "l2": "inputs larger than L2 (Q+K+V = 192 MiB per problem); consecutive launches read "
                  "different problems' inputs",
            "parallelism": "replicas" if ws > 1 else "single GPU"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    from dense_attention_forward_attn_gb300 import workloads as wl
    shapes = [(w, wl.workload_inputs_bits(w)) for w in wl.HEADLINE]
    step_s = 1.5
    vals, times = [], []
    for i in range(args.warmup + args.steps):
        v, cores, sample, t = oracle_sample_tflops(shapes, step_s, seed=i)
        if i >= args.warmup:
            vals.append(v)
            times.append(t)
    value = sum(vals) / len(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(WORKLOAD, wl.HEADLINE, args.reps, ws),
        "reference": "fp64 CPU oracle (oracle/attn_oracle.c), the only reference this path has",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: random query rows of each shape, about 0.5 s of "
                                   f"CPU work per shape (last step: {sample})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from dense_attention_forward_attn_gb300 import attn, workloads as wl

    row = args.row
    metric, workload, flop_factor = ROWS[row]
    causal = row in ("causal", "backward-causal")
    layout = "bshd" if row == "bshd" else "bhsd"
    soft = row == "soft-exp2"
    backward = row.startswith("backward")
    reps = max(1, args.reps)
    # Per shape: problem 0 from the seeded CPU generator (the inputs the oracle and the host-buffer
    # leg use), problems 1.. drawn on the device from seeded generators (the same N(0,1) inputs).
    shapes = []
    for si, w in enumerate(wl.HEADLINE):
        qb, kb, vb = wl.workload_inputs_bits(w)
        host = [wl.bits_to_torch(x) for x in (qb, kb, vb)]
        if layout == "bshd":
            host = [t.transpose(1, 2).contiguous() for t in host]
        host = [t.pin_memory() for t in host]
        probs = []
        for r in range(reps):
            if r == 0:
                d = [t.to(dev) for t in host]
            else:
                gen = torch.Generator(device=dev).manual_seed(1000 * (si + 1) + r)
                d = [torch.randn(t.shape, device=dev, generator=gen).to(torch.bfloat16) for t in host]
            o = torch.empty_like(d[0])
            lse = torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev)
            if backward:
                # O and LSE of the forward, an upstream gradient dO, and the gradient buffers
                attn.fwd_into(d[0], d[1], d[2], o, lse, w.scale, causal=causal)
                gen = torch.Generator(device=dev).manual_seed(5000 + 1000 * si + r)
                dout = torch.randn(d[0].shape, device=dev, generator=gen).to(torch.bfloat16)
                extra = (dout, torch.empty_like(d[0]), torch.empty_like(d[1]),
                         torch.empty_like(d[2]),
                         torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev))
            else:
                # attn_fwd_ws's workspace (None where the schedule runs whole items only)
                extra = attn.workspace_for(d[0], d[1], causal=causal, layout=layout, soft_exp2=soft)
            probs.append((d, o, lse, extra))
        shapes.append((w, (qb, kb, vb), host, probs))
    flops_step = flop_factor * reps * sum(w.flops for w, *_ in shapes)
    stream = torch.cuda.current_stream()
    attn.device_status(clear=True)
    lib = attn.library()
    bwd_flags = attn.ATTN_FLAG_CAUSAL if causal else 0

    def one(w, d, o, lse, extra):
        if not backward:
            attn.fwd_into(d[0], d[1], d[2], o, lse, w.scale, causal=causal, layout=layout,
                          soft_exp2=soft, workspace=extra)
            return
        dout, dq, dk, dv, delta = extra
        rc = lib.attn_bwd(d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), o.data_ptr(),
                          dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                          dv.data_ptr(), delta.data_ptr(), w.B, w.H, w.Sq, w.Sk, w.D, w.scale,
                          bwd_flags, stream.cuda_stream)
        if rc != attn.ATTN_OK:
            raise attn.AttnError(rc, "attn_bwd")

    def step(evs=None):
        # one step: every problem of every shape; evs[i][r] brackets launch r of shape i
        for i, (w, _, _, probs) in enumerate(shapes):
            for r, (d, o, lse, extra) in enumerate(probs):
                if evs is not None:
                    evs[i][r][0].record(stream)
                one(w, d, o, lse, extra)
                if evs is not None:
                    evs[i][r][1].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # ---------------- device-resident timed region
    n = len(shapes)
    mk = lambda: torch.cuda.Event(enable_timing=True)
    kev = [[[(mk(), mk()) for _ in range(reps)] for _ in range(n)] for _ in range(args.steps)]
    sev = [mk() for _ in range(args.steps + 1)]
    clocks = ClockSampler(local if ws > 1 else torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sev[0].record(stream)
    for s in range(args.steps):
        step(kev[s])
        sev[s + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_ms = [sev[s].elapsed_time(sev[s + 1]) for s in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    value = ws * flops_step / (ms_per_step * 1e-3) / 1e12
    p50_step = max_over_ranks(float(np.percentile(step_ms, 50)), dev)
    value_p50 = ws * flops_step / (p50_step * 1e-3) / 1e12
    per_cfg = {}
    kernel_ms_total = 0.0
    for i, (w, *_rest) in enumerate(shapes):
        ms = [a.elapsed_time(b) for s in range(args.steps) for (a, b) in kev[s][i]]
        avg = sum(ms) / len(ms)
        kernel_ms_total += avg * reps
        p10, p50, p90 = (float(np.percentile(ms, x)) for x in (10, 50, 90))
        # minimum HBM bytes of the forward: Q, K, V read once, O and LSE written once
        hbm = 2 * (2 * w.B * w.H * w.Sq * w.D + 2 * w.B * w.H * w.Sk * w.D) + 4 * w.B * w.H * w.Sq
        per_cfg[w.name] = {"launches": len(ms), "ms_avg": round(avg, 4), "ms_min": round(min(ms), 4),
                           "ms_p10": round(p10, 4), "ms_p50": round(p50, 4), "ms_p90": round(p90, 4),
                           "tflops": round(flop_factor * w.flops / (avg * 1e-3) / 1e12, 1),
                           "tflops_p50": round(flop_factor * w.flops / (p50 * 1e-3) / 1e12, 1)}
        if not backward:
            per_cfg[w.name]["hbm_min_gbs"] = round(hbm / (avg * 1e-3) / 1e9, 1)
    status = attn.device_status()

    # ---------------- end to end with host buffers (forward rows): attn.fwd_host_batch on pinned
    # CPU tensors runs attn_fwd_host (the C-ABI entry point that copies in chunks overlapped with
    # the kernels) for every problem of the step -- `reps` problems of each shape, each on its own
    # stream, every one copying its inputs in and its outputs back -- and returns their results
    # once all are complete; the library's copy streams keep the host link busy across problems
    e2e = None
    if not backward:
        h2d = reps * sum(sum(t.numel() * t.element_size() for t in host) for _, _, host, _ in shapes)
        d2h = reps * sum(p[1].numel() * p[1].element_size() + p[2].numel() * 4
                         for *_, probs in shapes for p in probs[:1])
        e2e_steps = max(2, min(args.steps, 10))
        problems = [dict(q=host[0], k=host[1], v=host[2], scale=w.scale, causal=causal, layout=layout,
                         soft_exp2=soft)
                    for w, _, host, _ in shapes]
        batch = problems * reps   # the step's problems (each shape's host inputs copied `reps` times)
        for _ in range(max(3, args.warmup)):   # warm-up: pinned output buffers, side streams
            results = attn.fwd_host_batch(batch)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            results = attn.fwd_host_batch(batch)   # one step: every problem, one call
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
        e2e = {"value": round(ws * flops_step / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 3), "steps": e2e_steps}

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak_burst, peak_sus, peak_kind = _peaks()
    # A timed region of back-to-back launches lasting half a second or more runs under the power
    # cap like the sustained cuBLAS loop; a shorter one is compared with the burst figure.
    sustained = total_ms >= 500.0
    peak = peak_sus if sustained else peak_burst
    achieved = flops_step / (kernel_ms_total * 1e-3) / 1e12
    traffic = None
    tr = [_traffic_for(w.name) for w, *_ in shapes]
    if row == "dense" and all(t is not None for t in tr):
        traffic = sum(tr) / len(tr)
    # co-roofline: one exp2 per score through the MUFU unit
    co = None
    if not backward and clk.get("sm_mhz"):
        exps = reps * sum(w.B * w.H * w.Sq * w.Sk * (0.5 if causal else 1.0) for w, *_ in shapes)
        ex_rate = exps / (kernel_ms_total * 1e-3)
        ex_peak = MUFU_EX2_PER_CLK_PER_SM * torch.cuda.get_device_properties(dev).multi_processor_count \
            * clk["sm_mhz"] * 1e6
        co = {"bound": "mufu", "achieved": round(ex_rate / 1e12, 3), "peak": round(ex_peak / 1e12, 3),
              "unit": "Texp2/s", "frac": round(ex_rate / ex_peak, 4),
              "peak_kind": "derived: 32 ex2/clk/SM (measured) x SMs x sampled SM clock"}
    cpu = None
    if ws == 1 and not args.no_cpu_baseline and row == "dense":
        v, cores, sample, _t = oracle_sample_tflops([(w, bits) for w, bits, *_ in shapes], 12.0)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{sample} (fp64 oracle, random query rows, ~12 s total)"}
    line = {
        "metric": metric, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4),
        "value_p50": round(value_p50, 2), "ms_per_step_p50": round(p50_step, 4),
        "timed_region_s": round(total_ms / 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(workload, [w for w, *_ in shapes], reps, ws, causal=causal,
                               layout=layout),
        "detail": {"per_shape": per_cfg, "frac_of_peak": round(value / peak, 4),
                   "frac_of_burst_peak": round(value / peak_burst, 4),
                   "device_status": status,
                   "inputs": "problem 0 of each shape from the seeded CPU generator (workloads.py), "
                             "the others N(0,1) from seeded torch CUDA generators"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": UNIT, "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": (f"{peak_kind} sustained bf16 (cuBLAS back to back under the "
                                   f"power cap; this timed region is {total_ms / 1e3:.2f} s of "
                                   f"back-to-back launches)") if sustained
                                  else f"{peak_kind} burst bf16 (cuBLAS)",
                     "burst_peak": peak_burst, "frac_of_burst_peak": round(achieved / peak_burst, 4)},
        "co_roofline": co,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * reps * len(shapes) * (3 if backward else 1),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=24,
                    help="independent problems of each shape per step (default 24: ~50 ms steps)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--row", choices=sorted(ROWS), default="dense",
                    help="which built row to time (default: the dense headline)")
    args = ap.parse_args()
    if args.impl == "reference" and args.row != "dense":
        ap.error("--impl reference times the dense headline only")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
