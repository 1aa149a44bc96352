#!/usr/bin/env python
"""Benchmark of the jagged flash-attention hot path on GB300.

One step = forward + backward of the jagged self-attention workload (B=32
packed sequences, lengths log-uniform in [32, 4096], H=8, head_dim 128, bf16),
run twice: non-causal and causal within each sequence.  Throughput is counted
on valid tokens only (4*D FLOPs per scored query-key pair forward, 2.5x that
backward) and reported as TFLOP/s of the whole job.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (weak scaling,
no data-path collective); the barrier and the max-over-ranks time use
torch.distributed.  `--impl reference` times the fp64 CPU oracle on a bounded
sample of the same workload instead (rank 0 only).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "jagged attn fwd/bwd TFLOP/s on valid tokens, bf16; % of BF16 tensor peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
PROFILE_FILE = os.path.join(ROOT, "profiles", "bwd_main_jagged_B32_H8_D128.txt")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    """Largest value of x over all ranks (the slowest rank sets the job time)."""
    if ws <= 1:
        return float(x)
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_flops: float, steps: int, max_ms: float, ws: int) -> float:
    """Whole-job TFLOP/s: every rank runs the same step (weak scaling)."""
    return ws * step_flops * steps / (max_ms * 1e-3) / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = dict(FALLBACK_PEAKS)
        for k in out:
            if k in d:
                out[k] = float(d[k])
        return out, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _workloads():
    from variable_length_attention_gb300 import workloads as W
    return [W.jagged(False), W.jagged(True)]


def _kernel_sha():
    h = hashlib.sha256()
    for f in ("bwd.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "variable_length_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic():
    """DRAM bytes per launch of the backward main kernel from a committed ncu
    summary, if it was taken on the current kernel source; else None."""
    if not os.path.exists(PROFILE_FILE):
        return None
    vals = {}
    with open(PROFILE_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != _kernel_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"jfa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(sample_flops_target=1e11, seed=7):
    """The fp64 oracle (as it stands) on a bounded sample of the workload's
    (sequence, head) units: forward + backward, non-causal and causal."""
    import oracle
    from variable_length_attention_gb300 import workloads as W
    ws = _workloads()
    w = ws[0]
    q, k, v, do = [t.float().numpy().astype(np.float64) for t in w.tensors("cpu")]
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.batch * w.num_heads)
    sel = np.zeros((w.batch, w.num_heads), dtype=bool)
    L = w.lengths.astype(np.float64)
    flops = 0.0
    for u in order:
        b = u // w.num_heads
        f = 4 * w.head_dim * (L[b] * L[b] + L[b] * (L[b] + 1) / 2) * 3.5  # nc + causal, fwd + 2.5x bwd
        sel.flat[u] = True
        flops += f
        if flops >= sample_flops_target:
            break
    t0 = time.perf_counter()
    threads = 0
    for wl in ws:
        _, _, threads = oracle.attn_fwd(q, k, v, w.offsets, scale=w.scale, causal=wl.causal, sel=sel)
        oracle.attn_bwd(q, k, v, do, w.offsets, scale=w.scale, causal=wl.causal, sel=sel)
    dt = time.perf_counter() - t0
    n_units = int(sel.sum())
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": int(threads), "kind": "oracle",
            "sample": f"{n_units} of {w.batch * w.num_heads} (sequence, head) units of the same workload, "
                      f"fwd+bwd, non-causal and causal, fp64 ({flops:.3g} FLOP counted on valid tokens) "
                      f"in {dt:.1f} s"}


def run_reference(args, ws, rank):
    """The oracle as the reference arm: each step is a bounded sample."""
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        if rank != 0:
            dist.destroy_process_group()
            return
    for _ in range(args.warmup):
        cpu_baseline(sample_flops_target=2e10, seed=1)
    vals = []
    t0 = time.perf_counter()
    for s in range(args.steps):
        vals.append(cpu_baseline(sample_flops_target=4e10, seed=100 + s))
    dt = time.perf_counter() - t0
    v = float(statistics.mean(x["value"] for x in vals))
    w = _workloads()[0]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name + " (+causal)", "batch": w.batch,
                                            "heads": w.num_heads, "head_dim": w.head_dim,
                                            "tokens": w.total_tokens},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = _args()
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    import variable_length_attention_gb300 as V
    from variable_length_attention_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench.py needs a GPU"
    dev = torch.device("cuda", local)
    wls = _workloads()
    w = wls[0]
    # identical inputs for both variants (same seeds); generated on the host, then resident in HBM
    hq, hk, hv, hdo = [t.pin_memory() for t in w.tensors("cpu")]
    q, k, v, do = [t.to(dev) for t in (hq, hk, hv, hdo)]
    offs_h = w.offsets
    offs = torch.from_numpy(offs_h).to(dev)
    outs = []
    for wl in wls:
        o = torch.empty_like(q)
        lse = torch.empty((w.num_heads, w.total_tokens), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        need = max(V.jfa_workspace_size(0, offs_h, w.batch, 0, w.num_heads, w.head_dim, wl.causal, 0),
                   V.jfa_workspace_size(1, offs_h, w.batch, 0, w.num_heads, w.head_dim, wl.causal, 0))
        wsb = torch.empty(need, dtype=torch.uint8, device=dev)
        outs.append((wl, o, lse, dq, dk, dv, wsb))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)
    fl = [W.flops(wl) for wl in wls]
    step_flops = float(sum(f + b for f, b in fl))

    def step(qq, kk, vv, dd):
        for wl, o, lse, dq, dk, dv, wsb in outs:
            V.jfa_fwd(qq, kk, vv, offs, offs_h, causal=wl.causal, out=o, lse=lse, workspace=wsb)
            V.jfa_bwd(qq, kk, vv, o, dd, lse, offs, offs_h, causal=wl.causal, dq=dq, dk=dk, dv=dv, workspace=wsb)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step(q, k, v, do)
    barrier()
    # ---------------------------------------------------------------- timed region (device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    V.jfa_profile_enable(True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        for i in range(args.steps):
            flush.zero_()  # L2 flush between timed steps, outside the events
            evs[i][0].record()
            step(q, k, v, do)
            evs[i][1].record()
        barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    prof = {kind: V.jfa_profile_read(kind) for kind in V.jfa.KERNEL_KINDS}
    V.jfa_profile_enable(False)
    total_ms = max_over_ranks(float(sum(step_ms)), ws)
    ms_per_step = total_ms / args.steps
    value = job_throughput(step_flops, args.steps, total_ms, ws)

    # ---------------------------------------------------------------- e2e through host buffers
    o_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for _, o, _, dq, dk, dv, _ in outs
           for t in (o, dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo)) + offs_h.nbytes
    d2h = sum(t.numel() * t.element_size() for t in o_h)

    def e2e_step():
        qq, kk, vv, dd = [t.to(dev, non_blocking=True) for t in (hq, hk, hv, hdo)]
        step(qq, kk, vv, dd)
        i = 0
        for _, o, _, dq, dk, dv, _ in outs:
            for t in (o, dq, dk, dv):
                o_h[i].copy_(t, non_blocking=True)
                i += 1

    for _ in range(2):
        e2e_step()
    barrier()
    e_ms = []
    for i in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        e2e_step()
        b.record()
        torch.cuda.synchronize()
        e_ms.append(a.elapsed_time(b))
    e_total = max_over_ranks(float(sum(e_ms)), ws)
    e2e_value = job_throughput(step_flops, args.steps, e_total, ws)

    # ---------------------------------------------------------------- roofline of the dominant kernel
    peaks, peak_src = _peaks()
    kind_ms = {k: v[0] for k, v in prof.items()}
    dominant = max(kind_ms, key=kind_ms.get)
    bwd_ms, bwd_n = prof["bwd_main"]
    fwd_ms, fwd_n = prof["fwd"]
    bwd_flops = args.steps * sum(b for _, b in fl)
    fwd_flops = args.steps * sum(f for f, _ in fl)
    achieved = bwd_flops / (bwd_ms * 1e-3) / 1e12 if bwd_ms > 0 else None
    peak = peaks["bf16_tflops"]
    traffic = _traffic()
    roofline = {"kernel": "bwd_main", "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None, "peak_source": f"{peak_src} bf16 burst",
                "traffic": traffic, "launches": bwd_n, "avg_launch_ms": bwd_ms / max(bwd_n, 1),
                "dominant_by_time": dominant}
    launches = int(sum(n for _, n in prof.values()))

    clocks = clk.summary()
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name + " fwd+bwd, non-causal and causal", "batch": w.batch,
                       "heads": w.num_heads, "head_dim": w.head_dim, "tokens": w.total_tokens,
                       "max_len": w.max_len, "parallelism": f"replicas x{ws}",
                       "l2": "flushed (256 MiB write) before every timed step, outside the events"},
            "pct_of_peak": value / ws / peak * 100.0,
            "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12 if fwd_ms > 0 else None,
            "bwd_tflops": achieved,
            "kernel_ms": {k: v for k, v in kind_ms.items() if v > 0},
            "roofline": roofline, "clocks": clocks, "gpu_launches": launches,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)}}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
