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
    ap.add_argument("--workload", choices=["jagged", "broadcast", "dense", "block", "window", "topk"],
                    default="jagged", help="jagged (default) is the headline step; the others are diagnostic lines")
    ap.add_argument("--window", type=int, default=1024,
                    help="window: keys a query sees (a causal sliding window over the jagged workload)")
    ap.add_argument("--topk", type=int, default=8, help="topk: key blocks of 128 each 256-row query block keeps")
    ap.add_argument("--rope", action="store_true", help="block: with the rotary embedding fused")
    ap.add_argument("--block-batch", type=int, default=1152)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--copy-streams", type=int, default=4,
                    help="copy streams per direction in the end-to-end measurement")
    ap.add_argument("--passes", type=int, default=0,
                    help="passes of the hot path per step (0: enough for --min-timed-s)")
    ap.add_argument("--min-timed-s", type=float, default=5.0,
                    help="timed region length the pass count is chosen for (clock samples every 200 ms)")
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


_SUFFIX = {"jagged": " fwd+bwd, non-causal and causal", "broadcast": " fwd+bwd",
           "dense": " fwd+bwd, plus the GQA 16/4 forward"}


def jagged_family_config(workload):
    """The config keys that describe the workload of a jagged-family line, the
    same for both arms."""
    from variable_length_attention_gb300 import workloads as W
    w = {"jagged": W.jagged(False), "broadcast": W.broadcast(), "dense": W.dense(False)}[workload]
    cfg = {"workload": w.name + _SUFFIX[workload], "batch": w.batch, "heads": w.num_heads,
           "head_dim": w.head_dim, "tokens": w.total_tokens, "max_len": w.max_len}
    if w.nq:
        cfg["nq_broadcast"] = w.nq
    return cfg


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
    """The oracle as the reference arm: each step is a bounded sample of the
    jagged workload (the configuration the metric is quoted on)."""
    if args.workload != "jagged":
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the oracle on the "
                                                                  "jagged workload only"}), flush=True)
        return
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
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(jagged_family_config("jagged"), parallelism=f"replicas x{ws}"),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _plan_ms(job, reps=50):
    """Host planning time of one pass of the hot path: the library's own planners
    (the calls each entry point makes before it enqueues work), on the pass's
    offsets, timed on the host.  With the host copy of the offsets the plan needs
    no device synchronisation and overlaps the previous kernels."""
    import ctypes
    from variable_length_attention_gb300 import jfa as J
    lib = J.load()
    plans = job["plans"]
    if not plans:
        return None
    t0 = time.perf_counter()
    for _ in range(reps):
        for entry in plans:
            if callable(entry):  # a planner with its own signature
                entry(lib)
                continue
            fn, offs, heads, nq, causal, n_cta = entry
            f = getattr(lib, fn)
            n = f(offs.ctypes.data_as(ctypes.c_void_p), len(offs) - 1, heads, nq, int(causal), 1, None, None)
            units = np.empty(4 * max(n, 1), dtype=np.int32)
            start = np.empty(n_cta + 1, dtype=np.int32)
            f(offs.ctypes.data_as(ctypes.c_void_p), len(offs) - 1, heads, nq, int(causal), n_cta,
              units.ctypes.data_as(ctypes.c_void_p), start.ctypes.data_as(ctypes.c_void_p))
    return (time.perf_counter() - t0) * 1e3 / reps


def main():
    args = _args()
    ws, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    import variable_length_attention_gb300 as V

    assert torch.cuda.is_available(), "bench.py needs a GPU"
    dev = torch.device("cuda", local)
    job = build_job(args, dev)
    step, flush = job["step"], torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > L2 (129 MB)
    pass_flops = float(sum(job["flops"].values()))

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        step(job["dev_inputs"])
    barrier()
    # A step is `passes` passes of the hot path, each after an L2 flush, so that
    # the K timed steps last long enough (--min-timed-s) for the clock sampler to
    # see the GPU under load; every pass is timed by its own pair of events.
    if args.passes > 0:
        passes = args.passes
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            step(job["dev_inputs"])
        e1.record()
        torch.cuda.synchronize()
        est = max(e0.elapsed_time(e1) / 3, 1e-3)
        passes = max(1, math.ceil(args.min_timed_s * 1e3 / (args.steps * est)))
        passes = int(max_over_ranks(passes, ws))
    # ---------------------------------------------------------------- timed region (device)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(passes)]
           for _ in range(args.steps)]
    # inside the timed region only the dominant kernel is bracketed by events
    # (every launch is still counted); the per-kernel breakdown comes from
    # separate passes afterwards
    V.jfa_profile_select([job["dominant"]])
    V.jfa_profile_enable(True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        for i in range(args.steps):
            for r in range(passes):
                flush.zero_()  # L2 flush between timed passes, outside the events
                evs[i][r][0].record()
                step(job["dev_inputs"])
                evs[i][r][1].record()
        barrier()
    step_ms = [sum(a.elapsed_time(b) for a, b in row) for row in evs]
    prof = {kind: V.jfa_profile_read(kind) for kind in V.jfa.KERNEL_KINDS}
    V.jfa_profile_enable(False)
    total_ms = max_over_ranks(float(sum(step_ms)), ws)
    ms_per_step = total_ms / args.steps
    median_step = max_over_ranks(float(statistics.median(step_ms)), ws)
    value = job_throughput(pass_flops * passes, args.steps, total_ms, ws)

    # ---------------------------------------------------------------- per-kernel and per-call breakdown
    # Outside the timed region: every kernel kind timed by the library over
    # `steps` passes, then each entry-point call of a pass on its own (CUDA
    # events around the call; the library's events around its kernels), so the
    # causal and non-causal variants are reported separately.
    n_bd = args.steps
    V.jfa_profile_select(None)
    V.jfa_profile_enable(True)
    for i in range(n_bd):
        flush.zero_()
        step(job["dev_inputs"])
    barrier()
    breakdown = {kind: V.jfa_profile_read(kind) for kind in V.jfa.KERNEL_KINDS}
    V.jfa_profile_enable(False)
    calls = {}
    # A ~1 ms spin kernel ahead of each timed call keeps the GPU busy while the
    # host plans and enqueues it, so the events bracket the call's device work
    # (its copies and kernels) and not the host's latency; the host time of
    # the call is measured on its own.
    spin = getattr(torch.cuda, "_sleep", None)
    host_call = {}
    for c in job["calls"]:
        ms_call, ms_main, ms_host = [], [], []
        for i in range(n_bd):
            flush.zero_()
            V.jfa_profile_select([c["main"]])
            V.jfa_profile_enable(True)
            if spin is not None:
                spin(2_000_000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            h0 = time.perf_counter()
            c["run"](job["dev_inputs"])
            ms_host.append((time.perf_counter() - h0) * 1e3)
            b.record()
            torch.cuda.synchronize()
            ms_call.append(a.elapsed_time(b))
            ms_main.append(V.jfa_profile_read(c["main"])[0])
            V.jfa_profile_enable(False)
        host_call[c["name"]] = statistics.median(ms_host)
        mc, mm = statistics.median(ms_call), statistics.median(ms_main)
        ent = {"median_call_ms": mc, "median_kernel_ms": mm, "kernel": c["main"]}
        if job["bound"] == "tensor":
            ent["call_tflops"] = c["flops"] / (mc * 1e-3) / 1e12
            ent["kernel_tflops"] = c["flops"] / (mm * 1e-3) / 1e12 if mm > 0 else None
        else:
            ent["call_gbs"] = c["bytes"] / (mc * 1e-3) / 1e9
            ent["kernel_gbs"] = c["bytes"] / (mm * 1e-3) / 1e9 if mm > 0 else None
        calls[c["name"]] = ent
    V.jfa_profile_select(None)

    # ---------------------------------------------------------------- e2e through host buffers
    # Every pass uploads its inputs from pinned host memory (q, k, v, dO and the
    # offsets), runs, and reads its results back (O, dQ, dK, dV) into pinned host
    # memory.  The copies run on their own copy streams and the kernels on the
    # compute stream, with two slots of device inputs and outputs: pass i+1's
    # upload and pass i-1's read-back overlap pass i's kernels, and a slot is
    # reused only after both its kernels and its read-back are done.  The timed
    # region spans the first upload to the last read-back of `steps` steps of
    # `passes` passes.
    e2e = None
    host_in = job["host_inputs"]
    if host_in is not None:
        s2 = job["new_slot"]()
        d_in = [job["dev_inputs"], [torch.empty_like(t) for t in job["dev_inputs"]]]
        outs = [job["outputs"](0), job["outputs"](s2)]
        o_h = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs[0]] for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in o_h[0])
        comp = torch.cuda.current_stream(dev)
        n_cs = max(1, args.copy_streams)  # tensors are dealt round-robin over the copy streams
        ups = [torch.cuda.Stream(dev) for _ in range(n_cs)]
        downs = [torch.cuda.Stream(dev) for _ in range(n_cs)]
        ran = [torch.cuda.Event(), torch.cuda.Event()]  # the slot's last pass has run
        loaded = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(2)]
        read = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(2)]  # results on the host

        def e2e_run(n):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(comp)
            for st in ups + downs:
                st.wait_stream(comp)
            for i in range(n):
                s = i & 1
                slot = 0 if s == 0 else s2
                pairs_in = list(zip(d_in[s], host_in))
                for c, st in enumerate(ups):
                    with torch.cuda.stream(st):
                        if i >= 2:
                            st.wait_event(ran[s])  # the slot's inputs are no longer read
                        for d, h in pairs_in[c::n_cs]:
                            d.copy_(h, non_blocking=True)
                        loaded[s][c].record(st)
                for ev in loaded[s]:
                    comp.wait_event(ev)
                if i >= 2:
                    for ev in read[s]:  # the slot's outputs have been read back
                        comp.wait_event(ev)
                job["step"](d_in[s], slot)
                ran[s].record(comp)
                pairs_out = list(zip(o_h[s], outs[s]))
                for c, st in enumerate(downs):
                    with torch.cuda.stream(st):
                        st.wait_event(ran[s])
                        for h, d in pairs_out[c::n_cs]:
                            h.copy_(d, non_blocking=True)
                        read[s][c].record(st)
            for st in ups + downs:
                comp.wait_stream(st)
            t1.record(comp)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)

        e2e_run(2)
        barrier()
        e_total = max_over_ranks(float(e2e_run(args.steps * passes)), ws)
        e2e = {"value": job_throughput(pass_flops * passes, args.steps, e_total, ws), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d) * passes, "d2h_bytes_per_step": int(d2h) * passes,
               "ms_per_step": e_total / args.steps, "copy_streams_per_direction": n_cs,
               "overlap": "uploads and read-backs on their own copy streams overlap the neighbouring passes' "
                          "kernels (two slots of device buffers); inputs copied from host every pass "
                          f"({h2d / 2**20:.0f} MiB, larger than L2)"}

    # ---------------------------------------------------------------- roofline of the dominant kernel
    peaks, peak_src = _peaks()
    kind_ms = {k: v[0] for k, v in breakdown.items()}
    dom = job["dominant"]
    dom_ms, dom_n = prof[dom]
    n_passes = args.steps * passes
    if job["bound"] == "tensor":
        achieved = n_passes * job["flops"][dom] / (dom_ms * 1e-3) / 1e12 if dom_ms > 0 else None
        peak, unit, psrc = peaks["bf16_tflops"], "TFLOP/s", f"{peak_src} bf16 burst"
    else:
        achieved = n_passes * job["bytes"][dom] / (dom_ms * 1e-3) / 1e9 if dom_ms > 0 else None
        peak, unit, psrc = peaks["hbm_gbs"], "GB/s", f"{peak_src} HBM copy"
    roofline = {"kernel": dom, "bound": job["bound"], "achieved": achieved, "peak": peak, "unit": unit,
                "frac": (achieved / peak) if achieved else None, "peak_source": psrc,
                "traffic": _traffic() if args.workload == "jagged" else None, "launches": dom_n,
                "avg_launch_ms": dom_ms / max(dom_n, 1), "dominant_by_time": max(kind_ms, key=kind_ms.get)}
    if job["bound"] == "tensor" and achieved:
        roofline["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    per_kind = {k: n_bd * f / (kind_ms[k] * 1e-3) / 1e12 for k, f in job["flops"].items() if kind_ms.get(k)}
    clocks = clk.summary()
    plan_ms = _plan_ms(job)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "median_ms_per_step": median_step,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(job["config"], parallelism=f"replicas x{ws}",
                           l2="flushed (256 MiB write) before every timed pass, outside the events"),
            "passes_per_step": passes,
            "passes_note": "a step is this many passes of the hot path, each after an L2 flush, so that the "
                           "timed region lasts long enough for the clock samples",
            "pct_of_peak": value / ws / peaks["bf16_tflops"] * 100.0,
            "kernel_tflops": per_kind,
            "kernel_frac_by_call": ({n: e["kernel_tflops"] / peaks["bf16_tflops"] for n, e in calls.items()
                                     if e.get("kernel_tflops")} if job["bound"] == "tensor" else
                                    {n: e["kernel_gbs"] / peaks["hbm_gbs"] for n, e in calls.items()
                                     if e.get("kernel_gbs")}),
            "kernel_frac_note": "each entry point's main kernel (the 'calls' entries: non-causal and causal "
                                "separately) as a fraction of the measured bf16 burst peak (HBM copy peak for "
                                "the block kernels)",
            "kernel_ms": {k: v for k, v in kind_ms.items() if v > 0},
            "kernel_ms_note": f"per kind, summed over {n_bd} passes after the timed region",
            "calls": calls,
            "calls_note": f"each entry-point call of a pass alone, median of {n_bd} after an L2 flush: the whole "
                          "call's device time (CUDA events around it, the GPU kept busy while the host enqueues "
                          "it) and its main kernel (the library's events)",
            "host_plan_ms": plan_ms,
            "host_plan_note": "host planning of one pass (every planner call the pass's entry points make), "
                              "timed on the host; it overlaps the previous kernels",
            "host_call_ms": host_call,
            "host_call_note": "host time of each entry-point call (Python binding, planning, enqueue) while the "
                              "GPU is busy, median",
            "roofline": roofline, "clocks": clocks, "gpu_launches": int(sum(n for _, n in prof.values())),
            "e2e": e2e}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and args.workload == "jagged":
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def build_job(args, dev):
    """Inputs, outputs and the step function of one workload.

    ``step(inputs, slot)`` runs one step on the current stream, writing the
    outputs of ``slot``; ``new_slot()`` allocates a further set of outputs (and
    workspaces) and returns its index, so that consecutive steps can keep their
    results apart while earlier ones are still being read back."""
    import variable_length_attention_gb300 as V
    from variable_length_attention_gb300 import workloads as W

    if args.workload in ("jagged", "broadcast", "dense"):
        wls = {"jagged": [W.jagged(False), W.jagged(True)], "broadcast": [W.broadcast()],
               "dense": [W.dense(False), W.dense(True)]}[args.workload]
        w = wls[0]
        offs_h = w.offsets
        # step inputs: q, k, v, dO, then the K, V of a GQA forward (fewer heads) if
        # the workload has one, then the offsets
        host = list(w.tensors("cpu"))
        gqa = [wl for wl in wls if wl.num_kv_heads != w.num_kv_heads]
        if gqa:
            g = gqa[0].tensors("cpu")
            host += [g[1], g[2]]
        host.append(torch.from_numpy(offs_h.copy()))
        host = [t.pin_memory() for t in host]
        dev_in = [t.to(dev) for t in host]
        max_len = w.max_len  # the caller's bound on sequence length, as the interface takes it

        def make_slot():
            calls, outputs = [], []
            for wl in wls:
                o = torch.empty((wl.o_rows, wl.num_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
                lse = torch.empty((wl.num_heads, wl.o_rows), dtype=torch.float32, device=dev)
                grads = None
                if wl.bwd:
                    grads = (torch.empty_like(dev_in[0]), torch.empty_like(dev_in[1]), torch.empty_like(dev_in[2]))
                    outputs += [o, *grads]
                else:
                    outputs.append(o)
                need = max(V.jfa_workspace_size(0, offs_h, wl.batch, wl.nq, wl.num_heads, wl.head_dim, wl.causal,
                                                wl.nq > 0),
                           V.jfa_workspace_size(1, offs_h, wl.batch, wl.nq, wl.num_heads, wl.head_dim, wl.causal,
                                                wl.nq > 0) if wl.bwd else 0)
                calls.append((wl, o, lse, grads, torch.empty(need, dtype=torch.uint8, device=dev)))
            return calls, outputs

        slots = [make_slot()]

        def new_slot():
            slots.append(make_slot())
            return len(slots) - 1

        def step(inp, slot=0):
            q, k, v, do, offs = inp[0], inp[1], inp[2], inp[3], inp[-1]
            for wl, o, lse, grads, wsb in slots[slot][0]:
                kk, vv = (inp[4], inp[5]) if wl.num_kv_heads != w.num_kv_heads else (k, v)
                V.jfa_fwd(q, kk, vv, offs, offs_h, max_len=max_len, causal=wl.causal, nq_broadcast=wl.nq, out=o,
                          lse=lse, workspace=wsb)
                if grads is not None:
                    V.jfa_bwd(q, kk, vv, o, do, lse, offs, offs_h, max_len=max_len, causal=wl.causal,
                              nq_broadcast=wl.nq, dq=grads[0], dk=grads[1], dv=grads[2], workspace=wsb)

        fl = [W.flops(wl) for wl in wls]
        flops = {"fwd": float(sum(f for f, _ in fl)),
                 "bwd_main": float(sum(b for (_, b), wl in zip(fl, wls) if wl.bwd))}
        cfg = jagged_family_config(args.workload)

        def one_call(i, which):
            def run(inp, slot=0):
                q, k, v, do, offs = inp[0], inp[1], inp[2], inp[3], inp[-1]
                wl, o, lse, grads, wsb = slots[slot][0][i]
                kk, vv = (inp[4], inp[5]) if wl.num_kv_heads != w.num_kv_heads else (k, v)
                if which == "fwd":
                    V.jfa_fwd(q, kk, vv, offs, offs_h, max_len=max_len, causal=wl.causal, nq_broadcast=wl.nq,
                              out=o, lse=lse, workspace=wsb)
                else:
                    V.jfa_bwd(q, kk, vv, o, do, lse, offs, offs_h, max_len=max_len, causal=wl.causal,
                              nq_broadcast=wl.nq, dq=grads[0], dk=grads[1], dv=grads[2], workspace=wsb)
            return run

        calls, plans = [], []
        for i, (wl, (f_fwd, f_bwd)) in enumerate(zip(wls, fl)):
            tag = ("_causal" if wl.causal else "") + ("_gqa" if wl.num_kv_heads != wl.num_heads else "")
            calls.append({"name": "fwd" + tag, "run": one_call(i, "fwd"), "flops": float(f_fwd), "main": "fwd"})
            plans.append(("jfa_plan_fwd", offs_h, wl.num_heads, wl.nq, wl.causal, 1))
            if wl.bwd:
                calls.append({"name": "bwd" + tag, "run": one_call(i, "bwd"), "flops": float(f_bwd),
                              "main": "bwd_main"})
                plans.append(("jfa_plan_bwd", offs_h, wl.num_kv_heads, wl.nq, wl.causal, 1))
        return {"step": step, "new_slot": new_slot, "outputs": lambda slot: slots[slot][1], "dev_inputs": dev_in,
                "host_inputs": host, "flops": flops, "bytes": {}, "dominant": "bwd_main", "bound": "tensor",
                "config": cfg, "calls": calls, "plans": plans}

    if args.workload in ("window", "topk"):
        return build_sparse_job(args, dev)

    # block-diagonal: inputs drawn on the device (the full workload is 4.8 GB per tensor)
    w = W.block(args.head_dim, batch=args.block_batch)
    offs_h = w.offsets
    dev_in = list(w.tensors(str(dev))) + [torch.from_numpy(offs_h.copy()).to(dev)]
    slots = []

    def new_slot():
        o = torch.empty_like(dev_in[0])
        grads = [torch.empty_like(dev_in[i]) for i in range(3)]
        # the rotary variants also hold rotated copies of q and k (op 6 instead of 2)
        wsb = torch.empty(V.jfa_workspace_size(6 if args.rope else 2, offs_h, w.batch, 0, w.num_heads, w.head_dim,
                                               0, 0), dtype=torch.uint8, device=dev)
        slots.append((o, grads, wsb))
        return len(slots) - 1

    new_slot()


    f, b = W.flops(w)
    t_bytes = dev_in[0].numel() * 2

    rope = None
    if args.rope:  # rotate-half tables, angle p * 10000^(-2i/D), fp32
        ang = np.arange(w.max_len)[:, None] * 10000.0 ** (-2.0 * np.arange(w.head_dim // 2) / w.head_dim)[None, :]
        rope = (torch.from_numpy(np.cos(ang)).float().to(dev), torch.from_numpy(np.sin(ang)).float().to(dev))

    def run_fwd(inp, slot=0):
        q, k, v, do, offs = inp
        V.block_attn_fwd(q, k, v, offs, offs_h, max_len=w.max_len, out=slots[slot][0], workspace=slots[slot][2],
                         rope=rope)

    def run_bwd(inp, slot=0):
        q, k, v, do, offs = inp
        o, grads, wsb = slots[slot]
        V.block_attn_bwd(q, k, v, o, do, offs, offs_h, max_len=w.max_len, dq=grads[0], dk=grads[1], dv=grads[2],
                         workspace=wsb, rope=rope)

    def step(inp, slot=0):
        run_fwd(inp, slot)
        run_bwd(inp, slot)

    calls = [{"name": "block_fwd", "run": run_fwd, "flops": float(f), "bytes": 4.0 * t_bytes, "main": "block_fwd"},
             {"name": "block_bwd", "run": run_bwd, "flops": float(b), "bytes": 7.0 * t_bytes, "main": "block_bwd"}]
    host = None
    if 4 * t_bytes <= (4 << 30):  # e2e only when the inputs fit a modest pinned host buffer
        host = [t.cpu().pin_memory() for t in dev_in]
    return {"step": step, "new_slot": new_slot, "outputs": lambda slot: [slots[slot][0]] + slots[slot][1],
            "dev_inputs": dev_in, "host_inputs": host,
            "flops": {"block_fwd": float(f), "block_bwd": float(b)},
            "bytes": {"block_fwd": 4.0 * t_bytes, "block_bwd": 7.0 * t_bytes}, "dominant": "block_bwd",
            "bound": "hbm", "calls": calls, "plans": [],
            "config": {"workload": w.name + (" rotary" if args.rope else "") + " fwd+bwd", "batch": w.batch,
                       "heads": w.num_heads, "head_dim": w.head_dim, "tokens": w.total_tokens, "block": 64}}



def build_sparse_job(args, dev):
    """Diagnostic lines on the jagged workload's inputs: a causal sliding window
    (forward + backward over the pairs inside the window), or the two-stage
    block-sparse forward (selection + attention over the chosen blocks)."""
    import variable_length_attention_gb300 as V
    from variable_length_attention_gb300 import workloads as W

    w = W.jagged(False)
    offs_h = w.offsets
    host = [t.pin_memory() for t in w.tensors("cpu")] + [torch.from_numpy(offs_h.copy()).pin_memory()]
    dev_in = [t.to(dev) for t in host]
    o = torch.empty((w.o_rows, w.num_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.num_heads, w.o_rows), dtype=torch.float32, device=dev)
    grads = [torch.empty_like(dev_in[i]) for i in range(3)]
    plans = []  # host planners a pass calls (timed for host_plan_ms)
    if args.workload == "window":
        left = args.window - 1
        L = w.lengths.astype(np.int64)
        pairs = sum(int(np.sum(np.minimum(np.arange(n) + 1, args.window))) for n in L) * w.num_heads
        f = 4.0 * w.head_dim * pairs
        wsb = torch.empty(max(V.jfa_workspace_size(0, offs_h, w.batch, 0, w.num_heads, w.head_dim, 0, 0),
                              V.jfa_workspace_size(1, offs_h, w.batch, 0, w.num_heads, w.head_dim, 0, 0)),
                          dtype=torch.uint8, device=dev)

        def run_fwd(inp, slot=0):
            V.jfa_fwd(inp[0], inp[1], inp[2], inp[-1], offs_h, max_len=w.max_len, window=(left, 0), out=o,
                      lse=lse, workspace=wsb)

        def run_bwd(inp, slot=0):
            V.jfa_bwd(inp[0], inp[1], inp[2], o, inp[3], lse, inp[-1], offs_h, max_len=w.max_len, window=(left, 0),
                      dq=grads[0], dk=grads[1], dv=grads[2], workspace=wsb)

        calls = [{"name": "fwd_window", "run": run_fwd, "flops": f, "main": "fwd"},
                 {"name": "bwd_window", "run": run_bwd, "flops": 2.5 * f, "main": "bwd_main"}]

        def plan_window(which):
            def run(lib):
                import ctypes
                po = offs_h.ctypes.data_as(ctypes.c_void_p)
                heads = w.num_kv_heads if which else w.num_heads  # backward units run over the K/V heads
                n = lib.jfa_plan_window(which, po, w.batch, heads, left, 0, 1, None, None)
                units = np.empty(4 * max(n, 1), dtype=np.int32)
                start = np.empty(2, dtype=np.int32)
                lib.jfa_plan_window(which, po, w.batch, heads, left, 0, 1,
                                    units.ctypes.data_as(ctypes.c_void_p), start.ctypes.data_as(ctypes.c_void_p))
            return run

        plans = [plan_window(0), plan_window(1)]
        flops = {"fwd": f, "bwd_main": 2.5 * f}
        outputs = [o] + grads
        cfg = {"workload": f"{w.name} causal sliding window of {args.window} keys fwd+bwd", "batch": w.batch,
               "heads": w.num_heads, "head_dim": w.head_dim, "tokens": w.total_tokens, "window": args.window}
        dominant = "bwd_main"
    else:
        k_sel = args.topk
        rows = V.jfa_topk_rows(offs_h, w.num_heads)
        sel = torch.empty((rows, k_sel), dtype=torch.int32, device=dev)
        ws1 = torch.empty(V.jfa_workspace_size(4, offs_h, w.batch, 0, w.num_heads, w.head_dim, 0, 0),
                          dtype=torch.uint8, device=dev)
        ws2 = torch.empty(V.jfa_workspace_size(5, offs_h, w.batch, 0, w.num_heads, w.head_dim, 0, 0),
                          dtype=torch.uint8, device=dev)
        V.jfa_topk_select(dev_in[0], dev_in[1], dev_in[-1], offs_h, topk=k_sel, selection=sel, workspace=ws1)
        # valid pairs: each query block's rows times the keys of its chosen blocks
        chosen = sel.cpu().numpy()
        pairs, u = 0, 0
        for b in range(w.batch):
            L = int(w.lengths[b])
            for _h in range(w.num_heads):
                for m in range(-(-L // 256)):
                    nrow = min(256, L - 256 * m)
                    keys = sum(min(128, L - 128 * int(j)) for j in chosen[u] if j >= 0)
                    pairs += nrow * keys
                    u += 1
        f = 4.0 * w.head_dim * pairs

        def run_select(inp, slot=0):
            V.jfa_topk_select(inp[0], inp[1], inp[-1], offs_h, topk=k_sel, selection=sel, workspace=ws1)

        def run_fwd(inp, slot=0):
            V.jfa_fwd_topk(inp[0], inp[1], inp[2], inp[-1], sel, offs_h, topk=k_sel, out=o, lse=lse, workspace=ws2)

        calls = [{"name": "topk_select", "run": run_select, "flops": 0.0, "main": "topk_select"},
                 {"name": "fwd_topk", "run": run_fwd, "flops": f, "main": "fwd"}]
        flops = {"fwd": f}
        outputs = [o]
        cfg = {"workload": f"{w.name} block-sparse top-{k_sel} of 128-key blocks per 256-row query block, fwd "
                           "(selection + attention)", "batch": w.batch, "heads": w.num_heads,
               "head_dim": w.head_dim, "tokens": w.total_tokens, "topk": k_sel}
        dominant = "fwd"

    def step(inp, slot=0):
        for c in calls:
            c["run"](inp, slot)

    return {"step": step, "new_slot": lambda: 0, "outputs": lambda slot: outputs, "dev_inputs": dev_in,
            "host_inputs": None, "flops": flops, "bytes": {}, "dominant": dominant, "bound": "tensor",
            "config": cfg, "calls": calls, "plans": plans}


if __name__ == "__main__":
    main()
