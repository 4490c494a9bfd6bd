#!/usr/bin/env python3
"""Benchmark of the fused flash-attention training step on GB300.

One step = the whole op over one batch of seeded synthetic input: forward
(O, LSE) then backward (D precompute, dQ/dK/dV, dQ convert). Workloads that
accumulate dK/dV run the accumulating variant, which also reads the chunk's own
K/V rows back out of the accumulator in the same kernel. Throughput is mask- and
causal-aware TFLOP/s: 4*D flops per visible (query head, query, key) triple in
the forward and 10*D in the backward; skipped or masked pairs are not counted.

Prints ONE JSON line (rank 0). `--impl reference` times the fp64 CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from backward_adapter_gb300 import workloads as wl  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, mask-aware FLOPs) and % of GB300 tensor peak"
DEFAULT_WORKLOAD = wl.CAUSAL_LM.name
L2_FLUSH_BYTES = 256 << 20  # > 129 MB of L2


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.BY_NAME))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="bitwise reproducible dQ (partials added in a fixed key-tile order)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------------------------
# peaks, clocks, traffic
# ---------------------------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.out.close()
        with open(self.path) as f:
            summary = parse_clock_samples(f)
        os.unlink(self.path)
        return summary


def parse_clock_samples(lines):
    """Summarise nvidia-smi rows of ClockSampler.FIELDS: the median SM clock of the busy samples
    (above half the highest seen), the maximum clock, and every throttle reason seen active."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
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
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    busy = [x for x in sm if x > 0.5 * max(sm)] or sm
    return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
            "samples": len(sm)}


def source_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(kernel_key: str, source_file: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha(source_file)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == kernel_key and parts[2] == sha:
                return float(parts[1])
    return None


# ---------------------------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs the same workload on its own GPU)
# ---------------------------------------------------------------------------------------------

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float, device: str = "cuda") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, rank_ms: float, device: str = "cuda"):
    """Replicas: (slowest rank's ms per step, every rank's work over that time in TFLOP/s)."""
    ms = max_over_ranks(world, rank_ms, device)
    return ms, world * flops_per_rank / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (the reported CPU baseline and the reference arm)
# ---------------------------------------------------------------------------------------------

def oracle_sample(w: wl.Workload, inputs: dict, n_heads: int):
    """Run the fp64 oracle fwd+bwd on the first n_heads query heads; return (seconds, flops, desc)."""
    from oracle import attention as ref
    G = w.Hq // w.Hkv
    n_heads = max(1, min(n_heads, w.Hq))
    kv = sorted({h // G for h in range(n_heads)})
    q, do = inputs["q"][:1, :n_heads], inputs["do"][:1, :n_heads]
    mask = inputs["mask"]
    if mask is not None:
        mask = mask[:1]
    t0 = time.perf_counter()
    if w.kv_format == "q8_0":   # the cache is read as its values, inside the timed sample
        k = ref.dequantize_q8_0(inputs["k_q8"][0][:1, kv], inputs["k_q8"][1][:1, kv])
        v = ref.dequantize_q8_0(inputs["v_q8"][0][:1, kv], inputs["v_q8"][1][:1, kv])
    else:
        k, v = inputs["k"][:1, kv], inputs["v"][:1, kv]
    # the sample keeps the GQA mapping: n_heads query heads over their kv heads
    if len(kv) * G != n_heads:
        k = np.repeat(k, G, axis=1)[:, :n_heads]
        v = np.repeat(v, G, axis=1)[:, :n_heads]
    ref.backward(q, k, v, do, w.scale, mask, inputs["mask_kind"], w.causal, w.q_offset, w.window)
    dt = time.perf_counter() - t0
    pairs_per_head = wl.visible_pairs(w.with_(B=1, Hq=1, Hkv=1))
    fl = 14.0 * w.D * pairs_per_head * n_heads
    desc = f"oracle fwd+bwd on batch 0, query heads 0..{n_heads - 1} of {w.Hq} (fp64 numpy)"
    return dt, fl, desc


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return 0
    w = wl.BY_NAME[args.workload]
    inputs = wl.make_inputs(w)
    heads = 1
    for _ in range(args.warmup):
        oracle_sample(w, inputs, heads)
    times, fl, desc = [], 0.0, ""
    for _ in range(args.steps):
        dt, fl, desc = oracle_sample(w, inputs, heads)
        times.append(dt)
    mean = statistics.mean(times)
    value = fl / mean / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
# the GPU path
# ---------------------------------------------------------------------------------------------

def gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9 if ms > 0 else None


def run_ours(args):
    import torch

    from backward_adapter_gb300 import fa_train as ft

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.BY_NAME[args.workload]
    inputs = wl.make_inputs(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    es = 2 if w.dtype == "bf16" else 4

    q8 = w.kv_format == "q8_0"
    host = {n: torch.from_numpy(inputs[n]).to(dt).pin_memory() for n in (("q", "do") if q8 else ("q", "k", "v", "do"))}
    if w.kv_format == "f16":   # an fp16 K/V cache, read in place (the library casts it for the tensor cores)
        for n in ("k", "v"):
            host[n] = torch.from_numpy(inputs[n]).to(torch.float16).pin_memory()
    if q8:   # the K/V cache in its own format: int8 values and fp16 scales, read in place
        for n in ("k", "v"):
            qv, dv_ = inputs[n + "_q8"]
            host[n + "_q"] = torch.from_numpy(qv).pin_memory()
            host[n + "_d"] = torch.from_numpy(dv_).pin_memory()
    if inputs["mask"] is not None:
        host["mask"] = torch.from_numpy(inputs["mask"]).pin_memory()
    d = {n: t.to(dev) for n, t in host.items()}
    mask = d.get("mask")
    kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset, window=w.window, deterministic=args.deterministic)
    kv_format = {"q8_0": ft.FA_KV_Q8_0, "f16": ft.FA_KV_F16}.get(w.kv_format, ft.FA_KV_DTYPE)
    p = ft.make_params(d["q"], d["k_q" if q8 else "k"], mask, kv_format=kv_format, **kw)
    ws_f = torch.empty(max(ft.fwd_workspace_size(p), 1), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(max(ft.bwd_workspace_size(p), 1), dtype=torch.uint8, device=dev)
    o = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
    dq = torch.empty_like(d["q"])
    if w.accum:
        dk = torch.from_numpy(inputs["dk_acc"]).to(dev)
        dv = torch.from_numpy(inputs["dv_acc"]).to(dev)
        # the chunk's own K/V rows (the last Sq keys of the window) are read back from the
        # accumulator in the same kernel (fused SET_ROWS backward)
        rows_shape = (w.B, w.Hkv, w.Sq, w.D)
        dk_rows = torch.empty(rows_shape, dtype=d["q"].dtype, device=dev)
        dv_rows = torch.empty(rows_shape, dtype=d["q"].dtype, device=dev)
    else:
        kv_shape = (w.B, w.Hkv, w.Sk, w.D)
        dk, dv = torch.empty(kv_shape, dtype=dt, device=dev), torch.empty(kv_shape, dtype=dt, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fkw = {k_: v_ for k_, v_ in kw.items() if k_ != "deterministic"}

    def fwd_call(src, o_, lse_):
        if q8:
            return ft.fwd_q8(src["q"], src["k_q"], src["k_d"], src["v_q"], src["v_d"], src.get("mask"), out=o_,
                             lse=lse_, workspace=ws_f, **fkw)
        return ft.fwd(src["q"], src["k"], src["v"], src.get("mask"), out=o_, lse=lse_, workspace=ws_f, **kw)

    def bwd_call(src, o_, lse_, dq_, dk_, dv_):
        if q8:
            kv = (src["k_q"], src["k_d"], src["v_q"], src["v_d"])
            if w.accum:
                ft.bwd_q8(src["q"], *kv, o_, lse_, src["do"], src.get("mask"), dq=dq_, dk_acc=dk_, dv_acc=dv_,
                          workspace=ws_b, **kw)
            else:
                ft.bwd_q8(src["q"], *kv, o_, lse_, src["do"], src.get("mask"), dq=dq_, dk=dk_, dv=dv_,
                          workspace=ws_b, **kw)
        elif w.accum:
            ft.bwd_accum_rows(src["q"], src["k"], src["v"], o_, lse_, src["do"], dk_, dv_, w.q_offset, w.Sq,
                              src.get("mask"), dq=dq_, dk_rows=dk_rows, dv_rows=dv_rows, workspace=ws_b, **kw)
        else:
            ft.bwd(src["q"], src["k"], src["v"], o_, lse_, src["do"], src.get("mask"), dq=dq_, dk=dk_, dv=dv_,
                   workspace=ws_b, **kw)

    def step(src):
        fwd_call(src, o, lse)
        bwd_call(src, o, lse, dq, dk, dv)

    fl = wl.flops(w)
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()

    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ev = [(ev(), ev()) for _ in range(K)]
    kern = {kid: [(ev(), ev()) for _ in range(K)] for kid in (ft.FA_KERNEL_FWD, ft.FA_KERNEL_BWD_MAIN,
                                                              ft.FA_KERNEL_BWD_DSUM, ft.FA_KERNEL_BWD_DQ_CONVERT)}
    # torch creates the CUDA event lazily at its first record(): materialise every handle
    # before the library is asked to record it
    for evs in kern.values():
        for a_, b_ in evs:
            a_.record()
            b_.record()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = ft.profile_launch_count()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.zero_()                      # evict L2 between timed steps (not inside the step events)
        for kid, evs in kern.items():
            ft.profile_set_events(kid, *evs[i])
        step_ev[i][0].record()
        step(d)
        step_ev[i][1].record()
    torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall
    launches = ft.profile_launch_count() - launches0
    for kid in kern:
        ft.profile_set_events(kid, None, None)
    clock_info = clocks.stop()

    step_ms = [a.elapsed_time(b) for a, b in step_ev]

    def mean_or_zero(evs):
        try:
            return statistics.mean(a.elapsed_time(b) for a, b in evs)
        except (RuntimeError, ValueError):  # this path does not launch that kernel
            return 0.0

    kern_ms = {kid: mean_or_zero(evs) for kid, evs in kern.items()}
    mean_ms, value = job_tflops(world, fl["total"], statistics.mean(step_ms))

    peaks = load_peaks()
    fwd_ms, bwd_main_ms = kern_ms[ft.FA_KERNEL_FWD], kern_ms[ft.FA_KERNEL_BWD_MAIN]
    dominant = "bwd_main" if bwd_main_ms >= fwd_ms else "fwd"
    dom_ms = bwd_main_ms if dominant == "bwd_main" else fwd_ms
    dom_flops = fl["bwd"] if dominant == "bwd_main" else fl["fwd"]
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    rows = w.B * w.Hq * w.Sq
    dsum_bytes = rows * w.D * es * 2 + rows * 4 + rows * w.D * 4
    dqconv_bytes = rows * w.D * 4 + rows * w.D * es
    csrc = os.path.join(ROOT, "backward_adapter_gb300", "csrc")
    dom_src = os.path.join(csrc, "fa_tc_bwd.cu" if dominant == "bwd_main" else "fa_tc_fwd.cu")
    traffic = measured_traffic(dominant, dom_src) if os.path.exists(dom_src) else None

    # End to end through the public API from pinned host buffers: every step copies its inputs
    # host -> device and its results (dQ, dK, dV) device -> host. Copies run on a second stream
    # into double-buffered device inputs, so step i+1's inputs arrive while step i computes.
    out_host = [{"dq": torch.empty_like(dq, device="cpu").pin_memory(),
                 "dk": torch.empty_like(dk, device="cpu").pin_memory(),
                 "dv": torch.empty_like(dv, device="cpu").pin_memory()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())
    bufs = [d, {n: torch.empty_like(t) for n, t in d.items()}]
    outs = [(dq, dk, dv), (torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv))]
    fwd_outs = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
    if w.accum:
        outs[1][1].copy_(dk)
        outs[1][2].copy_(dv)
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()        # host -> device
    copy_out = torch.cuda.Stream()    # device -> host (both directions at once)
    E = max(1, args.e2e_steps)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    in_ready = [ev(), ev()]
    done = [ev(), ev()]
    read_back = [ev(), ev()]
    e0.record(comp)
    copy.wait_event(e0)
    for i in range(E):
        sl = i % 2
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(done[sl])          # step i-2 has finished with this buffer set
            for n, t in host.items():
                bufs[sl][n].copy_(t, non_blocking=True)
            in_ready[sl].record(copy)
        comp.wait_event(in_ready[sl])
        if i >= 2:
            comp.wait_event(read_back[sl])          # step i-2's results have been read back
        src = bufs[sl]
        o_, lse_ = fwd_call(src, fwd_outs[sl][0], fwd_outs[sl][1])
        dq_, dk_, dv_ = outs[sl]
        bwd_call(src, o_, lse_, dq_, dk_, dv_)
        done[sl].record(comp)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(done[sl])
            out_host[sl]["dq"].copy_(dq_, non_blocking=True)
            out_host[sl]["dk"].copy_(dk_, non_blocking=True)
            out_host[sl]["dv"].copy_(dv_, non_blocking=True)
            read_back[sl].record(copy_out)
    last = ev()
    last.record(copy_out)
    comp.wait_event(last)
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms, e2e_value = job_tflops(world, fl["total"], e0.elapsed_time(e1) / E)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # grow the sample one GQA group at a time until ~10 s of oracle work (or every head)
        G = w.Hq // w.Hkv
        heads = G
        dt_cpu, fl_cpu, desc = oracle_sample(w, inputs, heads)
        while dt_cpu < 10.0 and heads < w.Hq:
            heads = min(w.Hq, max(heads + G, int(heads * 10.0 / max(dt_cpu, 1e-3)) // G * G))
            dt_cpu, fl_cpu, desc = oracle_sample(w, inputs, heads)
        cpu = {"value": fl_cpu / dt_cpu / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": desc, "seconds": dt_cpu}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                   "causal": w.causal, "q_offset": w.q_offset, "window": w.window, "mask": w.mask, "accum": w.accum,
                   "rows_read_back": [w.q_offset, w.Sq] if w.accum and not q8 else None,
                   "kv_format": w.kv_format,
                   "deterministic": bool(args.deterministic),
                   "visible_pairs": fl["pairs"], "gflop_per_step": fl["total"] / 1e9,
                   "l2": "flushed (256 MiB write) between timed steps, outside the step events",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / peaks["bf16_tflops"],
        "fwd_tflops": fl["fwd"] / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": fl["bwd"] / ((bwd_main_ms + kern_ms[ft.FA_KERNEL_BWD_DSUM] +
                                    kern_ms[ft.FA_KERNEL_BWD_DQ_CONVERT]) * 1e-3) / 1e12,
        "kernel_ms": {"fwd": fwd_ms, "bwd_main": bwd_main_ms, "bwd_dsum": kern_ms[ft.FA_KERNEL_BWD_DSUM],
                      "bwd_dq_convert": kern_ms[ft.FA_KERNEL_BWD_DQ_CONVERT]},
        "hbm_passes_gbs": {"bwd_dsum": gbs(dsum_bytes, kern_ms[ft.FA_KERNEL_BWD_DSUM]),
                           "bwd_dq_convert": gbs(dqconv_bytes, kern_ms[ft.FA_KERNEL_BWD_DQ_CONVERT]),
                           "peak": peaks["hbm_gbs"]},
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 dense burst",
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "copies": "pinned host buffers; inputs and results on their own streams, double-buffered"},
        "gpu_launches": launches,
        "wall_s_timed_region": t_wall,
        "clocks": clock_info,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
