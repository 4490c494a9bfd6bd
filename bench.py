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
    ap.add_argument("--workload-steps", type=int, default=30,
                    help="timed steps of each of the other workloads in by_workload")
    ap.add_argument("--no-by-workload", action="store_true")
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


KERNELS = ("fwd", "bwd_main", "bwd_dsum", "bwd_dq_convert", "mask_classify")


def stats(ms):
    """mean, median and min of a list of times (ms); None when there are none."""
    if not ms:
        return None
    return {"mean": statistics.mean(ms), "median": statistics.median(ms), "min": min(ms)}


class Prepared:
    """Device inputs, outputs and the two public-API calls of one step of a workload."""

    def __init__(self, ft, torch, w, dev, deterministic=False):
        self.w = w
        inputs = wl.make_inputs(w)
        self.inputs = inputs
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.es = 2 if w.dtype == "bf16" else 4
        self.q8 = q8 = w.kv_format == "q8_0"
        host = {n: torch.from_numpy(inputs[n]).to(dt).pin_memory()
                for n in (("q", "do") if q8 else ("q", "k", "v", "do"))}
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
        self.host = host
        self.d = d = {n: t.to(dev) for n, t in host.items()}
        self.kw = kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset, window=w.window,
                            deterministic=deterministic)
        kv_format = {"q8_0": ft.FA_KV_Q8_0, "f16": ft.FA_KV_F16}.get(w.kv_format, ft.FA_KV_DTYPE)
        p = ft.make_params(d["q"], d["k_q" if q8 else "k"], d.get("mask"), kv_format=kv_format, **kw)
        self.ws_f = torch.empty(max(ft.fwd_workspace_size(p), 1), dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(max(ft.bwd_workspace_size(p), 1), dtype=torch.uint8, device=dev)
        self.o = torch.empty_like(d["q"])
        self.lse = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(d["q"])
        self.dk_rows = self.dv_rows = None
        if w.accum:
            self.dk = torch.from_numpy(inputs["dk_acc"]).to(dev)
            self.dv = torch.from_numpy(inputs["dv_acc"]).to(dev)
            # the chunk's own K/V rows (the last Sq keys of the window) are read back from the
            # accumulator in the same kernel (fused SET_ROWS backward)
            rows_shape = (w.B, w.Hkv, w.Sq, w.D)
            self.dk_rows = torch.empty(rows_shape, dtype=d["q"].dtype, device=dev)
            self.dv_rows = torch.empty(rows_shape, dtype=d["q"].dtype, device=dev)
        else:
            kv_shape = (w.B, w.Hkv, w.Sk, w.D)
            self.dk = torch.empty(kv_shape, dtype=dt, device=dev)
            self.dv = torch.empty(kv_shape, dtype=dt, device=dev)
        self.ft = ft

    def fwd_call(self, src, o_, lse_):
        ft, w = self.ft, self.w
        fkw = {k_: v_ for k_, v_ in self.kw.items() if k_ != "deterministic"}
        if self.q8:
            return ft.fwd_q8(src["q"], src["k_q"], src["k_d"], src["v_q"], src["v_d"], src.get("mask"), out=o_,
                             lse=lse_, workspace=self.ws_f, **fkw)
        return ft.fwd(src["q"], src["k"], src["v"], src.get("mask"), out=o_, lse=lse_, workspace=self.ws_f,
                      **self.kw)

    def bwd_call(self, src, o_, lse_, dq_, dk_, dv_):
        ft, w, kw = self.ft, self.w, self.kw
        if self.q8:
            kv = (src["k_q"], src["k_d"], src["v_q"], src["v_d"])
            if w.accum:
                ft.bwd_q8(src["q"], *kv, o_, lse_, src["do"], src.get("mask"), dq=dq_, dk_acc=dk_, dv_acc=dv_,
                          workspace=self.ws_b, **kw)
            else:
                ft.bwd_q8(src["q"], *kv, o_, lse_, src["do"], src.get("mask"), dq=dq_, dk=dk_, dv=dv_,
                          workspace=self.ws_b, **kw)
        elif w.accum:
            ft.bwd_accum_rows(src["q"], src["k"], src["v"], o_, lse_, src["do"], dk_, dv_, w.q_offset, w.Sq,
                              src.get("mask"), dq=dq_, dk_rows=self.dk_rows, dv_rows=self.dv_rows,
                              workspace=self.ws_b, **kw)
        else:
            ft.bwd(src["q"], src["k"], src["v"], o_, lse_, src["do"], src.get("mask"), dq=dq_, dk=dk_, dv=dv_,
                   workspace=self.ws_b, **kw)

    def step(self):
        self.fwd_call(self.d, self.o, self.lse)
        self.bwd_call(self.d, self.o, self.lse, self.dq, self.dk, self.dv)


def timed_steps(torch, ft, prep, K, W, flush, kernel_reps=None):
    """W untimed steps, then K timed ones with the L2 flushed before each (outside the events).
    The step times come from a pass with no per-kernel events in the stream (an event recorded
    between two of the library's kernels would keep the second from starting under the first's
    tail); a second pass of kernel_reps steps records the per-kernel events.
    Returns (per-step ms list, {kernel: per-step ms list}, library launches in the K steps)."""
    for _ in range(W):
        prep.step()
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ev = [(ev(), ev()) for _ in range(K)]
    torch.cuda.synchronize()
    launches0 = ft.profile_launch_count()
    for i in range(K):
        flush.zero_()                      # evict L2 between timed steps (not inside the step events)
        step_ev[i][0].record()
        prep.step()
        step_ev[i][1].record()
    torch.cuda.synchronize()
    launches = ft.profile_launch_count() - launches0
    step_ms = [a.elapsed_time(b) for a, b in step_ev]

    R = K if kernel_reps is None else max(1, min(K, kernel_reps))
    kids = {"fwd": ft.FA_KERNEL_FWD, "bwd_main": ft.FA_KERNEL_BWD_MAIN, "bwd_dsum": ft.FA_KERNEL_BWD_DSUM,
            "bwd_dq_convert": ft.FA_KERNEL_BWD_DQ_CONVERT, "mask_classify": ft.FA_KERNEL_MASK_CLASSIFY}
    kstep = [(ev(), ev()) for _ in range(R)]
    kern = {name: [(ev(), ev()) for _ in range(R)] for name in kids}
    # torch creates the CUDA event lazily at its first record(): materialise every handle
    # before the library is asked to record it
    for evs in kern.values():
        for a_, b_ in evs:
            a_.record()
            b_.record()
    torch.cuda.synchronize()
    for i in range(R):
        flush.zero_()
        for name, evs in kern.items():
            ft.profile_set_events(kids[name], *evs[i])
        kstep[i][0].record()
        prep.step()
        kstep[i][1].record()
    torch.cuda.synchronize()
    for kid in kids.values():
        ft.profile_set_events(kid, None, None)
    kern_ms = {}
    for name, evs in kern.items():
        # a pair the library recorded during step i starts inside that step; a pair it never
        # recorded still holds its materialising record from before the timed steps (this path
        # does not launch that kernel)
        kern_ms[name] = [a.elapsed_time(b) for (a, b), (s0, _) in zip(evs, kstep) if s0.elapsed_time(a) >= 0.0]
    return step_ms, kern_ms, launches


def workload_summary(w, fl, step_ms, kern_ms, peak):
    """One workload's line: step, forward and backward times (mean / median / min), TFLOP/s on the
    median and its fraction of the dense bf16 peak."""
    st = stats(step_ms)
    ks = {n: stats(v) for n, v in kern_ms.items() if v}
    bwd = [sum(x) for x in zip(*(kern_ms[n] for n in ("bwd_main", "bwd_dsum", "bwd_dq_convert") if kern_ms[n]))]
    out = {"config": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D, "dtype": w.dtype,
                      "causal": w.causal, "q_offset": w.q_offset, "window": w.window, "mask": w.mask,
                      "accum": w.accum, "kv_format": w.kv_format},
           "visible_pairs": fl["pairs"], "gflop_per_step": fl["total"] / 1e9,
           "step_ms": st, "kernel_ms": ks,
           "tflops": fl["total"] / (st["median"] * 1e-3) / 1e12,
           "frac_of_peak": fl["total"] / (st["median"] * 1e-3) / 1e12 / peak}
    if ks.get("fwd"):
        out["fwd_tflops"] = fl["fwd"] / (ks["fwd"]["median"] * 1e-3) / 1e12
    if bwd:
        out["bwd_tflops"] = fl["bwd"] / (statistics.median(bwd) * 1e-3) / 1e12
    return out


def run_ours(args):
    import torch

    from backward_adapter_gb300 import fa_train as ft

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.BY_NAME[args.workload]
    prep = Prepared(ft, torch, w, dev, deterministic=args.deterministic)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fl = wl.flops(w)
    peaks = load_peaks()

    clocks = ClockSampler(local)
    clocks.start()
    K = args.steps
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    step_ms, kern_ms, launches = timed_steps(torch, ft, prep, K, args.warmup, flush, kernel_reps=50)
    barrier(world)
    t_wall = time.perf_counter() - t_wall
    clock_info = clocks.stop()

    mean_ms, value = job_tflops(world, fl["total"], statistics.mean(step_ms))

    def mean_or_zero(v):
        return statistics.mean(v) if v else 0.0

    fwd_ms, bwd_main_ms = mean_or_zero(kern_ms["fwd"]), mean_or_zero(kern_ms["bwd_main"])
    dsum_ms, dqconv_ms = mean_or_zero(kern_ms["bwd_dsum"]), mean_or_zero(kern_ms["bwd_dq_convert"])
    dominant = "bwd_main" if bwd_main_ms >= fwd_ms else "fwd"
    dom_ms = bwd_main_ms if dominant == "bwd_main" else fwd_ms
    dom_flops = fl["bwd"] if dominant == "bwd_main" else fl["fwd"]
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    rows = w.B * w.Hq * w.Sq
    es = prep.es
    dsum_bytes = rows * w.D * es * 2 + rows * 4 + rows * w.D * 4
    dqconv_bytes = rows * w.D * 4 + rows * w.D * es
    csrc = os.path.join(ROOT, "backward_adapter_gb300", "csrc")
    dom_src = os.path.join(csrc, "fa_tc_bwd.cu" if dominant == "bwd_main" else "fa_tc_fwd.cu")
    traffic = measured_traffic(dominant, dom_src) if os.path.exists(dom_src) else None

    # End to end through the public API from pinned host buffers: every step copies its inputs
    # host -> device and its results (O, LSE, dQ, dK, dV) device -> host. Copies run on their
    # own streams into double-buffered device buffers, so step i+1's inputs arrive while step i
    # computes.
    d, host = prep.d, prep.host
    o, lse, dq, dk, dv = prep.o, prep.lse, prep.dq, prep.dk, prep.dv
    out_host = [{n: torch.empty_like(t, device="cpu").pin_memory() for n, t in
                 (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host[0].values())
    bufs = [d, {n: torch.empty_like(t) for n, t in d.items()}]
    outs = [(o, lse, dq, dk, dv),
            (torch.empty_like(o), torch.empty_like(lse), torch.empty_like(dq), torch.empty_like(dk),
             torch.empty_like(dv))]
    if w.accum:
        outs[1][3].copy_(dk)
        outs[1][4].copy_(dv)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
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
        o_, lse_, dq_, dk_, dv_ = outs[sl]
        prep.fwd_call(src, o_, lse_)
        prep.bwd_call(src, o_, lse_, dq_, dk_, dv_)
        done[sl].record(comp)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(done[sl])
            for n, t in zip(("o", "lse", "dq", "dk", "dv"), outs[sl]):
                out_host[sl][n].copy_(t, non_blocking=True)
            read_back[sl].record(copy_out)
    last = ev()
    last.record(copy_out)
    comp.wait_event(last)
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms, e2e_value = job_tflops(world, fl["total"], e0.elapsed_time(e1) / E)

    # The other workloads of the op, each timed the same way (not part of the headline's timed
    # region): rank 0 at N = 1 only, so the multi-GPU launch stays short.
    by_workload = None
    if rank == 0 and world == 1 and not args.no_by_workload:
        by_workload = {}
        for ow in wl.WORKLOADS:
            if ow.name == w.name:
                continue
            op = Prepared(ft, torch, ow, dev)
            s_ms, k_ms, _ = timed_steps(torch, ft, op, args.workload_steps, max(3, args.warmup), flush)
            by_workload[ow.name] = workload_summary(ow, wl.flops(ow), s_ms, k_ms, peaks["bf16_tflops"])
            del op
        torch.cuda.synchronize()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # grow the sample one GQA group at a time until ~10 s of oracle work (or every head)
        G = w.Hq // w.Hkv
        heads = G
        dt_cpu, fl_cpu, desc = oracle_sample(w, prep.inputs, heads)
        while dt_cpu < 10.0 and heads < w.Hq:
            heads = min(w.Hq, max(heads + G, int(heads * 10.0 / max(dt_cpu, 1e-3)) // G * G))
            dt_cpu, fl_cpu, desc = oracle_sample(w, prep.inputs, heads)
        cpu = {"value": fl_cpu / dt_cpu / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": desc, "seconds": dt_cpu}

    if rank != 0:
        return 0
    st = stats(step_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": mean_ms, "ms_per_step_median": st["median"], "ms_per_step_min": st["min"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
                   "causal": w.causal, "q_offset": w.q_offset, "window": w.window, "mask": w.mask, "accum": w.accum,
                   "rows_read_back": [w.q_offset, w.Sq] if w.accum and not prep.q8 else None,
                   "kv_format": w.kv_format,
                   "deterministic": bool(args.deterministic),
                   "visible_pairs": fl["pairs"], "gflop_per_step": fl["total"] / 1e9,
                   "l2": "flushed (256 MiB write) between timed steps, outside the step events",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": value / world / peaks["bf16_tflops"],
        "fwd_tflops": fl["fwd"] / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": fl["bwd"] / ((bwd_main_ms + dsum_ms + dqconv_ms) * 1e-3) / 1e12,
        "kernel_ms": {"fwd": fwd_ms, "bwd_main": bwd_main_ms, "bwd_dsum": dsum_ms, "bwd_dq_convert": dqconv_ms},
        "kernel_ms_median_min": {n: {"median": v["median"], "min": v["min"]}
                                 for n, v in ((n, stats(x)) for n, x in kern_ms.items()) if v},
        "hbm_passes_gbs": {"bwd_dsum": gbs(dsum_bytes, dsum_ms),
                           "bwd_dq_convert": gbs(dqconv_bytes, dqconv_ms),
                           "peak": peaks["hbm_gbs"]},
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 dense burst",
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "copies": "pinned host buffers; inputs and results (O, LSE, dQ, dK, dV) on their own streams, "
                          "double-buffered"},
        "gpu_launches": launches,
        "wall_s_timed_region": t_wall,
        "clocks": clock_info,
        "by_workload": by_workload,
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
