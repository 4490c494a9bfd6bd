"""Helpers for the GPU parity tests: run the CUDA path (through the C-ABI
binding) and the fp64 oracle on the same seeded inputs and compare them."""
from __future__ import annotations

import numpy as np
import torch

from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl
from oracle import attention as ref

# Tolerances: bf16 inputs with fp32 accumulation vs fp32 inputs.
TOL = {"bf16": (1e-2, 1e-3), "f32": (1e-4, 0.0)}
LSE_ABS = 1e-3


def torch_dtype(w: wl.Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def to_device(inputs: dict, w: wl.Workload, device="cuda"):
    dt = torch_dtype(w)
    t = {n: torch.from_numpy(inputs[n]).to(device).to(dt).contiguous() for n in ("q", "k", "v", "do")}
    if w.kv_format == "f16":   # the fp16 cache as it is (its values are exact in fp16)
        for n in ("k", "v"):
            t[n] = torch.from_numpy(inputs[n]).to(device).to(torch.float16).contiguous()
    m = inputs["mask"]
    t["mask"] = None if m is None else torch.from_numpy(m).to(device).contiguous()
    if w.accum:
        t["dk_acc"] = torch.from_numpy(inputs["dk_acc"]).to(device).contiguous()
        t["dv_acc"] = torch.from_numpy(inputs["dv_acc"]).to(device).contiguous()
    if w.kv_format == "q8_0":
        for n in ("k", "v"):
            qv, dv = inputs[n + "_q8"]
            t[n + "_q"] = torch.from_numpy(qv).to(device).contiguous()
            t[n + "_d"] = torch.from_numpy(dv).to(device).contiguous()
    return t


def run_gpu(w: wl.Workload, t: dict, deterministic: bool = False) -> dict:
    """Forward + backward on the GPU; returns float64 numpy copies of every output."""
    kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset, window=w.window, deterministic=deterministic)
    if w.kv_format == "q8_0":
        kv = (t["k_q"], t["k_d"], t["v_q"], t["v_d"])
        fkw = {k_: v_ for k_, v_ in kw.items() if k_ != "deterministic"}
        o, lse = ft.fwd_q8(t["q"], *kv, t["mask"], **fkw)
        if w.accum:
            dk, dv = t["dk_acc"].clone(), t["dv_acc"].clone()
            dq = ft.bwd_q8(t["q"], *kv, o, lse, t["do"], t["mask"], dk_acc=dk, dv_acc=dv, **kw)
        else:
            dq, dk, dv = ft.bwd_q8(t["q"], *kv, o, lse, t["do"], t["mask"], **kw)
    elif w.accum:
        o, lse = ft.fwd(t["q"], t["k"], t["v"], t["mask"], **kw)
        dk, dv = t["dk_acc"].clone(), t["dv_acc"].clone()
        dq = ft.bwd_accum(t["q"], t["k"], t["v"], o, lse, t["do"], dk, dv, t["mask"], **kw)
    else:
        o, lse = ft.fwd(t["q"], t["k"], t["v"], t["mask"], **kw)
        dq, dk, dv = ft.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], t["mask"], **kw)
    torch.cuda.synchronize()
    status = ft.device_status()
    assert status == 0, f"a bounded wait inside a kernel ran out of time (site {status & 0xffff})"
    return {n: x.double().cpu().numpy() for n, x in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


def run_oracle(w: wl.Workload, inputs: dict, q_heads=None, kv_heads=None) -> dict:
    """Oracle on all heads, or on the given query heads and the key/value heads they read."""
    q, k, v, do = inputs["q"], inputs["k"], inputs["v"], inputs["do"]
    if w.kv_format == "q8_0":
        k = ref.dequantize_q8_0(*inputs["k_q8"])
        v = ref.dequantize_q8_0(*inputs["v_q8"])
    if q_heads is not None:
        q, do = q[:, q_heads], do[:, q_heads]
        k, v = k[:, kv_heads], v[:, kv_heads]
    args = (q, k, v, do)
    kw = dict(mask=inputs["mask"], mask_kind=inputs["mask_kind"], causal=w.causal, q_offset=w.q_offset,
              window=w.window)
    if w.accum:
        dka, dva = inputs["dk_acc"], inputs["dv_acc"]
        if kv_heads is not None:
            dka, dva = dka[:, kv_heads], dva[:, kv_heads]
        return ref.backward_accumulate(*args, dka, dva, w.scale, **kw)
    return ref.backward(*args, w.scale, **kw)


def max_err(got, exp):
    return float(np.abs(got - exp).max()) if got.size else 0.0


def assert_parity(w: wl.Workload, got: dict, exp: dict, where: str = "", lse_extra: float = 0.0):
    """Max-abs error of O, dQ, dK, dV within rel * max|ref| + abs; LSE within LSE_ABS absolute.

    With one key per head, softmax is constant (P = 1), so dQ and dK are exactly
    zero and only dV carries a gradient; otherwise every gradient reference must
    be non-zero so that no comparison passes 0 vs 0.
    """
    rel, abs_ = TOL[w.dtype]
    for n in ("o", "dq", "dk", "dv"):
        e = max_err(got[n], exp[n])
        bound = rel * float(np.abs(exp[n]).max()) + abs_
        assert e <= bound, f"{w.name}{where}: {n} max-abs err {e:.3e} > {bound:.3e}"
    for n in (("dv",) if w.Sk == 1 else ("dq", "dk", "dv")):
        assert float(np.abs(exp[n]).max()) > 0, f"{n} reference is vacuously zero"
    e = max_err(got["lse"], exp["lse"])
    assert e <= LSE_ABS + lse_extra, f"{w.name}{where}: lse max-abs err {e:.3e} (allowed {LSE_ABS + lse_extra:.3e})"


def assert_exact_zeros(w: wl.Workload, inputs: dict, got: dict, q_heads=None):
    """Query rows that see no key: O = 0, LSE = 0, dQ = 0 exactly. Keys no query sees (mask,
    causal rule or window): dK = dV = 0 exactly (the accumulator unchanged under accumulation)."""
    mask, kind = inputs["mask"], inputs["mask_kind"]
    for b in range(w.B):
        mb = None if mask is None else mask[b if mask.shape[0] > 1 else 0]
        vis = ref.visibility(w.Sq, w.Sk, mb, kind, w.causal, w.q_offset, w.window)
        rows = np.nonzero(~vis.any(axis=1))[0]
        if rows.size:
            assert np.all(got["o"][b][:, rows] == 0) and np.all(got["lse"][b][:, rows] == 0)
            assert np.all(got["dq"][b][:, rows] == 0)
        cols = np.nonzero(~vis.any(axis=0))[0]
        if cols.size and not w.accum:
            assert np.all(got["dk"][b][:, cols] == 0) and np.all(got["dv"][b][:, cols] == 0)
        if cols.size and w.accum:
            np.testing.assert_array_equal(got["dk"][b][:, cols], inputs["dk_acc"][b][:, cols])


def cache_lse_allowance(w: wl.Workload, inputs: dict, q_heads=None, kv_heads=None) -> float:
    """Extra LSE tolerance for a q8_0 or fp16 K/V cache: the kernels round each key to bf16, the
    oracle uses the cache's exact values. LSE is 1-Lipschitz in the scores, so it moves by at most
    max |scale * <q_i, bf16(k_j) - k_j>| over the compared heads (0 for a bf16 K/V)."""
    from oracle import set_rows as rows_ref
    if w.kv_format == "q8_0":
        k = ref.dequantize_q8_0(*inputs["k_q8"])
    elif w.kv_format == "f16":
        k = inputs["k"].astype(np.float64)
    else:
        return 0.0
    dk = rows_ref.to_bf16_bits(k.astype(np.float32)).astype(np.float64) - k
    G = w.Hq // w.Hkv
    q = inputs["q"].astype(np.float64)
    shift = 0.0
    for h in (range(w.Hq) if q_heads is None else q_heads):
        kv = h // G
        if kv_heads is not None and kv not in kv_heads:
            continue
        sc = np.einsum("bid,bjd->bij", q[:, h], dk[:, kv]) * w.scale
        shift = max(shift, float(np.abs(sc).max()))
    return shift

