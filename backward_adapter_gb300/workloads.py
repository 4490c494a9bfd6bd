"""Seeded synthetic inputs for the fused flash-attention training op.

This module is shared by the oracle-side tests, the GPU parity tests and the
benchmark. It holds shapes, seeds and random draws only: none of the
attention arithmetic lives here. Every tensor is drawn in float32 from a
seeded numpy PCG64 generator; where the workload is bf16 the draw is rounded
to bf16 (round-to-nearest-even) here, so the oracle and the GPU see the same
values (the oracle widens the rounded values to float64).

Workload shapes follow the pages' use of the op:
  * DiT self-attention with padded key columns and GQA (HOT-Step TRAINING.md,
    "DiT micro-batching": padded KV columns are masked for valid query rows,
    padded query rows keep the pad columns open), with or without the sliding
    window of the other self-attention layer type;
  * DiT cross-attention with a per-batch encoder length (flash-attn-training
    skill, trap list item 8: the cross mask is the one that masks whole key
    columns; item 9: fully-masked query rows);
  * causal LM attention;
  * a 512-token query chunk attending causally to a cached K/V window of
    67,584 tokens, accumulating dK/dV into caller-owned fp32 buffers
    (llama.cpp PR #57, "Why" and commit 86c140d).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

NEG_INF = np.float32(-np.inf)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    dtype: str = "bf16"          # "f32" or "bf16": input/output element type
    causal: bool = False
    q_offset: int = 0            # query row i sits at key position q_offset + i
    window: int = 0              # sliding window half-width (0 = none)
    kv_format: str = "bf16"      # "bf16" (K/V in dtype), "q8_0" (8-bit values + fp16 scale per 32 features)
    #                              or "f16" (an fp16 K/V cache under bf16 Q / dO)
    mask: str = "none"           # none | extra_row | pad_self | cross | random_bool | random_add
    accum: bool = False          # dK/dV accumulate into prefilled fp32 buffers
    do_std: float = 1.0          # standard deviation of dO
    acc_std: float = 0.01        # standard deviation of the accumulator prefill
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the op is specified on, smallest first.
TINY_F32 = Workload("tiny_f32_gqa_extra_masked_row", B=1, Hq=2, Hkv=1, Sq=65, Sk=64, D=64,
                    dtype="f32", mask="extra_row", seed=1001)
DIT_SELF = Workload("dit_self_gqa_pad_s1024_d64", B=1, Hq=16, Hkv=8, Sq=1024, Sk=1024, D=64,
                    mask="pad_self", seed=1002)
DIT_CROSS = Workload("dit_cross_b2_sq2048_sk256_d128", B=2, Hq=16, Hkv=16, Sq=2048, Sk=256, D=128,
                     mask="cross", seed=1003)
CAUSAL_LM = Workload("causal_lm_h32_kv8_s4096_d128", B=1, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128,
                     causal=True, do_std=0.1, seed=1004)
LONG_WINDOW = Workload("chunk512_window67584_h16_kv4_d128_accum", B=1, Hq=16, Hkv=4, Sq=512,
                       Sk=67584, D=128, causal=True, q_offset=67072, accum=True, seed=1005)

WORKLOADS = [TINY_F32, DIT_SELF, DIT_CROSS, CAUSAL_LM, LONG_WINDOW]

# The other DiT self-attention mask: a sliding window plus the padded key columns (the pages give
# no width; 128 keys on either side is the reading used here).
DIT_SELF_WINDOW = Workload("dit_self_window128_gqa_pad_s1024_d64", B=1, Hq=16, Hkv=8, Sq=1024, Sk=1024, D=64,
                           window=128, mask="pad_self", seed=1006)

# The long-window chunk over a q8_0 K/V cache read in place (the cache format the walk trains in).
LONG_WINDOW_Q8 = LONG_WINDOW.with_(name="chunk512_window67584_h16_kv4_d128_accum_q8cache", kv_format="q8_0")
# The same chunk over an fp16 cache (the other cache type the walk reads in place).
LONG_WINDOW_F16 = LONG_WINDOW.with_(name="chunk512_window67584_h16_kv4_d128_accum_f16cache", kv_format="f16")

BY_NAME = {w.name: w for w in WORKLOADS + [DIT_SELF_WINDOW, LONG_WINDOW_Q8, LONG_WINDOW_F16]}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).reshape(x.shape)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def cross_lengths(w: Workload) -> np.ndarray:
    """Per-batch encoder length L_b ~ U{64..min(256, Sk)} drawn from the workload seed."""
    rng = np.random.default_rng(w.seed + 7919)
    lo = min(64, w.Sk)
    return rng.integers(lo, w.Sk + 1, size=w.B)


def cross_masked_rows(w: Workload, per_batch: int = 2) -> np.ndarray:
    """Two distinct fully-masked query rows per batch, drawn from the workload seed."""
    rng = np.random.default_rng(w.seed + 104729)
    return np.stack([rng.choice(w.Sq, size=per_batch, replace=False) for _ in range(w.B)])


def pad_length(w: Workload) -> int:
    """Valid length L of the padded self-attention workload: the last 20% of keys are pad."""
    return w.Sk - int(round(0.2 * w.Sk))


def make_mask(w: Workload) -> tuple[Optional[np.ndarray], str]:
    """Return (mask, kind) with kind in {"none", "add", "bool"}.

    An additive mask is float32 [Bm, Sq, Sk] with -inf where masked; a
    boolean mask is uint8 [Bm, Sq, Sk] with 1 = attend, 0 = masked.
    """
    if w.mask == "none":
        return None, "none"
    if w.mask == "extra_row":
        m = np.zeros((1, w.Sq, w.Sk), np.float32)
        m[0, w.Sq - 1, :] = NEG_INF
        return m, "add"
    if w.mask == "pad_self":
        L = pad_length(w)
        m = np.zeros((1, w.Sq, w.Sk), np.float32)
        m[0, :L, L:] = NEG_INF          # valid query rows never see pad keys
        return m, "add"                  # pad query rows stay fully open
    if w.mask == "cross":
        lens = cross_lengths(w)
        rows = cross_masked_rows(w)
        m = np.zeros((w.B, w.Sq, w.Sk), np.float32)
        for b in range(w.B):
            m[b, :, lens[b]:] = NEG_INF
            m[b, rows[b], :] = NEG_INF
        return m, "add"
    if w.mask in ("random_bool", "random_add"):
        rng = np.random.default_rng(w.seed + 31337)
        keep = rng.random((w.B, w.Sq, w.Sk)) < 0.7
        if w.Sq > 2:
            keep[:, 1, :] = False        # one fully-masked query row
        if w.Sk > 3:
            keep[:, :, 2] = False        # one fully-masked key column
        if w.mask == "random_bool":
            return keep.astype(np.uint8), "bool"
        bias = _normal(rng, (w.B, w.Sq, w.Sk), 0.5)
        bias[~keep] = NEG_INF
        return bias, "add"
    raise ValueError(f"unknown mask recipe {w.mask!r}")


def make_inputs(w: Workload) -> dict:
    """Draw Q, K, V, dO (and the fp32 accumulator prefill) for a workload.

    Returns float32 arrays holding exactly the values the op computes on
    (already rounded to bf16 when the workload is bf16), plus the mask.
    """
    rng = np.random.default_rng(w.seed)
    q = _normal(rng, (w.B, w.Hq, w.Sq, w.D), 1.0)
    k = _normal(rng, (w.B, w.Hkv, w.Sk, w.D), 1.0)
    v = _normal(rng, (w.B, w.Hkv, w.Sk, w.D), 1.0)
    do = _normal(rng, (w.B, w.Hq, w.Sq, w.D), w.do_std)
    if w.kv_format == "f16":   # the cache holds fp16 values (finer than bf16: the cast is exercised)
        k, v = (t.astype(np.float16).astype(np.float32) for t in (k, v))
    if w.dtype == "bf16":
        q, do = round_to_bf16(q), round_to_bf16(do)
        if w.kv_format != "f16":
            k, v = round_to_bf16(k), round_to_bf16(v)
    out = {"q": q, "k": k, "v": v, "do": do}
    if w.kv_format == "q8_0":
        out["k_q8"] = quantize_q8_0(k)
        out["v_q8"] = quantize_q8_0(v)
    out["mask"], out["mask_kind"] = make_mask(w)
    if w.accum:
        out["dk_acc"] = _normal(rng, (w.B, w.Hkv, w.Sk, w.D), w.acc_std)
        out["dv_acc"] = _normal(rng, (w.B, w.Hkv, w.Sk, w.D), w.acc_std)
    return out


def quantize_q8_0(x: np.ndarray):
    """Encode float32 [..., D] as a q8_0-style cache: per block of 32 features a float16 scale
    d = max|x| / 127 and int8 values q = round(x / d) (computed with the stored float16 d,
    clipped to [-127, 127]). Returns (q int8 [..., D], d float16 [..., D / 32])."""
    x = np.asarray(x, dtype=np.float32)
    blocks = x.reshape(*x.shape[:-1], x.shape[-1] // 32, 32)
    d = (np.abs(blocks).max(axis=-1) / np.float32(127.0)).astype(np.float16)
    dd = d.astype(np.float32)[..., None]
    safe = np.where(dd > 0, dd, np.float32(1.0))
    q = np.where(dd > 0, np.rint(blocks / safe), 0.0)
    q = np.clip(q, -127, 127).astype(np.int8)
    return q.reshape(x.shape), d


def visible_pairs(w: Workload) -> int:
    """Number of (query head, query row, key) triples whose score is not masked.

    This is the unit of the mask- and causal-aware FLOP count: the forward
    does 4*D flops per visible pair (QK^T and PV), the backward 10*D
    (QK^T recompute, dO V^T, P^T dO, dS K and dS^T Q).
    """
    mask, kind = make_mask(w)
    i = np.arange(w.Sq)[:, None]
    j = np.arange(w.Sk)[None, :]
    total = 0
    for b in range(w.B):
        vis = np.ones((w.Sq, w.Sk), bool)
        if mask is not None:
            mb = mask[b if mask.shape[0] > 1 else 0]
            vis &= (mb != 0) if kind == "bool" else (mb > -1e9)
        if w.causal:
            vis &= j <= w.q_offset + i
        if w.window > 0:
            vis &= np.abs(w.q_offset + i - j) <= w.window
        total += int(vis.sum())
    return total * w.Hq


def flops(w: Workload) -> dict:
    p = visible_pairs(w)
    return {"fwd": 4.0 * w.D * p, "bwd": 10.0 * w.D * p, "total": 14.0 * w.D * p, "pairs": p}
