"""The op over an fp16 K/V cache read in place (kv_format FA_KV_F16, through the plain entry points).

Each case is compared with the oracle on the cache's fp16 values. The library rounds K and V to
bf16 for the tensor cores; the LSE tolerance adds the largest score change that rounding can cause,
computed from the data. A cache whose fp16 values are exact in bf16 must give bitwise the results
of the bf16 path run on those values, and an fp16 cache in [B, S, H, D] bitwise those of the same
cache in [B, H, S, D]: those pin the cast pass to the bf16 path, which the parity tests pin to the
oracle.
"""
import numpy as np
import pytest

from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl

W = wl.Workload
CASES = [
    W("f16_causal_gqa_d128", B=1, Hq=4, Hkv=2, Sq=300, Sk=300, D=128, causal=True, kv_format="f16", seed=91),
    W("f16_window_bool_d64", B=2, Hq=2, Hkv=1, Sq=260, Sk=333, D=64, window=70, q_offset=40, mask="random_bool",
      kv_format="f16", seed=92),
    W("f16_chunk_long_keys_accum", B=1, Hq=4, Hkv=1, Sq=64, Sk=2000, D=128, causal=True, q_offset=1936, accum=True,
      kv_format="f16", seed=93),
    W("f16_ragged_keys_additive_d128", B=1, Hq=2, Hkv=2, Sq=130, Sk=333, D=128, mask="random_add", kv_format="f16",
      seed=94),
]


def score_shift_from_bf16_keys(w, inputs) -> float:
    """max over (i, j) of |scale * <q_i, bf16(k_j) - k_j>| for the cache's fp16 keys: LSE is
    1-Lipschitz in the scores, so the bf16 rounding of K moves it by at most this much."""
    from oracle import set_rows as rows_ref
    k = inputs["k"].astype(np.float64)
    dk = rows_ref.to_bf16_bits(inputs["k"].astype(np.float32)).astype(np.float64) - k
    G = w.Hq // w.Hkv
    q = inputs["q"].astype(np.float64)
    shift = 0.0
    for h in range(w.Hq):
        s = np.einsum("bid,bjd->bij", q[:, h], dk[:, h // G]) * w.scale
        shift = max(shift, float(np.abs(s).max()))
    return shift


def test_f16_inputs_are_fp16_values_finer_than_bf16():
    w = CASES[0]
    x = wl.make_inputs(w)
    k = x["k"]
    assert np.array_equal(k.astype(np.float16).astype(np.float32), k)      # exact in fp16
    assert not np.array_equal(wl.round_to_bf16(k), k)                      # not all exact in bf16
    # Q and dO stay bf16
    assert np.array_equal(wl.round_to_bf16(x["q"]), x["q"])


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_f16_cache_matches_oracle(w):
    from tests import parity_util as pu
    inputs = wl.make_inputs(w)
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    exp = pu.run_oracle(w, inputs)
    pu.assert_parity(w, got, exp, lse_extra=score_shift_from_bf16_keys(w, inputs))
    pu.assert_exact_zeros(w, inputs, got)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_f16_with_bf16_exact_values_is_bitwise_the_bf16_path(D):
    import torch
    rng = np.random.default_rng(95 + D)
    B, Hq, Hkv, Sq, Sk = 1, 4, 2, 200, 270
    q = torch.from_numpy(rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    do = torch.from_numpy(rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    # integers / 64: exact in fp16 and in bf16
    kv = [torch.from_numpy((rng.integers(-128, 128, (B, Hkv, Sk, D)) / 64.0).astype(np.float32)).cuda()
          for _ in range(2)]
    k16, v16 = (t.to(torch.float16) for t in kv)
    kbf, vbf = (t.to(torch.bfloat16) for t in kv)
    kw = dict(causal=True, q_offset=Sk - Sq)
    o16, lse16 = ft.fwd(q, k16, v16, **kw)
    dq16, dk16, dv16 = ft.bwd(q, k16, v16, o16, lse16, do, deterministic=True, **kw)
    o, lse = ft.fwd(q, kbf, vbf, **kw)
    dq, dk, dv = ft.bwd(q, kbf, vbf, o, lse, do, deterministic=True, **kw)
    acc16 = [torch.zeros(B, Hkv, Sk, D, device="cuda") for _ in range(2)]
    acc = [torch.zeros(B, Hkv, Sk, D, device="cuda") for _ in range(2)]
    ft.bwd_accum(q, k16, v16, o16, lse16, do, *acc16, deterministic=True, **kw)
    ft.bwd_accum(q, kbf, vbf, o, lse, do, *acc, deterministic=True, **kw)
    torch.cuda.synchronize()
    assert ft.device_status() == 0
    assert dk16.dtype == torch.bfloat16 and dv16.dtype == torch.bfloat16
    for a, b in ((o16, o), (lse16, lse), (dq16, dq), (dk16, dk), (dv16, dv), (acc16[0], acc[0]), (acc16[1], acc[1])):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_f16_cache_bshd_is_bitwise_the_bhsd_result():
    import torch
    rng = np.random.default_rng(97)
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 150, 290, 128
    q = torch.from_numpy(rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    do = torch.from_numpy(rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    k, v = (torch.from_numpy(rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)).cuda().to(torch.float16)
            for _ in range(2))
    kw = dict(causal=True, q_offset=Sk - Sq)
    o, lse = ft.fwd(q, k, v, **kw)
    dq, dk, dv = ft.bwd(q, k, v, o, lse, do, deterministic=True, **kw)
    t = lambda x: x.transpose(1, 2).contiguous()   # noqa: E731
    ob, lseb = ft.fwd(t(q), t(k), t(v), layout="bshd", **kw)
    dqb, dkb, dvb = ft.bwd(t(q), t(k), t(v), ob, lseb, t(do), layout="bshd", deterministic=True, **kw)
    torch.cuda.synchronize()
    assert ft.device_status() == 0
    assert torch.equal(lseb, lse)
    for a, b in ((ob, o), (dqb, dq), (dkb, dk), (dvb, dv)):   # dQ added in a fixed order on both
        assert torch.equal(a, t(b))
