"""The op over a q8_0-style K/V cache read in place (fa_train_*_q8).

Each case is compared with the oracle on the cache's dequantized values. A cache whose values
are exact in bf16 (power-of-two scales) must give bitwise the same results as the bf16 entry
points run on those values: that pins the on-chip dequantization and its swizzled layout to the
bf16 path, which the parity tests pin to the oracle.
"""
import ctypes

import numpy as np
import pytest

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl


def test_q8_requires_bf16_queries_and_a_descriptor():
    fbuild.build()
    lib = ft.load_library()
    p = ft.FaParams(1, 2, 1, 64, 64, 64, ft.FA_F32, 0.125, 0, ft.FA_MASK_NONE, 1, 0, 0, 0, ft.FA_KV_Q8_0)
    fake = 1 << 30
    kv = ft.FaKvQ8(2 * fake, 3 * fake, 4 * fake, 5 * fake)
    st = lib.fa_train_fwd_q8(ctypes.byref(p), fake, ctypes.byref(kv), None, 6 * fake, 7 * fake, None, 0, None)
    assert st == ft.FA_ERR_UNSUPPORTED and b"bf16" in lib.fa_last_error()
    p.dtype = ft.FA_BF16
    assert lib.fa_train_fwd_q8(ctypes.byref(p), fake, None, None, 6 * fake, 7 * fake, None, 0, None) == \
        ft.FA_ERR_INVALID_ARG
    kv.k_d = 0
    st = lib.fa_train_fwd_q8(ctypes.byref(p), fake, ctypes.byref(kv), None, 6 * fake, 7 * fake, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"k_d is NULL" in lib.fa_last_error()


W = wl.Workload
CASES = [
    W("q8_causal_gqa_d128", B=1, Hq=4, Hkv=2, Sq=300, Sk=300, D=128, causal=True, kv_format="q8_0", seed=81),
    W("q8_window_bool_d64", B=2, Hq=2, Hkv=1, Sq=260, Sk=333, D=64, window=70, q_offset=40, mask="random_bool",
      kv_format="q8_0", seed=82),
    W("q8_chunk_long_keys_accum", B=1, Hq=4, Hkv=1, Sq=64, Sk=2000, D=128, causal=True, q_offset=1936, accum=True,
      kv_format="q8_0", seed=83),
    W("q8_ragged_keys_d128", B=1, Hq=2, Hkv=2, Sq=130, Sk=333, D=128, kv_format="q8_0", seed=84),
]


def score_shift_from_bf16_keys(w, inputs) -> float:
    """The kernels round each dequantized key to bf16 before the QK^T product; the oracle uses
    the cache's exact values (the page's cast to F32). LSE is 1-Lipschitz in the scores, so it
    moves by at most max_ij |scale * <q_i, bf16(k_j) - k_j>|, computed here from the data."""
    from oracle import attention as ref
    from oracle import set_rows as rows_ref
    k = ref.dequantize_q8_0(*inputs["k_q8"])
    dk = rows_ref.to_bf16_bits(k.astype(np.float32)).astype(np.float64) - k
    G = w.Hq // w.Hkv
    q = inputs["q"].astype(np.float64)
    shift = 0.0
    for h in range(w.Hq):
        s = np.einsum("bid,bjd->bij", q[:, h], dk[:, h // G]) * w.scale
        shift = max(shift, float(np.abs(s).max()))
    return shift


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_q8_cache_matches_oracle(w):
    from tests import parity_util as pu
    inputs = wl.make_inputs(w)
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    exp = pu.run_oracle(w, inputs)
    pu.assert_parity(w, got, exp, lse_extra=score_shift_from_bf16_keys(w, inputs))
    pu.assert_exact_zeros(w, inputs, got)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_q8_with_bf16_exact_values_is_bitwise_the_bf16_path(D):
    import torch
    rng = np.random.default_rng(85 + D)
    B, Hq, Hkv, Sq, Sk = 1, 4, 2, 200, 270
    q = torch.from_numpy(rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    do = torch.from_numpy(rng.standard_normal((B, Hq, Sq, D)).astype(np.float32)).cuda().to(torch.bfloat16)
    planes, vals = [], []
    for _ in range(2):
        qv = rng.integers(-127, 128, (B, Hkv, Sk, D)).astype(np.int8)
        dv = (2.0 ** rng.integers(-8, -3, (B, Hkv, Sk, D // 32))).astype(np.float16)   # exact: q * d fits bf16
        planes += [torch.from_numpy(qv).cuda(), torch.from_numpy(dv).cuda()]
        vals.append(torch.from_numpy((qv.astype(np.float32) * np.repeat(dv.astype(np.float32), 32, -1))).cuda()
                    .to(torch.bfloat16))
    kw = dict(causal=True, q_offset=Sk - Sq)
    o8, lse8 = ft.fwd_q8(q, *planes, **kw)
    dq8, dk8, dv8 = ft.bwd_q8(q, *planes, o8, lse8, do, deterministic=True, **kw)
    o, lse = ft.fwd(q, vals[0], vals[1], **kw)
    dq, dk, dv = ft.bwd(q, vals[0], vals[1], o, lse, do, deterministic=True, **kw)
    torch.cuda.synchronize()
    assert ft.device_status() == 0
    for a, b in ((o8, o), (lse8, lse), (dq8, dq), (dk8, dk), (dv8, dv)):   # dQ in a fixed order on both
        assert torch.equal(a, b)
