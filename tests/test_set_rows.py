"""SET_ROWS backward: the chunk's K/V gradient read back out of the window accumulator.

The standalone gather (fa_set_rows_backward) is compared bit for bit with the oracle
(a copy, or a copy rounded to bf16); the fused form (fa_train_bwd_accum_rows) must
return exactly the bf16 rounding of its own finished accumulator rows, and those
rows must match the oracle within the backward's tolerance.
"""
import ctypes

import numpy as np
import pytest

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl
from oracle import set_rows as rows_ref


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return ft.load_library()


BAD_GATHER = [
    ("D_not_multiple_of_4", dict(D=6), ft.FA_ERR_INVALID_ARG),
    ("D_too_big", dict(D=2048), ft.FA_ERR_INVALID_ARG),
    ("S_zero", dict(S=0), ft.FA_ERR_INVALID_ARG),
    ("n_rows_negative", dict(n=-1), ft.FA_ERR_INVALID_ARG),
    ("out_dtype", dict(dt=7), ft.FA_ERR_INVALID_ARG),
    ("null_out", dict(out=0), ft.FA_ERR_INVALID_ARG),
    ("misaligned_acc", dict(acc=(1 << 30) + 4), ft.FA_ERR_INVALID_ARG),
    ("out_overlaps_acc", dict(out=(1 << 30) + 64), ft.FA_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,kw,code", BAD_GATHER, ids=[b[0] for b in BAD_GATHER])
def test_gather_arguments_are_checked_before_launch(lib, name, kw, code):
    a = dict(acc=1 << 30, B=1, H=2, S=16, D=64, idx=2 << 30, n=4, out=3 << 30, dt=ft.FA_BF16)
    a.update(kw)
    st = lib.fa_set_rows_backward(a["acc"], a["B"], a["H"], a["S"], a["D"], a["idx"], a["n"], a["out"] or None,
                                  a["dt"], None)
    assert st == code, lib.fa_last_error()


def test_fused_rows_outside_the_keys_are_rejected(lib):
    p = ft.FaParams(1, 4, 2, 100, 130, 64, ft.FA_BF16, 0.125, 1, ft.FA_MASK_NONE, 1, 0, 30)
    fake = 1 << 34
    for begin, n in ((-1, 4), (120, 11), (0, -2)):
        st = lib.fa_train_bwd_accum_rows(ctypes.byref(p), fake, 2 * fake, 3 * fake, None, 4 * fake, 5 * fake,
                                         6 * fake, 7 * fake, 8 * fake, 9 * fake, begin, n, 10 * fake, 11 * fake,
                                         None, 0, None)
        assert st == ft.FA_ERR_INVALID_ARG and b"rows" in lib.fa_last_error()


# ---- GPU ------------------------------------------------------------------------------------------

GATHER_CASES = [(2, 3, 37, 128, [0, 36, 5, 5, 17, 2, 36]), (1, 2, 70, 64, list(range(69, -1, -3))),
                (1, 1, 5, 4, [4, 0])]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,S,D,idx", GATHER_CASES, ids=["d128_repeats", "d64_reversed", "d4"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gather_is_bit_exact(B, H, S, D, idx, out):
    import torch
    rng = np.random.default_rng(B * 1000 + S)
    acc = rng.standard_normal((B, H, S, D)).astype(np.float32) * np.float32(3.0)
    got = ft.set_rows_backward(torch.from_numpy(acc).cuda(), torch.tensor(idx, dtype=torch.int64).cuda(),
                               out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
    torch.cuda.synchronize()
    assert ft.device_status() == 0
    want = rows_ref.set_rows_backward(acc, idx, out)
    np.testing.assert_array_equal(got.float().cpu().numpy(), want)


@pytest.mark.gpu
def test_gather_index_outside_the_rows_gives_zeros_and_a_status():
    import torch
    rng = np.random.default_rng(7)
    acc = rng.standard_normal((1, 2, 20, 64)).astype(np.float32)
    idx = [3, 20, 7, -1, 19]
    ft.device_status()
    got = ft.set_rows_backward(torch.from_numpy(acc).cuda(), torch.tensor(idx, dtype=torch.int64).cuda(),
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ft.device_status() == (0x40000000 | 950)
    got = got.cpu().numpy()
    for r, j in enumerate(idx):
        if 0 <= j < 20:
            np.testing.assert_array_equal(got[:, :, r], acc[:, :, j])
        else:
            assert np.all(got[:, :, r] == 0)


FUSED = [
    wl.Workload("rows_chunk_at_window_end", B=1, Hq=4, Hkv=2, Sq=130, Sk=517, D=128, causal=True, q_offset=387,
                accum=True, seed=61),
    wl.Workload("rows_window_d64_bool", B=2, Hq=2, Hkv=1, Sq=96, Sk=300, D=64, q_offset=150, window=40,
                mask="random_bool", accum=True, seed=62),
    wl.Workload("rows_f32_simt", B=1, Hq=2, Hkv=1, Sq=40, Sk=150, D=64, dtype="f32", causal=True, q_offset=110,
                accum=True, seed=63),
    # key tiles cut into parts: the part that finishes last writes the read-back rows
    wl.Workload("rows_split_parts_d64", B=1, Hq=8, Hkv=2, Sq=768, Sk=1024, D=64, causal=True, q_offset=256,
                accum=True, seed=64),
    wl.Workload("rows_planned_full_grid", B=1, Hq=16, Hkv=16, Sq=1280, Sk=1280, D=128, causal=True, q_offset=0,
                accum=True, seed=65),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", FUSED, ids=[w.name for w in FUSED])
@pytest.mark.parametrize("where", ["chunk", "middle"])
def test_fused_read_back_rows(w, where):
    import torch
    from tests import parity_util as pu
    begin, n = (w.q_offset, w.Sq) if where == "chunk" else (w.Sk // 3, w.Sk // 4)
    inputs = wl.make_inputs(w)
    t = pu.to_device(inputs, w)
    kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset, window=w.window)
    o, lse = ft.fwd(t["q"], t["k"], t["v"], t["mask"], **kw)
    dk, dv = t["dk_acc"].clone(), t["dv_acc"].clone()
    dq, dk_rows, dv_rows = ft.bwd_accum_rows(t["q"], t["k"], t["v"], o, lse, t["do"], dk, dv, begin, n, t["mask"],
                                             **kw)
    torch.cuda.synchronize()
    assert ft.device_status() == 0
    out = "bf16" if w.dtype == "bf16" else "f32"
    idx = np.arange(begin, begin + n)
    # the read-back rows are exactly the finished accumulator rows in the input dtype
    for rows, acc in ((dk_rows, dk), (dv_rows, dv)):
        np.testing.assert_array_equal(rows.float().cpu().numpy(),
                                      rows_ref.set_rows_backward(acc.cpu().numpy(), idx, out))
    # and they match the oracle's accumulate-then-read-back
    exp = pu.run_oracle(w, inputs)
    rel, abs_ = pu.TOL[w.dtype]
    for name, rows in (("dk", dk_rows), ("dv", dv_rows)):
        want = rows_ref.set_rows_backward(exp[name], idx)
        err = float(np.abs(rows.double().cpu().numpy() - want).max())
        bound = rel * float(np.abs(want).max()) + abs_ + (float(np.abs(want).max()) * 2.0 ** -8 if out == "bf16" else 0)
        assert err <= bound, f"{name}_rows: {err:.3e} > {bound:.3e}"


@pytest.mark.gpu
def test_fused_read_back_with_no_query_rows_returns_the_accumulator_rows():
    import torch
    rng = np.random.default_rng(64)
    q = torch.zeros((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.from_numpy(rng.standard_normal((1, 1, 90, 128)).astype(np.float32)).cuda().to(torch.bfloat16)
    v = k.clone()
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 2, 0), dtype=torch.float32, device="cuda")
    acc_k = torch.from_numpy(rng.standard_normal((1, 1, 90, 128)).astype(np.float32)).cuda()
    acc_v = acc_k * 2
    before = acc_k.clone()
    _, dk_rows, dv_rows = ft.bwd_accum_rows(q, k, v, o, lse, o, acc_k, acc_v, 10, 30, causal=True, q_offset=90)
    torch.cuda.synchronize()
    assert torch.equal(acc_k, before)
    np.testing.assert_array_equal(dk_rows.float().cpu().numpy(),
                                  rows_ref.set_rows_backward(before.cpu().numpy(), np.arange(10, 40), "bf16"))
