"""The allocation-free backward, fa_train_bwd_noalloc.

It serves callers that cannot allocate device memory: their GPU memory belongs to
another allocator (a framework pool, or a plugin host that hands over only its own
tensors), or they run where a cudaMalloc and the synchronisation it can bring are
not allowed. It keeps its scratch in one 16 MiB static device array inside the
library. These tests check that it gives the same results as the workspace entry
point, on two calls in a row (the array keeps the previous call's contents), and
that shapes needing more scratch are refused before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl


def test_shapes_beyond_the_static_scratch_are_refused_before_any_launch():
    fbuild.build()
    lib = ft.load_library()
    # causal LM shape: 64.5 MiB of backward scratch, more than the 16 MiB array
    p = ft.FaParams(1, 32, 8, 4096, 4096, 128, ft.FA_BF16, 0.088, 1, ft.FA_MASK_NONE, 1, 0, 0)
    assert ft.bwd_workspace_size(p) > ft.NOALLOC_SCRATCH_BYTES
    fake = 1 << 34  # never dereferenced: the size check comes first
    st = lib.fa_train_bwd_noalloc(ctypes.byref(p), fake, 2 * fake, 3 * fake, None, 4 * fake, 5 * fake, 6 * fake,
                                  7 * fake, 8 * fake, 9 * fake, None)
    assert st == ft.FA_ERR_WORKSPACE
    assert str(ft.NOALLOC_SCRATCH_BYTES).encode() in lib.fa_last_error()


CASES = [
    wl.Workload("noalloc_causal_offset_d128", B=1, Hq=4, Hkv=2, Sq=700, Sk=900, D=128, causal=True, q_offset=200,
                seed=41),
    wl.Workload("noalloc_bool_mask_d64", B=2, Hq=4, Hkv=1, Sq=300, Sk=260, D=64, mask="random_bool", seed=42),
    # the fp32 path (SIMT kernels) and the ordered dQ adds (turn counters in the static array)
    wl.Workload("noalloc_f32_causal_d64", B=1, Hq=4, Hkv=2, Sq=90, Sk=130, D=64, dtype="f32", causal=True,
                q_offset=40, seed=43),
    wl.Workload("noalloc_deterministic_causal_d128", B=1, Hq=4, Hkv=1, Sq=400, Sk=400, D=128, causal=True, seed=44),
]


def _deterministic(w):
    return w.name.startswith("noalloc_deterministic")


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_backward_matches_workspace_backward_on_two_calls(w):
    import torch

    from tests import parity_util as pu

    inputs = wl.make_inputs(w)
    t = pu.to_device(inputs, w)
    kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset, deterministic=_deterministic(w))
    fkw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset)
    o, lse = ft.fwd(t["q"], t["k"], t["v"], t["mask"], **fkw)
    ref = ft.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], t["mask"], **kw)
    torch.cuda.synchronize()
    ref = [x.double().cpu().numpy() for x in ref]
    rel, abs_ = pu.TOL[w.dtype]
    for call in range(2):
        got = ft.bwd_noalloc(t["q"], t["k"], t["v"], o, lse, t["do"], t["mask"], **kw)
        torch.cuda.synchronize()
        assert ft.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            g = g.double().cpu().numpy()
            if _deterministic(w):
                # same kernels, same ordered adds: the same bits as the workspace backward
                assert np.array_equal(g, r), f"call {call}: deterministic {name} differs from the workspace backward"
            err = float(np.abs(g - r).max())
            bound = rel * float(np.abs(r).max()) + abs_
            assert err <= bound, f"call {call}: {name} differs from the workspace backward by {err:.3e} > {bound:.3e}"


@pytest.mark.gpu
def test_noalloc_backward_matches_the_oracle():
    """One case compared with the fp64 oracle directly, not only with the workspace backward."""
    import torch

    from tests import parity_util as pu

    w = CASES[0]
    inputs = wl.make_inputs(w)
    t = pu.to_device(inputs, w)
    kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset)
    o, lse = ft.fwd(t["q"], t["k"], t["v"], t["mask"], **kw)
    dq, dk, dv = ft.bwd_noalloc(t["q"], t["k"], t["v"], o, lse, t["do"], t["mask"], **kw)
    torch.cuda.synchronize()
    assert ft.device_status() == 0
    got = {n: x.double().cpu().numpy() for n, x in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    pu.assert_parity(w, got, pu.run_oracle(w, inputs))
