"""The binding checks every tensor against the parameters before the C ABI sees a pointer.

The library receives bare device pointers, so a tensor of the wrong shape would reach the kernels
as out-of-bounds accesses. These run on the CPU: tensors with consistent shapes get as far as the
device check (they are not CUDA tensors), inconsistent ones are refused before it.
"""
import pytest
import torch

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft

B, HQ, HKV, SQ, SK, D = 2, 4, 2, 40, 70, 64
CUDA_ERR = "contiguous CUDA tensor"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    ft.load_library()


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _args(layout="bhsd", kv_dtype=torch.bfloat16):
    if layout == "bhsd":
        qs, ks = (B, HQ, SQ, D), (B, HKV, SK, D)
    else:
        qs, ks = (B, SQ, HQ, D), (B, SK, HKV, D)
    return dict(q=_t(*qs), k=_t(*ks, dtype=kv_dtype), v=_t(*ks, dtype=kv_dtype), o=_t(*qs),
                lse=_t(B, HQ, SQ, dtype=torch.float32), do=_t(*qs)), qs, ks


def _bwd_args(a):
    return a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"]


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float16])
def test_consistent_shapes_reach_the_device_check(layout, kv_dtype):
    a, qs, ks = _args(layout, kv_dtype)
    mask = _t(1, SQ, SK, dtype=torch.bool)
    calls = [
        lambda: ft.fwd(a["q"], a["k"], a["v"], mask, layout=layout, causal=True),
        lambda: ft.fwd(a["q"], a["k"], a["v"], layout=layout, out=_t(*qs), lse=_t(B, HQ, SQ, dtype=torch.float32)),
        lambda: ft.bwd(*_bwd_args(a), mask, layout=layout),
        lambda: ft.bwd(*_bwd_args(a), layout=layout, dq=_t(*qs), dk=_t(*ks), dv=_t(*ks)),
        lambda: ft.bwd_accum(*_bwd_args(a), _t(*ks, dtype=torch.float32), _t(*ks, dtype=torch.float32), layout=layout),
        lambda: ft.bwd_accum_rows(*_bwd_args(a), _t(*ks, dtype=torch.float32), _t(*ks, dtype=torch.float32), 10, 30,
                                  layout=layout, causal=True),
        lambda: ft.bwd_noalloc(*_bwd_args(a), layout=layout),
    ]
    for call in calls:
        with pytest.raises(ValueError, match=CUDA_ERR):
            call()


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_q8_planes_reach_the_device_check(layout):
    a, qs, ks = _args(layout)
    planes = (_t(B, HKV, SK, D, dtype=torch.int8), _t(B, HKV, SK, D // 32, dtype=torch.float16),
              _t(B, HKV, SK, D, dtype=torch.int8), _t(B, HKV, SK, D // 32, dtype=torch.float16))
    with pytest.raises(ValueError, match=CUDA_ERR):
        ft.fwd_q8(a["q"], *planes, layout=layout)
    with pytest.raises(ValueError, match=CUDA_ERR):
        ft.bwd_q8(a["q"], *planes, a["o"], a["lse"], a["do"], layout=layout)
    with pytest.raises(ValueError, match=CUDA_ERR):
        ft.bwd_q8(a["q"], *planes, a["o"], a["lse"], a["do"], layout=layout,
                  dk_acc=_t(*ks, dtype=torch.float32), dv_acc=_t(*ks, dtype=torch.float32))
    bad = (planes[0], _t(B, HKV, SK, D // 16, dtype=torch.float16), planes[2], planes[3])
    with pytest.raises(ValueError, match="k_d has shape"):
        ft.fwd_q8(a["q"], *bad, layout=layout)


def test_inconsistent_shapes_and_dtypes_are_refused():
    a, qs, ks = _args()
    cases = [
        (lambda: ft.fwd(a["q"], a["k"], _t(B, HKV, SK - 1, D)), ValueError, "v has shape"),
        (lambda: ft.fwd(a["q"], a["k"], a["v"], _t(1, SQ, SK + 1, dtype=torch.float32)), ValueError, "mask has shape"),
        (lambda: ft.fwd(a["q"], a["k"], a["v"], out=_t(B, HQ, SQ, D, dtype=torch.float32)), TypeError, "o has dtype"),
        (lambda: ft.fwd(a["q"], a["k"], a["v"], lse=_t(B, HQ, SQ + 1, dtype=torch.float32)), ValueError,
         "lse has shape"),
        (lambda: ft.bwd(a["q"], a["k"], a["v"], _t(B, HQ, SQ, D // 2), a["lse"], a["do"]), ValueError, "o has shape"),
        (lambda: ft.bwd(*_bwd_args(a), dk=_t(B, HKV, SK, D, dtype=torch.float16)), TypeError, "dk has dtype"),
        (lambda: ft.bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], _t(B, HQ, SQ - 1, D)), ValueError, "do has shape"),
        (lambda: ft.bwd_accum(*_bwd_args(a), _t(*ks, dtype=torch.float32), _t(B, HKV, SK, D - 1, dtype=torch.float32)),
         ValueError, "dv_acc has shape"),
        (lambda: ft.bwd_accum_rows(*_bwd_args(a), _t(*ks, dtype=torch.float32), _t(*ks, dtype=torch.float32), 0, 5,
                                   dk_rows=_t(B, HKV, 6, D)), ValueError, "dk_rows has shape"),
        (lambda: ft.fwd(a["q"], _t(B, HKV, SK, D, dtype=torch.float16), _t(B, HKV, SK, D)), TypeError,
         "one dtype"),
        (lambda: ft.fwd(_t(B, HQ, SQ, D, dtype=torch.float32), _t(B, HKV, SK, D, dtype=torch.float16),
                        _t(B, HKV, SK, D, dtype=torch.float16)), TypeError, "float16 under bfloat16"),
        (lambda: ft.fwd(a["q"][0], a["k"], a["v"]), ValueError, "4-D"),
        (lambda: ft.set_rows_backward(_t(B, HKV, SK, D, dtype=torch.float32), torch.zeros(5, dtype=torch.int64),
                                      out=_t(B, HKV, 4, D)), ValueError, "out has shape"),
    ]
    for call, exc, msg in cases:
        with pytest.raises(exc, match=msg):
            call()


def _gpu_test_workloads():
    from backward_adapter_gb300 import workloads as wl
    from tests import test_kv_f16, test_kv_q8, test_layout_bshd, test_parity_gpu
    ws = list(test_parity_gpu.SMALL) + list(test_kv_q8.CASES) + list(test_kv_f16.CASES) + list(test_layout_bshd.CASES)
    return ws + [wl.DIT_SELF, wl.DIT_SELF_WINDOW, wl.DIT_CROSS, wl.LONG_WINDOW_F16]


def test_every_gpu_test_call_pattern_passes_the_checks():
    """The argument patterns of the GPU tests (run_gpu, the layout comparison) on CPU copies of
    their inputs: each call gets as far as the device check."""
    from backward_adapter_gb300 import workloads as wl
    from tests import parity_util as pu
    for w in _gpu_test_workloads():
        t = pu.to_device(wl.make_inputs(w), w, device="cpu")
        for layout in ("bhsd", "bshd"):
            T = (lambda x: x) if layout == "bhsd" else (lambda x: x.transpose(1, 2).contiguous())  # noqa: E731
            kw = dict(scale=w.scale, causal=w.causal, q_offset=w.q_offset, window=w.window, layout=layout)
            q, do = T(t["q"]), T(t["do"])
            o, lse = torch.empty_like(q), torch.empty(q.shape[0], w.Hq, w.Sq, dtype=torch.float32)
            if w.kv_format == "q8_0":
                kv = (t["k_q"], t["k_d"], t["v_q"], t["v_d"])
                calls = [lambda: ft.fwd_q8(q, *kv, t["mask"], **kw),
                         lambda: ft.bwd_q8(q, *kv, o, lse, do, t["mask"], deterministic=True, **kw)]
                if w.accum:
                    calls.append(lambda: ft.bwd_q8(q, *kv, o, lse, do, t["mask"], dk_acc=T(t["dk_acc"]),
                                                   dv_acc=T(t["dv_acc"]), **kw))
            else:
                k, v = T(t["k"]), T(t["v"])
                calls = [lambda: ft.fwd(q, k, v, t["mask"], **kw),
                         lambda: ft.bwd(q, k, v, o, lse, do, t["mask"], deterministic=True, **kw)]
                if w.accum:
                    acc = (T(t["dk_acc"]), T(t["dv_acc"]))
                    calls += [lambda: ft.bwd_accum(q, k, v, o, lse, do, *acc, t["mask"], **kw),
                              lambda: ft.bwd_accum_rows(q, k, v, o, lse, do, *acc, w.q_offset, w.Sq, t["mask"], **kw)]
            for call in calls:
                with pytest.raises(ValueError, match=CUDA_ERR):
                    call()


def test_empty_chunk_and_explicit_buffer_patterns_pass_the_checks():
    # an empty query chunk (Sq = 0), with and without the fused read-back
    q = _t(1, 2, 0, 128)
    k = _t(1, 1, 90, 128)
    o, lse = torch.zeros_like(q), _t(1, 2, 0, dtype=torch.float32)
    acc = _t(1, 1, 90, 128, dtype=torch.float32)
    for call in (lambda: ft.fwd(q, k, k),
                 lambda: ft.bwd(q, k, k, o, lse, o, dk=torch.full_like(k, 7.0), dv=torch.full_like(k, 7.0)),
                 lambda: ft.bwd_accum_rows(q, k, k, o, lse, o, acc, acc.clone(), 10, 30, causal=True, q_offset=90)):
        with pytest.raises(ValueError, match=CUDA_ERR):
            call()
    # the benchmark's calls: every output and the workspace given explicitly
    a, qs, ks = _args()
    ws = _t(1 << 10, dtype=torch.uint8)
    with pytest.raises(ValueError, match=CUDA_ERR):
        ft.fwd(a["q"], a["k"], a["v"], None, out=_t(*qs), lse=_t(B, HQ, SQ, dtype=torch.float32), workspace=ws,
               causal=True)
    with pytest.raises(ValueError, match=CUDA_ERR):
        ft.bwd(*_bwd_args(a), None, dq=_t(*qs), dk=_t(*ks), dv=_t(*ks), workspace=ws, deterministic=True)
    rows = (B, HKV, SQ, D)
    with pytest.raises(ValueError, match=CUDA_ERR):
        ft.bwd_accum_rows(*_bwd_args(a), _t(*ks, dtype=torch.float32), _t(*ks, dtype=torch.float32), SK - SQ, SQ, None,
                          dq=_t(*qs), dk_rows=_t(*rows), dv_rows=_t(*rows), workspace=ws, causal=True)
