"""Host-only checks of the C-ABI library: it builds, loads without a GPU, exports
every symbol the header declares, agrees with the header's struct layout, and
rejects invalid calls before touching CUDA."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_train.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    fbuild.build()
    return ft.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(ft.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", fbuild.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)", nm))
    assert set(declared_functions()) <= exported
    assert not [s for s in exported if s.startswith("_ZN2fa")], "internal C++ symbols leak from the library"


def test_struct_layout_matches_header(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "fa_train.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(fa_params), offsetof(fa_params, scale),'
                   ' offsetof(fa_params, mask_batch), offsetof(fa_params, q_offset), offsetof(fa_params, deterministic),'
                   ' offsetof(fa_params, kv_format), offsetof(fa_params, layout), sizeof(fa_status));return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    P = ft.FaParams
    assert [int(x) for x in got] == [ctypes.sizeof(P), P.scale.offset, P.mask_batch.offset, P.q_offset.offset,
                                     P.deterministic.offset, P.kv_format.offset, P.layout.offset,
                                     ctypes.sizeof(ctypes.c_int)]


def good_params(**kw):
    p = ft.FaParams(1, 4, 2, 100, 130, 64, ft.FA_BF16, 0.125, 0, ft.FA_MASK_NONE, 1, 0, 0)
    for k_, v_ in kw.items():
        setattr(p, k_, v_)
    return p


BAD = [
    ("B0", dict(B=0), ft.FA_ERR_INVALID_ARG),
    ("gqa_ratio", dict(Hq=3, Hkv=2), ft.FA_ERR_INVALID_ARG),
    ("Hkv0", dict(Hkv=0), ft.FA_ERR_INVALID_ARG),
    ("Sk0", dict(Sk=0), ft.FA_ERR_INVALID_ARG),
    ("Sq_neg", dict(Sq=-1), ft.FA_ERR_INVALID_ARG),
    ("D96", dict(D=96), ft.FA_ERR_UNSUPPORTED),
    ("D0", dict(D=0), ft.FA_ERR_INVALID_ARG),
    ("dtype", dict(dtype=7), ft.FA_ERR_INVALID_ARG),
    ("scale_nan", dict(scale=float("nan")), ft.FA_ERR_INVALID_ARG),
    ("causal2", dict(causal=2), ft.FA_ERR_INVALID_ARG),
    ("mask_kind", dict(mask_kind=5), ft.FA_ERR_INVALID_ARG),
    ("mask_batch", dict(mask_kind=ft.FA_MASK_ADD_F32, mask_batch=3), ft.FA_ERR_INVALID_ARG),
    ("window_negative", dict(window=-1), ft.FA_ERR_INVALID_ARG),
    ("deterministic2", dict(deterministic=2), ft.FA_ERR_INVALID_ARG),
    ("kv_format", dict(kv_format=3), ft.FA_ERR_INVALID_ARG),
    ("kv_f16_needs_bf16", dict(kv_format=2, dtype=0), ft.FA_ERR_UNSUPPORTED),
    ("layout", dict(layout=2), ft.FA_ERR_INVALID_ARG),
    ("reserved", dict(reserved=1), ft.FA_ERR_INVALID_ARG),
    ("q_too_large", dict(B=65535, Hq=65535, Hkv=65535, Sq=1 << 16), ft.FA_ERR_INVALID_ARG),
    ("kv_too_large", dict(B=1024, Hq=4096, Hkv=4096, Sk=1 << 24), ft.FA_ERR_INVALID_ARG),
    ("mask_too_large", dict(B=65535, Sq=1 << 20, Sk=1 << 20, mask_kind=ft.FA_MASK_BOOL_U8, mask_batch=65535),
     ft.FA_ERR_INVALID_ARG),
    ("window_offset_too_big", dict(window=8, q_offset=31), ft.FA_ERR_INVALID_ARG),
    ("causal_offset_too_big", dict(causal=1, q_offset=31), ft.FA_ERR_INVALID_ARG),
    ("causal_offset_negative", dict(causal=1, q_offset=-1), ft.FA_ERR_INVALID_ARG),
]


@pytest.mark.parametrize("name,kw,code", BAD, ids=[b[0] for b in BAD])
def test_invalid_params_are_rejected_before_launch(lib, name, kw, code):
    p = good_params(**kw)
    fake = 1 << 20  # never dereferenced: validation fails first
    st = lib.fa_train_fwd(ctypes.byref(p), fake, fake, fake, None, fake, fake, None, 0, None)
    assert st == code, lib.fa_last_error()
    assert lib.fa_last_error().decode() != ""
    st = lib.fa_train_bwd(ctypes.byref(p), fake, fake, fake, None, fake, fake, fake, fake, fake, fake, None, 0, None)
    assert st == code
    assert lib.fa_train_fwd_workspace_size(ctypes.byref(p)) == 0


def test_null_and_misaligned_pointers_are_rejected(lib):
    p = good_params()
    assert lib.fa_train_fwd(None, 16, 16, 16, None, 16, 16, None, 0, None) == ft.FA_ERR_INVALID_ARG
    st = lib.fa_train_fwd(ctypes.byref(p), None, 1 << 30, 2 << 30, None, 3 << 30, 4 << 30, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"q is NULL" in lib.fa_last_error()
    st = lib.fa_train_fwd(ctypes.byref(p), (1 << 30) + 8, 2 << 30, 3 << 30, None, 4 << 30, 5 << 30, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"aligned" in lib.fa_last_error()
    # an additive mask kind without a mask pointer
    pm = good_params(mask_kind=ft.FA_MASK_ADD_F32)
    st = lib.fa_train_fwd(ctypes.byref(pm), 1 << 30, 2 << 30, 3 << 30, None, 4 << 30, 5 << 30, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"mask is NULL" in lib.fa_last_error()


def test_aliasing_outputs_are_rejected(lib):
    p = good_params()
    base = 1 << 32
    # o overlaps q
    st = lib.fa_train_fwd(ctypes.byref(p), base, 2 * base, 3 * base, None, base + 4096, 4 * base, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"overlaps" in lib.fa_last_error()
    # dk and dv the same buffer
    st = lib.fa_train_bwd(ctypes.byref(p), base, 2 * base, 3 * base, None, 4 * base, 5 * base, 6 * base,
                          7 * base, 8 * base, 8 * base, 9 * base, 1 << 30, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"overlap" in lib.fa_last_error()


def test_workspace_too_small_is_rejected(lib):
    p = good_params()
    need = lib.fa_train_bwd_workspace_size(ctypes.byref(p))
    assert need > 0
    base = 1 << 32
    st = lib.fa_train_bwd(ctypes.byref(p), base, 2 * base, 3 * base, None, 4 * base, 5 * base, 6 * base,
                          7 * base, 8 * base, 9 * base, 10 * base, need - 1, None)
    assert st == ft.FA_ERR_WORKSPACE


def test_workspace_sizes_scale_with_shape(lib):
    small = good_params()
    big = good_params(Sq=1000)
    assert lib.fa_train_bwd_workspace_size(ctypes.byref(big)) > lib.fa_train_bwd_workspace_size(ctypes.byref(small))


def test_status_strings(lib):
    for code in range(5):
        assert lib.fa_status_str(code)
    assert lib.fa_status_str(99) == b"unknown status"


def test_kv_format_must_match_the_entry_point(lib):
    p = good_params(kv_format=ft.FA_KV_Q8_0)
    fake = 1 << 20
    st = lib.fa_train_fwd(ctypes.byref(p), fake, fake, fake, None, fake, fake, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"_q8" in lib.fa_last_error()
    # the q8 forward's workspace holds the dequantized bf16 K and V
    plain = good_params()
    extra = lib.fa_train_fwd_workspace_size(ctypes.byref(p)) - lib.fa_train_fwd_workspace_size(ctypes.byref(plain))
    assert extra >= 2 * 1 * 2 * 130 * 64 * 2


def test_f16_cache_workspace_holds_the_bf16_copy(lib):
    # an fp16 K/V cache under bf16 queries: both passes cast K and V to bf16 in the workspace
    f16 = good_params(kv_format=ft.FA_KV_F16)
    plain = good_params()
    copy = 2 * f16.B * f16.Hkv * f16.Sk * f16.D * 2
    for size in (lib.fa_train_fwd_workspace_size, lib.fa_train_bwd_workspace_size):
        extra = size(ctypes.byref(f16)) - size(ctypes.byref(plain))
        assert copy <= extra < copy + 512
    # the plain entry points take it; the _q8 ones refuse it
    kv = ft.FaKvQ8(1 << 20, 1 << 20, 1 << 20, 1 << 20)
    st = lib.fa_train_fwd_q8(ctypes.byref(f16), 1 << 20, ctypes.byref(kv), None, 1 << 20, 1 << 20, None, 0, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"_q8" in lib.fa_last_error()


def test_set_rows_backward_refuses_sizes_that_overflow(lib):
    st = lib.fa_set_rows_backward(1 << 20, 65535, 32767, 1 << 24, 1024, 1 << 20, 1, 2 << 20, ft.FA_BF16, None)
    assert st == ft.FA_ERR_INVALID_ARG and b"2^40" in lib.fa_last_error()

