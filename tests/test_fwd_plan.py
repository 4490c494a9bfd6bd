"""The forward's launch (host only): persistent CTAs, one per SM, exactly when the 256-row units
outnumber the SMs and there is no mask and no key split; otherwise one unit (or one key split of
it) per CTA. The expected values are recomputed here from the unit count and the split rule."""
import ctypes

import pytest
import torch

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    ft.load_library()


def _sms():
    # the library asks the device; without one it takes 152 (a GB300)
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def _params(B, Hq, Hkv, Sq, Sk, D=128, dtype=torch.bfloat16, causal=False, window=0, mask=False):
    q = torch.empty((B, Hq, Sq, D), dtype=dtype, device="meta")
    k = torch.empty((B, Hkv, Sk, D), dtype=dtype, device="meta")
    m = torch.empty((1, Sq, Sk), dtype=torch.bool, device="meta") if mask else None
    return ft.make_params(q, k, m, causal=causal, window=window)


def _units(p):
    return p.B * p.Hq * ((p.Sq + 255) // 256)


@pytest.mark.parametrize("shape, persistent", [
    (dict(B=1, Hq=32, Hkv=8, Sq=4096, Sk=4096, causal=True), True),             # causal LM
    (dict(B=1, Hq=32, Hkv=8, Sq=4096, Sk=4096, causal=True, mask=True), False),  # a mask: one unit per CTA
    (dict(B=2, Hq=48, Hkv=12, Sq=600, Sk=600, window=90), True),                 # sliding window, ragged rows
    (dict(B=3, Hq=32, Hkv=4, Sq=257, Sk=333, D=64), True),                       # D = 64
    (dict(B=1, Hq=76, Hkv=38, Sq=512, Sk=512), False),                           # units == SMs (152)
    (dict(B=1, Hq=77, Hkv=7, Sq=512, Sk=512), True),                             # two units more than SMs
    (dict(B=1, Hq=16, Hkv=8, Sq=1024, Sk=1024, D=64), False),                    # DiT self-attention
])
def test_persistent_exactly_when_units_outnumber_sms_without_mask(shape, persistent):
    p = _params(**shape)
    ctas, splits, pers = ft.fwd_plan(p)
    units, sms = _units(p), _sms()
    assert pers == (units > sms and not shape.get("mask", False) and splits == 1)
    if sms == 152:
        assert pers == persistent
    if pers:
        assert ctas == sms
    else:
        assert ctas == units * splits


def test_few_units_over_long_keys_split_the_keys():
    """A 512-row chunk at the end of 67,584 keys has 32 units: the keys are split four waves deep
    (4 x SMs // units), capped at one split per 8 key tiles; one CTA per (unit, split)."""
    p = _params(B=1, Hq=16, Hkv=4, Sq=512, Sk=67584, causal=True)
    ctas, splits, pers = ft.fwd_plan(p)
    units = _units(p)
    kv_tiles = (67584 + 127) // 128
    assert not pers
    assert splits == max(1, min(4 * _sms() // units, kv_tiles // 8))
    assert splits > 1 and ctas == units * splits


def test_fp32_is_not_on_the_tensor_core_path():
    p = _params(B=1, Hq=4, Hkv=4, Sq=300, Sk=300, dtype=torch.float32)
    with pytest.raises(ft.FaError) as e:
        ft.fwd_plan(p)
    assert e.value.status == ft.FA_ERR_UNSUPPORTED


def test_null_outputs_are_rejected():
    lib = ft.load_library()
    p = _params(B=1, Hq=32, Hkv=8, Sq=4096, Sk=4096, causal=True)
    n = ctypes.c_int32(0)
    assert lib.fa_train_fwd_plan(ctypes.byref(p), None, ctypes.byref(n), ctypes.byref(n)) == ft.FA_ERR_INVALID_ARG
