"""GPU parity: the CUDA path (called through the C-ABI) against the fp64 oracle
on the same seeded inputs, element by element."""
import numpy as np
import pytest
import torch

from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

W = wl.Workload
SMALL = [
    wl.TINY_F32,
    W("f32_causal_offset_d128", B=1, Hq=4, Hkv=2, Sq=70, Sk=150, D=128, dtype="f32", causal=True,
      q_offset=80, seed=11),
    W("f32_bool_mask_gqa", B=2, Hq=4, Hkv=1, Sq=45, Sk=97, D=64, dtype="f32", mask="random_bool", seed=12),
    W("bf16_plain_d64_ragged", B=2, Hq=4, Hkv=2, Sq=200, Sk=333, D=64, seed=13),
    W("bf16_causal_d128", B=1, Hq=4, Hkv=1, Sq=300, Sk=300, D=128, causal=True, seed=14),
    W("bf16_causal_offset_accum", B=1, Hq=4, Hkv=2, Sq=130, Sk=517, D=128, causal=True, q_offset=387,
      accum=True, seed=15),
    W("bf16_random_add_mask_d64", B=2, Hq=2, Hkv=2, Sq=257, Sk=190, D=64, mask="random_add", seed=16),
    W("bf16_random_bool_d128", B=2, Hq=4, Hkv=1, Sq=129, Sk=385, D=128, mask="random_bool", seed=17),
    W("bf16_mask_and_causal", B=1, Hq=2, Hkv=1, Sq=200, Sk=260, D=128, mask="random_add", causal=True,
      q_offset=60, seed=18),
    W("bf16_pad_self_small", B=1, Hq=4, Hkv=2, Sq=300, Sk=300, D=64, mask="pad_self", seed=19),
    W("bf16_cross_small", B=2, Hq=2, Hkv=2, Sq=260, Sk=256, D=128, mask="cross", seed=20),
    W("bf16_single_key", B=1, Hq=2, Hkv=1, Sq=33, Sk=1, D=64, seed=21),
    W("bf16_single_query", B=1, Hq=2, Hkv=2, Sq=1, Sk=700, D=128, causal=True, q_offset=699, seed=22),
    W("bf16_long_keys_small_q", B=1, Hq=4, Hkv=1, Sq=64, Sk=5000, D=128, causal=True, q_offset=4936,
      accum=True, seed=23),
    # a query chunk in the middle of the keys: key tiles past the chunk have no step at all
    W("bf16_causal_chunk_mid", B=1, Hq=4, Hkv=2, Sq=150, Sk=600, D=128, causal=True, q_offset=100, seed=30),
    # sliding window (half-width w: |q_offset + i - j| <= w)
    W("f32_window_offset", B=1, Hq=2, Hkv=1, Sq=70, Sk=150, D=64, dtype="f32", q_offset=40, window=20,
      seed=31),
    W("bf16_window_d128_ragged", B=1, Hq=4, Hkv=2, Sq=900, Sk=900, D=128, window=130, seed=32),
    W("bf16_window_pad_self_d64", B=1, Hq=4, Hkv=2, Sq=700, Sk=700, D=64, window=100, mask="pad_self", seed=33),
    W("bf16_window_narrow_bool", B=2, Hq=2, Hkv=1, Sq=400, Sk=400, D=128, window=5, mask="random_bool",
      seed=34),
    W("bf16_window_causal_accum", B=1, Hq=4, Hkv=1, Sq=300, Sk=1000, D=128, causal=True, q_offset=650,
      window=200, accum=True, seed=35),
    W("bf16_window_chunk_mid_d64", B=1, Hq=2, Hkv=2, Sq=200, Sk=900, D=64, q_offset=100, window=64, seed=36),
    # a full grid whose first causal key tiles are cut in two and packed onto the SMs ahead of time
    # (the part that finishes last sums the parts)
    W("bf16_full_grid_planned_split", B=1, Hq=16, Hkv=16, Sq=1280, Sk=1280, D=128, causal=True, seed=37),
    W("bf16_full_grid_planned_accum", B=2, Hq=8, Hkv=8, Sq=1280, Sk=1280, D=128, causal=True, accum=True, seed=38),
    W("bf16_full_grid_planned_bool_mask", B=2, Hq=8, Hkv=8, Sq=1280, Sk=1280, D=128, causal=True, mask="random_bool",
      seed=39),
    # more 256-row query units than SMs: persistent forward CTAs chain several units each (the
    # next unit's loads and first score MMAs overlapping the current one's epilogue)
    W("bf16_persistent_causal_gqa_ragged", B=4, Hq=24, Hkv=6, Sq=500, Sk=500, D=128, causal=True, seed=40),
    W("bf16_persistent_offset_d64", B=2, Hq=40, Hkv=8, Sq=300, Sk=700, D=64, causal=True, q_offset=400, seed=41),
    W("bf16_persistent_window", B=2, Hq=48, Hkv=12, Sq=600, Sk=600, D=128, window=90, seed=42),
    W("bf16_persistent_plain_accum_d64", B=3, Hq=32, Hkv=4, Sq=257, Sk=333, D=64, accum=True, seed=43),
    # ... but not under a mask (its tile map may skip every key tile of a unit): one unit per CTA
    W("bf16_many_units_bool_mask", B=2, Hq=24, Hkv=6, Sq=600, Sk=600, D=128, causal=True, mask="random_bool",
      seed=44),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_workloads_match_oracle(w):
    inputs = wl.make_inputs(w)
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    exp = pu.run_oracle(w, inputs)
    pu.assert_parity(w, got, exp)
    pu.assert_exact_zeros(w, inputs, got)


def test_broadcast_mask_over_batch():
    w = W("bf16_bcast_mask", B=2, Hq=2, Hkv=1, Sq=150, Sk=140, D=64, mask="random_add", seed=24)
    inputs = wl.make_inputs(w)
    inputs["mask"] = inputs["mask"][:1].copy()
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    exp = pu.run_oracle(w, inputs)
    pu.assert_parity(w, got, exp)


def test_empty_query_chunk_zeroes_gradients():
    w = W("bf16_empty", B=1, Hq=2, Hkv=1, Sq=0, Sk=100, D=64, seed=25)
    t = pu.to_device(wl.make_inputs(w), w)
    o, lse = ft.fwd(t["q"], t["k"], t["v"])
    dk = torch.full_like(t["k"], 7.0)
    dv = torch.full_like(t["v"], 7.0)
    ft.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert o.numel() == 0 and torch.all(dk == 0) and torch.all(dv == 0)


def test_dirty_pad_is_bitwise_invisible():
    """Garbage in hidden key/value columns leaves every output bit-identical."""
    w = W("bf16_dirty_pad", B=2, Hq=4, Hkv=2, Sq=256, Sk=256, D=128, mask="cross", seed=26)
    inputs = wl.make_inputs(w)
    t = pu.to_device(inputs, w)
    a = pu.run_gpu(w, t)
    lens = wl.cross_lengths(w)
    for b in range(w.B):
        t["k"][b, :, lens[b]:] = 300.0
        t["v"][b, :, lens[b]:] = -200.0
    bb = pu.run_gpu(w, t)
    for n in ("o", "lse", "dq"):
        assert np.array_equal(a[n], bb[n]), n
    for b in range(w.B):
        assert np.array_equal(a["dk"][b, :, :lens[b]], bb["dk"][b, :, :lens[b]])
        assert np.array_equal(a["dv"][b, :, :lens[b]], bb["dv"][b, :, :lens[b]])


DETERMINISTIC = [
    W("det_causal_gqa_d128", B=1, Hq=8, Hkv=2, Sq=640, Sk=640, D=128, causal=True, seed=71),
    W("det_cross_skip_tiles_d128", B=2, Hq=2, Hkv=2, Sq=300, Sk=520, D=128, mask="cross", seed=72),
    W("det_window_pad_d64", B=1, Hq=4, Hkv=2, Sq=700, Sk=700, D=64, window=100, mask="pad_self", seed=73),
    W("det_causal_offset_accum_d64", B=1, Hq=4, Hkv=1, Sq=200, Sk=900, D=64, causal=True, q_offset=700,
      accum=True, seed=74),
    W("det_window_chunk_mid_d128", B=1, Hq=2, Hkv=1, Sq=300, Sk=1000, D=128, q_offset=200, window=150, seed=75),
    # many more key tiles than query tiles: groups of 8 key tiles, two accumulators summed in order
    W("det_long_keys_two_groups_of_8", B=1, Hq=4, Hkv=1, Sq=128, Sk=1500, D=128, causal=True, q_offset=1372,
      seed=76),
    # a causal square past 32 key tiles: two groups of 32
    W("det_causal_two_groups_of_32", B=1, Hq=1, Hkv=1, Sq=4224, Sk=4224, D=64, causal=True, seed=77),
]


@pytest.mark.parametrize("w", DETERMINISTIC, ids=[w.name for w in DETERMINISTIC])
def test_deterministic_dq_is_bitwise_reproducible_and_matches_oracle(w):
    """With deterministic set, dQ (whose partials come from many key tiles) is bitwise identical
    from run to run, including tiles the mask skips; every output still matches the oracle."""
    inputs = wl.make_inputs(w)
    t = pu.to_device(inputs, w)
    runs = [pu.run_gpu(w, t, deterministic=True) for _ in range(3)]
    for n in ("o", "lse", "dq", "dk", "dv"):
        for r in runs[1:]:
            assert np.array_equal(runs[0][n], r[n]), n
    exp = pu.run_oracle(w, inputs)
    pu.assert_parity(w, runs[0], exp)
    pu.assert_exact_zeros(w, inputs, runs[0])


def test_dk_dv_are_deterministic():
    w = W("bf16_determinism", B=1, Hq=8, Hkv=2, Sq=512, Sk=512, D=128, causal=True, seed=27)
    t = pu.to_device(wl.make_inputs(w), w)
    a, b = pu.run_gpu(w, t), pu.run_gpu(w, t)
    for n in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[n], b[n]), n


# ---- full-size workloads ------------------------------------------------------------------------

@pytest.mark.parametrize("w", [wl.DIT_SELF, wl.DIT_SELF_WINDOW, wl.DIT_CROSS], ids=lambda w: w.name)
def test_full_dit_workloads_match_oracle(w):
    inputs = wl.make_inputs(w)
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    exp = pu.run_oracle(w, inputs)
    pu.assert_parity(w, got, exp)
    pu.assert_exact_zeros(w, inputs, got)


FULL_SIZE = [wl.CAUSAL_LM, wl.LONG_WINDOW, wl.LONG_WINDOW_F16, wl.LONG_WINDOW_Q8]


@pytest.mark.parametrize("w", FULL_SIZE, ids=lambda w: w.name)
def test_full_size_workloads_match_oracle_on_every_group(w):
    """At full size the oracle checks every GQA group, one at a time (each group's query heads and
    the key/value head they share: every output they own); over an fp16 or q8_0 cache LSE may also
    move by the kernels' bf16 rounding of the keys. The GPU runs the whole op once, in the launch
    configuration the benchmark times."""
    inputs = wl.make_inputs(w)
    got = pu.run_gpu(w, pu.to_device(inputs, w))
    G = w.Hq // w.Hkv
    for kv in range(w.Hkv):
        qh = list(range(kv * G, (kv + 1) * G))
        exp = pu.run_oracle(w, inputs, q_heads=qh, kv_heads=[kv])
        sub = {"o": got["o"][:, qh], "lse": got["lse"][:, qh], "dq": got["dq"][:, qh],
               "dk": got["dk"][:, [kv]], "dv": got["dv"][:, [kv]]}
        pu.assert_parity(w, sub, exp, where=f" kv-head {kv}",
                         lse_extra=pu.cache_lse_allowance(w, inputs, q_heads=qh, kv_heads=[kv]))
