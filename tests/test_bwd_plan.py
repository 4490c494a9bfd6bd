"""The backward's work plan (host only): every key tile of every (batch, kv head) is walked once,
a split key tile's parts partition its query rows, and the rows are the ones the causal rule and
the sliding window let see the tile. The rows are recomputed here from the masking rules."""
import pytest
import torch

from backward_adapter_gb300 import build as fbuild
from backward_adapter_gb300 import fa_train as ft
from backward_adapter_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fbuild.build()
    ft.load_library()


def _params(B, Hq, Hkv, Sq, Sk, D=128, causal=False, q_offset=None, window=0, deterministic=False):
    q = torch.empty((B, Hq, Sq, D), dtype=torch.bfloat16, device="meta")
    k = torch.empty((B, Hkv, Sk, D), dtype=torch.bfloat16, device="meta")
    return ft.make_params(q, k, None, causal=causal, q_offset=q_offset, window=window,
                          deterministic=deterministic)


def _rows(p, kt):
    """Query rows [first, end) in which some row sees a key of tile kt, first rounded down to 128."""
    j0, j1 = 128 * kt, min(128 * kt + 127, p.Sk - 1)
    lo, hi = 0, p.Sq - 1
    if p.causal:
        lo = max(lo, j0 - p.q_offset)
    if p.window > 0:
        lo = max(lo, j0 - p.q_offset - p.window)
        hi = min(hi, j1 - p.q_offset + p.window)
    if lo > hi:
        return None
    return lo // 128 * 128, hi + 1


SHAPES = {
    "causal_lm": dict(B=1, Hq=32, Hkv=8, Sq=4096, Sk=4096, causal=True),
    "causal_lm_b2": dict(B=2, Hq=16, Hkv=4, Sq=4096, Sk=4096, causal=True),
    "causal_long_gqa8": dict(B=1, Hq=64, Hkv=8, Sq=8192, Sk=8192, causal=True),
    "causal_chunk": dict(B=1, Hq=8, Hkv=2, Sq=1000, Sk=5000, causal=True, q_offset=4000),
    "causal_mid": dict(B=3, Hq=6, Hkv=3, Sq=1500, Sk=2600, causal=True, q_offset=700),
    "causal_full_grid_small": dict(B=1, Hq=16, Hkv=16, Sq=1280, Sk=1280, causal=True),
    "causal_full_grid_b2": dict(B=2, Hq=8, Hkv=8, Sq=1280, Sk=1280, causal=True),
    "window": dict(B=1, Hq=16, Hkv=4, Sq=4096, Sk=4096, window=700),
    "dit_self": dict(B=1, Hq=24, Hkv=8, Sq=1024, Sk=1024, D=64),
    "dit_cross": dict(B=2, Hq=16, Hkv=16, Sq=2048, Sk=256),
    "long_window_chunk": dict(B=1, Hq=16, Hkv=4, Sq=512, Sk=67584, window=67072, q_offset=67072),
    "deterministic_causal": dict(B=1, Hq=32, Hkv=8, Sq=4096, Sk=4096, causal=True, deterministic=True),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_plan_walks_every_key_tile_once(name):
    p = _params(**SHAPES[name])
    plan = ft.bwd_plan(p)
    nkt, nbkv = (p.Sk + 127) // 128, p.B * p.Hkv
    parts = {}
    for kt, bkv, part, nparts, first, end in plan:
        assert 0 <= kt < nkt and 0 <= bkv < nbkv and 0 <= part < nparts
        assert (kt, bkv, part) not in parts, "a CTA appears twice"
        parts[(kt, bkv, part)] = (nparts, first, end)
    for kt in range(nkt):
        want = _rows(p, kt)
        for bkv in range(nbkv):
            assert (kt, bkv, 0) in parts, (kt, bkv)
            nparts = parts[(kt, bkv, 0)][0]
            spans = []
            for q in range(nparts):
                n2, first, end = parts.pop((kt, bkv, q))
                assert n2 == nparts
                spans.append((first, end))
            if want is None:
                assert nparts == 1 and spans[0][0] >= spans[0][1], "a key tile nobody sees walks rows"
                continue
            # consecutive parts of whole 128-row query tiles, covering the rows exactly
            assert spans[0][0] == want[0] and spans[-1][1] == want[1], (kt, spans, want)
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0 and a0 < a1 and (a1 - a0) % 128 == 0
    assert not parts, "CTAs outside the key tiles"


def test_causal_plan_splits_the_heaviest_key_tiles():
    """On a full grid the first key tiles of a causal backward have far more query tiles than the
    per-SM share: they are cut, and no CTA walks all of them."""
    p = _params(**SHAPES["causal_lm"])
    plan = ft.bwd_plan(p)
    G = p.Hq // p.Hkv
    steps = [G * ((end - first) // 128) for _, _, _, _, first, end in plan]
    assert any(r[3] > 1 for r in plan)
    assert max(steps) < G * 32
    assert len(plan) > 32 * p.B * p.Hkv


@pytest.mark.parametrize("name", ["causal_full_grid_small", "causal_full_grid_b2"])
def test_small_full_grids_take_the_planned_order(name):
    """The shapes the GPU parity cases use for the planned split: a full grid, parts, and a launch
    order other than key-tile-major."""
    p = _params(**SHAPES[name])
    plan = ft.bwd_plan(p)
    nkt, nbkv = (p.Sk + 127) // 128, p.B * p.Hkv
    assert nkt * nbkv >= 152
    assert any(r[3] > 1 for r in plan) and len(plan) > nkt * nbkv


def test_deterministic_plan_keeps_key_tile_order():
    p = _params(**SHAPES["deterministic_causal"])
    plan = ft.bwd_plan(p)
    nbkv = p.B * p.Hkv
    assert [(r[0], r[1], r[3]) for r in plan] == [(i // nbkv, i % nbkv, 1) for i in range(len(plan))]


def test_plan_is_stable_across_calls():
    p = _params(**SHAPES["causal_mid"])
    assert ft.bwd_plan(p) == ft.bwd_plan(p)
    for w in (wl.CAUSAL_LM, wl.DIT_SELF):
        q = _params(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, D=w.D, causal=w.causal, q_offset=w.q_offset, window=w.window)
        assert ft.bwd_plan(q) == ft.bwd_plan(q)
