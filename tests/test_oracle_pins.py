"""Pins of the fp64 oracle against facts the pages and mathematics fix.

None of these re-type the oracle's formula: they check it against finite
differences, closed forms, invariants, a library routine (PyTorch's
scaled_dot_product_attention with autograd, in float64) and the conventions
the pages state (fully-masked rows give O = 0 and LSE = 0; a masked key
column gets exactly zero gradient; GQA equals explicitly expanded heads).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as ref
from backward_adapter_gb300 import workloads as wl


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _tiny(seed=0, B=1, Hq=2, Hkv=1, Sq=5, Sk=7, D=4):
    rng = np.random.default_rng(seed)
    return (_rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D),
            _rand(rng, B, Hq, Sq, D))


def _variants():
    """(name, mask, kind, causal, q_offset, window) over a 5x7 score matrix."""
    rng = np.random.default_rng(42)
    bias = rng.standard_normal((1, 5, 7)) * 0.7
    bias_masked = bias.copy()
    bias_masked[0, 0, 3] = -np.inf
    bias_masked[0, 2, [1, 5]] = -1e9           # the floor itself counts as masked
    boolm = (rng.random((1, 5, 7)) < 0.6).astype(np.uint8)
    boolm[0, :, 0] = 1                          # keep every row alive
    return [
        ("plain", None, "none", False, 0, 0),
        ("causal_offset", None, "none", True, 2, 0),
        ("additive_bias", bias_masked, "add", False, 0, 0),
        ("bool", boolm, "bool", False, 0, 0),
        ("causal_and_bias", bias, "add", True, 3, 0),
        ("window_sym", None, "none", False, 1, 2),
        ("window_causal_bias", bias, "add", True, 2, 1),
    ]


VARIANTS = _variants()


@pytest.mark.parametrize("name,mask,kind,causal,off,win", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_softmax_rows_sum_to_one(name, mask, kind, causal, off, win):
    q, k, v, _ = _tiny(1)
    p = ref.probabilities(q, k, 0.5, mask, kind, causal, off, win)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    vis = ref.visibility(5, 7, None if mask is None else mask[0], kind, causal, off, win)
    assert np.all(p[..., ~vis] == 0.0)


@pytest.mark.parametrize("name,mask,kind,causal,off,win", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_gradients_match_central_differences(name, mask, kind, causal, off, win):
    """Central differences of L = sum(G * O) with a seeded non-zero G.

    The skill page's trap list (item 7) warns that a zero loss gradient
    makes both arms compare 0 vs 0; here G is random and the analytic
    gradient is asserted non-zero before it is compared.
    """
    q, k, v, g = _tiny(2)
    scale = 0.6
    r = ref.backward(q, k, v, g, scale, mask, kind, causal, off, win)

    def loss(q_, k_, v_):
        o, _ = ref.forward(q_, k_, v_, scale, mask, kind, causal, off, win)
        return float((g * o).sum())

    h = 1e-6
    for name_, x, an in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        assert np.abs(an).max() > 1e-3, f"d{name_} is vacuously zero"
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}; args_p[name_] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name_] = xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                       loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        np.testing.assert_allclose(an, fd, rtol=1e-6, atol=1e-6 * np.abs(an).max())


def _sdpa_fp64(q, k, v, g, scale, mask, kind, causal, off, win=0):
    """PyTorch's scaled_dot_product_attention (float64, CPU) with autograd."""
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    ke = tk.repeat_interleave(G, dim=1)
    ve = tv.repeat_interleave(G, dim=1)
    attn = torch.zeros(mask.shape[0] if mask is not None else 1, 1, Sq, Sk, dtype=torch.float64)
    if mask is not None:
        m = torch.tensor(np.asarray(mask))
        if kind == "bool":
            attn = attn.masked_fill(~m.bool()[:, None], -math.inf)
        else:
            attn = attn + torch.where(m <= -1e9, torch.tensor(-math.inf, dtype=torch.float64),
                                      m.double())[:, None]
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Sk)[None, :]
    if causal:
        attn = attn.masked_fill(~(j <= off + i), -math.inf)
    if win > 0:
        attn = attn.masked_fill((off + i - j).abs() > win, -math.inf)
    o = torch.nn.functional.scaled_dot_product_attention(tq, ke, ve, attn_mask=attn, scale=scale)
    o.backward(torch.tensor(g))
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("name,mask,kind,causal,off,win", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_matches_torch_sdpa_float64(name, mask, kind, causal, off, win):
    q, k, v, g = _tiny(3, B=1, Hq=4, Hkv=2, Sq=5, Sk=7, D=8)
    r = ref.backward(q, k, v, g, 0.35, mask, kind, causal, off, win)
    o, dq, dk, dv = _sdpa_fp64(q, k, v, g, 0.35, mask, kind, causal, off, win)
    for a, b in ((r["o"], o), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_matches_torch_sdpa_larger_gqa_batch():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 2, 33, 47, 16
    q, k, v, g = (_rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D),
                  _rand(rng, B, Hq, Sq, D))
    mask = rng.standard_normal((B, Sq, Sk)) * 0.3
    mask[rng.random((B, Sq, Sk)) < 0.3] = -np.inf
    mask[:, :, 0] = 0.0
    r = ref.backward(q, k, v, g, 0.25, mask, "add", True, Sk - Sq)
    o, dq, dk, dv = _sdpa_fp64(q, k, v, g, 0.25, mask, "add", True, Sk - Sq)
    for a, b in ((r["o"], o), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_fully_masked_query_row_is_zero():
    """Skill page trap 9: a fully-masked query row has O = 0 and LSE = 0."""
    q, k, v, g = _tiny(4)
    mask = np.zeros((1, 5, 7))
    mask[0, 3, :] = -np.inf
    r = ref.backward(q, k, v, g, 0.5, mask, "add")
    assert np.all(r["o"][:, :, 3] == 0.0)
    assert np.all(r["lse"][:, :, 3] == 0.0)
    assert np.all(r["dq"][:, :, 3] == 0.0)
    # the dead row contributes nothing to dK/dV, whatever its dO holds
    g2 = g.copy()
    g2[:, :, 3] = 1e3
    r2 = ref.backward(q, k, v, g2, 0.5, mask, "add")
    assert np.array_equal(r["dk"], r2["dk"]) and np.array_equal(r["dv"], r2["dv"])


def test_fully_masked_key_column_has_zero_gradient():
    """Skill page trap 8: a cross mask hides whole key columns; their dK/dV are exactly 0."""
    q, k, v, g = _tiny(5)
    mask = np.zeros((1, 5, 7))
    mask[0, :, 4:] = -np.inf
    r = ref.backward(q, k, v, g, 0.5, mask, "add")
    assert np.all(r["dk"][:, :, 4:] == 0.0) and np.all(r["dv"][:, :, 4:] == 0.0)
    assert np.abs(r["dk"][:, :, :4]).max() > 1e-3


def test_gqa_equals_expanded_heads():
    """Native GQA equals explicitly expanded key/value heads with dK/dV summed per group."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 2, 9, 11, 8
    G = Hq // Hkv
    q, k, v, g = (_rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D),
                  _rand(rng, B, Hq, Sq, D))
    r = ref.backward(q, k, v, g, 0.3, causal=True, q_offset=2)
    ke, ve = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    e = ref.backward(q, ke, ve, g, 0.3, causal=True, q_offset=2)
    np.testing.assert_allclose(r["o"], e["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["lse"], e["lse"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["dq"], e["dq"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["dk"], e["dk"].reshape(B, Hkv, G, Sk, D).sum(2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["dv"], e["dv"].reshape(B, Hkv, G, Sk, D).sum(2), rtol=0, atol=1e-13)


def test_zero_query_closed_form():
    """Q = 0: P is uniform over the visible keys, so O is their mean and LSE = ln(#visible) + c."""
    rng = np.random.default_rng(7)
    Sq, Sk, D = 6, 9, 5
    q = np.zeros((1, 2, Sq, D))
    k, v = _rand(rng, 1, 1, Sk, D), _rand(rng, 1, 1, Sk, D)
    c = -0.75
    mask = np.full((1, Sq, Sk), c)
    mask[0, 1, [2, 3, 7]] = -np.inf
    o, lse = ref.forward(q, k, v, 0.9, mask, "add", causal=True, q_offset=3)
    for i in range(Sq):
        vis = [j for j in range(Sk) if j <= 3 + i and not (i == 1 and j in (2, 3, 7))]
        np.testing.assert_allclose(o[0, :, i], np.broadcast_to(v[0, 0, vis].mean(0), (2, D)), atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], math.log(len(vis)) + c, atol=1e-14)


def test_single_key_closed_form():
    """One visible key: O = v_0, LSE = s_00, and no gradient reaches Q or K."""
    q, k, v, g = _tiny(8, Sk=1)
    r = ref.backward(q, k, v, g, 0.5)
    np.testing.assert_allclose(r["o"], np.broadcast_to(v, r["o"].shape), atol=1e-15)
    np.testing.assert_allclose(r["lse"][0, :, :], 0.5 * (q[0] @ k[0, 0, 0]), atol=1e-14)
    assert np.abs(r["dq"]).max() < 1e-14 and np.abs(r["dk"]).max() < 1e-14
    np.testing.assert_allclose(r["dv"][0, 0, 0], g[0].sum(axis=(0, 1)), atol=1e-13)


@pytest.mark.parametrize("name,mask,kind,causal,off,win", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_dk_sums_to_zero_and_d_is_p_dot_dp(name, mask, kind, causal, off, win):
    """sum_j dS_ij = 0 (hence sum_j dK_j = 0), and D_i = sum_j P_ij dP_ij."""
    q, k, v, g = _tiny(9)
    r = ref.backward(q, k, v, g, 0.5, mask, kind, causal, off, win)
    np.testing.assert_allclose(r["dk"].sum(axis=2), 0.0, atol=1e-13)
    p = ref.probabilities(q, k, 0.5, mask, kind, causal, off, win)
    dp = np.einsum("bhid,bjd->bhij", g, v[:, 0])
    np.testing.assert_allclose((p * dp).sum(-1), r["d"], atol=1e-13)


def test_mask_row_shift_invariance():
    """Adding c to a row's additive mask leaves O unchanged and shifts LSE by c."""
    q, k, v, _ = _tiny(10)
    rng = np.random.default_rng(11)
    mask = rng.standard_normal((1, 5, 7))
    mask[0, 2, 4] = -np.inf
    shift = np.array([0.0, 1.5, -2.0, 0.25, 3.0])[None, :, None]
    o1, l1 = ref.forward(q, k, v, 0.5, mask, "add")
    o2, l2 = ref.forward(q, k, v, 0.5, mask + shift, "add")
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, np.broadcast_to(shift[..., 0], l1.shape), atol=1e-13)


def test_lse_gradient_is_attention_over_keys():
    """dLSE_i/dq_i = scale * sum_j P_ij k_j, which is the op's own O with V := K."""
    q, k, _, _ = _tiny(12)
    scale = 0.7
    _, lse = ref.forward(q, k, k, scale, causal=True, q_offset=2)
    o_kk, _ = ref.forward(q, k, k, scale, causal=True, q_offset=2)
    h = 1e-6
    for idx in np.ndindex(q.shape):
        qp = q.copy(); qp[idx] += h
        qm = q.copy(); qm[idx] -= h
        b, hh, i, d = idx
        fd = (ref.forward(qp, k, k, scale, causal=True, q_offset=2)[1][b, hh, i] -
              ref.forward(qm, k, k, scale, causal=True, q_offset=2)[1][b, hh, i]) / (2 * h)
        assert abs(fd - scale * o_kk[b, hh, i, d]) < 1e-7


def test_dirty_pad_leaves_outputs_bitwise_unchanged():
    """HOT-Step TRAINING.md, DiT micro-batching: pad must not reach any output.

    Garbage written into masked key/value columns changes nothing, bit for bit.
    """
    q, k, v, g = _tiny(13)
    mask = np.zeros((1, 5, 7))
    mask[0, :, 5:] = -np.inf
    r1 = ref.backward(q, k, v, g, 0.5, mask, "add")
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 5:] = 1234.5
    v2[:, :, 5:] = -987.25
    r2 = ref.backward(q, k2, v2, g, 0.5, mask, "add")
    for key in ("o", "lse", "dq"):
        assert np.array_equal(r1[key], r2[key]), key
    assert np.array_equal(r1["dk"][:, :, :5], r2["dk"][:, :, :5])
    assert np.array_equal(r1["dv"][:, :, :5], r2["dv"][:, :, :5])


def test_accumulate_adds_to_prefill():
    q, k, v, g = _tiny(14)
    rng = np.random.default_rng(15)
    acc_k, acc_v = rng.standard_normal(k.shape) * 0.01, rng.standard_normal(v.shape) * 0.01
    r = ref.backward(q, k, v, g, 0.5, causal=True, q_offset=2)
    a = ref.backward_accumulate(q, k, v, g, acc_k, acc_v, 0.5, causal=True, q_offset=2)
    np.testing.assert_allclose(a["dk"] - acc_k, r["dk"], atol=1e-15)
    np.testing.assert_allclose(a["dv"] - acc_v, r["dv"], atol=1e-15)


# ---- the seeded workload recipes ------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(16)
    x = (rng.standard_normal(100000) * rng.choice([1e-3, 1.0, 1e3], 100000)).astype(np.float32)
    ours = wl.round_to_bf16(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ours, theirs)


def test_workload_visible_pair_counts():
    """Mask-aware FLOP model units: closed-form counts of visible (head, query, key) triples."""
    assert wl.visible_pairs(wl.TINY_F32) == 2 * 64 * 64
    L = wl.pad_length(wl.DIT_SELF)
    assert L == 819
    assert wl.visible_pairs(wl.DIT_SELF) == 16 * (L * L + (1024 - L) * 1024)
    assert wl.visible_pairs(wl.CAUSAL_LM) == 32 * 4096 * 4097 // 2
    w = wl.LONG_WINDOW
    assert wl.visible_pairs(w) == 16 * sum(w.q_offset + i + 1 for i in range(w.Sq))
    lens = wl.cross_lengths(wl.DIT_CROSS)
    assert all(64 <= L_ <= 256 for L_ in lens)
    assert wl.visible_pairs(wl.DIT_CROSS) == 16 * 2046 * int(lens.sum())


def test_mask_recipes_have_the_stated_structure():
    m, kind = wl.make_mask(wl.DIT_SELF)
    assert kind == "add"
    assert not np.any(np.all(m[0] == -np.inf, axis=0)), "self mask must not hide a whole key column"
    assert not np.any(np.all(m[0] == -np.inf, axis=1)), "self mask has no fully-masked query row"
    m, _ = wl.make_mask(wl.DIT_CROSS)
    lens = wl.cross_lengths(wl.DIT_CROSS)
    for b in range(2):
        assert np.all(m[b, :, lens[b]:] == -np.inf)
        assert int(np.all(m[b] == -np.inf, axis=1).sum()) == 2
    m, _ = wl.make_mask(wl.TINY_F32)
    assert np.all(m[0, 64] == -np.inf) and np.all(m[0, :64] == 0)


def test_window_equals_the_same_band_as_an_explicit_mask():
    """The sliding window gives exactly what an additive mask hiding the same pairs gives."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 9, 13, 8
    q, k, v, g = (_rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D),
                  _rand(rng, B, Hq, Sq, D))
    for causal, off, win in ((False, 2, 3), (True, 4, 2), (False, 0, 1)):
        i = np.arange(Sq)[:, None]
        j = np.arange(Sk)[None, :]
        band = np.abs(off + i - j) <= win
        mask = np.where(band, 0.0, -np.inf)[None]
        a = ref.backward(q, k, v, g, 0.4, causal=causal, q_offset=off, window=win)
        b = ref.backward(q, k, v, g, 0.4, mask, "add", causal=causal, q_offset=off)
        for key in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_array_equal(a[key], b[key])


def test_window_wider_than_the_sequence_changes_nothing():
    q, k, v, g = _tiny(18)
    a = ref.backward(q, k, v, g, 0.5, causal=True, q_offset=2)
    b = ref.backward(q, k, v, g, 0.5, causal=True, q_offset=2, window=100)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[key], b[key])


def test_window_zero_width_band_is_the_diagonal():
    """Window 1 around the diagonal with Sq = Sk: closed form for Q = 0 (mean of <= 3 values)."""
    rng = np.random.default_rng(19)
    S, D = 6, 4
    q = np.zeros((1, 1, S, D))
    k, v = _rand(rng, 1, 1, S, D), _rand(rng, 1, 1, S, D)
    o, lse = ref.forward(q, k, v, 0.5, window=1)
    for i in range(S):
        vis = [j for j in range(S) if abs(i - j) <= 1]
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, vis].mean(0), atol=1e-14)
        np.testing.assert_allclose(lse[0, 0, i], math.log(len(vis)), atol=1e-14)


# ---- SET_ROWS backward (the chunk's K/V gradient read back out of the window accumulator) ----

from oracle import set_rows as rows_ref  # noqa: E402


def test_set_rows_backward_is_the_autograd_of_a_row_write():
    """torch autograd of index_copy (the row write of SET_ROWS) gives the source exactly the oracle's rows."""
    rng = np.random.default_rng(31)
    B, H, S, D = 2, 3, 11, 8
    # the second index set repeats a row: each source row still receives the gradient at its row
    for idx in (np.array([4, 9, 0, 7, 10]), np.array([4, 9, 4, 2])):
        cache = torch.tensor(rng.standard_normal((B, H, S, D)))
        src = torch.tensor(rng.standard_normal((B, H, len(idx), D)), requires_grad=True)
        out = cache.index_copy(2, torch.tensor(idx), src)
        g = torch.tensor(rng.standard_normal((B, H, S, D)))
        (out * g).sum().backward()
        np.testing.assert_array_equal(rows_ref.set_rows_backward(g.numpy(), idx), src.grad.numpy())


def test_set_rows_backward_through_attention_on_the_cache():
    """End to end: K/V written into a cache, attention over the cache; dL/d(written K/V) equals the
    attention backward's dK/dV read back at the written rows (fp64 autograd vs oracle)."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 5, 12, 8
    off = Sk - Sq
    q = rng.standard_normal((B, Hq, Sq, D))
    cache_k = rng.standard_normal((B, Hkv, Sk, D))
    cache_v = rng.standard_normal((B, Hkv, Sk, D))
    k_src = rng.standard_normal((B, Hkv, Sq, D))
    v_src = rng.standard_normal((B, Hkv, Sq, D))
    g = rng.standard_normal((B, Hq, Sq, D))
    idx = np.arange(off, Sk)
    tk = torch.tensor(k_src, requires_grad=True)
    tv = torch.tensor(v_src, requires_grad=True)
    kc = torch.tensor(cache_k).index_copy(2, torch.tensor(idx), tk)
    vc = torch.tensor(cache_v).index_copy(2, torch.tensor(idx), tv)
    G = Hq // Hkv
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Sk)[None, :]
    bias = torch.zeros(Sq, Sk, dtype=torch.float64).masked_fill(j > off + i, -math.inf)
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), kc.repeat_interleave(G, 1), vc.repeat_interleave(G, 1), attn_mask=bias, scale=0.3)
    (o * torch.tensor(g)).sum().backward()
    kk = cache_k.copy(); kk[:, :, idx] = k_src
    vv = cache_v.copy(); vv[:, :, idx] = v_src
    r = ref.backward(q, kk, vv, g, 0.3, causal=True, q_offset=off)
    np.testing.assert_allclose(rows_ref.set_rows_backward(r["dk"], idx), tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(rows_ref.set_rows_backward(r["dv"], idx), tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_bf16_rounding_matches_torch_including_ties():
    rng = np.random.default_rng(33)
    x = (rng.standard_normal(4096) * 10.0 ** rng.integers(-6, 6, 4096)).astype(np.float32)
    # exact ties: bf16 patterns with the dropped half equal to 0x8000, odd and even kept parts
    base = rng.integers(0, 1 << 15, 512).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    ties_odd = ((base | 0x10000) | 0x8000).view(np.float32)
    for v in (x, ties, ties_odd, np.array([0.0, -0.0, 1.0, -3.5, 1e-40], np.float32), x.reshape(4, 8, 128)):
        want = torch.tensor(v).to(torch.bfloat16).float().numpy()
        np.testing.assert_array_equal(rows_ref.to_bf16_bits(v), want)


# ---- q8_0 K/V cache ----------------------------------------------------------------------------

def test_q8_0_dequantization_uses_one_scale_per_32_features():
    """Block f // 32 of each row scales features [32 b, 32 b + 32): distinct scales per block and
    unit values give each scale repeated 32 times; a row-major slip or a transposed block fails."""
    q = np.ones((2, 3, 128), np.int8)
    q[1, 2, 70] = -5
    d = (np.arange(2 * 3 * 4, dtype=np.float64).reshape(2, 3, 4) + 1.0).astype(np.float16) / 8
    got = ref.dequantize_q8_0(q, d)
    want = np.repeat(d.astype(np.float64), 32, axis=-1)
    want[1, 2, 70] *= -5
    np.testing.assert_array_equal(got, want)


def test_q8_0_encoding_round_trip_is_within_half_a_step():
    """The cache encoding of the seeded inputs: |x - d q| <= d / 2 per element (plus the float16
    rounding of d, which can push max|x| / d a hair past 127)."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal((2, 4, 50, 128)).astype(np.float32)
    q, d = wl.quantize_q8_0(x)
    back = ref.dequantize_q8_0(q, d)
    step = np.repeat(d.astype(np.float64), 32, axis=-1)
    amax = np.repeat(np.abs(x.reshape(2, 4, 50, 4, 32)).max(-1), 32, axis=-1)
    assert np.all(np.abs(back - x) <= step / 2 + amax * 2.0 ** -10)


def test_attention_on_a_q8_0_cache_is_attention_on_its_values():
    """The op over the cache equals the op over the dequantized K/V (so the gradients are those of
    the cache's values), checked against PyTorch float64 SDPA with autograd."""
    rng = np.random.default_rng(42)
    q = rng.standard_normal((1, 2, 5, 32))
    kq, kd = wl.quantize_q8_0(rng.standard_normal((1, 1, 9, 32)).astype(np.float32))
    vq, vd = wl.quantize_q8_0(rng.standard_normal((1, 1, 9, 32)).astype(np.float32))
    g = rng.standard_normal((1, 2, 5, 32))
    k, v = ref.dequantize_q8_0(kq, kd), ref.dequantize_q8_0(vq, vd)
    r = ref.backward(q, k, v, g, 0.3, causal=True, q_offset=4)
    o, dq, dk, dv = _sdpa_fp64(q, k, v, g, 0.3, None, "none", True, 4)
    for a, b in ((r["o"], o), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)
