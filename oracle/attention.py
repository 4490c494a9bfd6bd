"""fp64 CPU oracle for the fused flash-attention training op.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the product path (the
C-ABI library and its Python binding) never does, and shares no code with it.

What it computes, written out plainly with explicit score and probability
matrices (no tiling, no online softmax, no fusion):

  forward (flash-attn-training skill, trap list item 9; llama.cpp PR #57,
  commit 86c140d "tiled flash-attention backward": the op returns O and the
  per-row LSE):
      s_ij    = scale * <q_i, k_j> + bias_ij
      vis_ij  = (mask does not hide (i, j)) and (not causal or j <= q_offset + i)
      P_ij    = exp(s_ij - M_i) / l_i on visible pairs, exactly 0 elsewhere,
                with M_i = max_vis s_ij and l_i = sum_vis exp(s_ij - M_i)
      LSE_i   = M_i + ln l_i
      O_i     = sum_j P_ij v_j
      a query row with no visible key has O_i = 0 and LSE_i = 0 (trap 9).

  backward (chain rule of L = sum(dO * O); PR #57 commit 86c140d lists its
  ingredients: LSE, D, per-tile gradients, GQA group-sum):
      D_i     = <dO_i, O_i>
      dP_ij   = <dO_i, v_j>
      dS_ij   = P_ij (dP_ij - D_i)
      dQ_i    = scale * sum_j dS_ij k_j
      dK_j    = scale * sum_{h in group} sum_i dS_ij q_i      (GQA group-sum)
      dV_j    = sum_{h in group} sum_i P_ij dO_i

Readings where the pages are silent (each listed in the design notes):
  * an additive mask value <= -1e9 (the "mask floor" of PR #57) or -inf means
    masked: P is exactly 0 there, not exp(-1e9). Larger values are a bias;
  * a boolean mask uses 1 = attend, 0 = masked;
  * the mask is added after scaling (s = scale * qk + mask);
  * LSE is a natural logarithm;
  * GQA maps query head h to key/value head floor(h / G), G = Hq / Hkv
    (consecutive query heads share one key/value head);
  * causal: key j is visible to query i iff j <= q_offset + i;
  * sliding window w > 0 (the DiT self-attention mask of HOT-Step TRAINING.md, "DiT
    micro-batching": a sliding window plus padded key columns): key j is visible to query i
    only if |q_offset + i - j| <= w; with causal only the left side applies
    (q_offset + i - w <= j <= q_offset + i).

Arrays are numpy, [B, H, S, D] row-major; masks are [Bm, Sq, Sk] with Bm in
{1, B}. All arithmetic is float64 on the exact input values.
"""
from __future__ import annotations

import numpy as np

MASK_FLOOR = -1e9


def visibility(Sq: int, Sk: int, mask_b, mask_kind: str, causal: bool, q_offset: int, window: int = 0) -> np.ndarray:
    """Boolean [Sq, Sk]: True where query i may attend to key j."""
    vis = np.ones((Sq, Sk), dtype=bool)
    if mask_b is not None and mask_kind != "none":
        if mask_kind == "bool":
            vis &= np.asarray(mask_b) != 0
        elif mask_kind == "add":
            vis &= np.asarray(mask_b, dtype=np.float64) > MASK_FLOOR
        else:
            raise ValueError(mask_kind)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    if causal:
        vis &= j <= q_offset + i
    if window > 0:
        vis &= np.abs(q_offset + i - j) <= window
    return vis


def _bias(mask_b, mask_kind: str, vis: np.ndarray) -> np.ndarray:
    if mask_b is None or mask_kind != "add":
        return np.zeros(vis.shape)
    return np.where(vis, np.asarray(mask_b, dtype=np.float64), 0.0)


def _mask_for_batch(mask, b):
    if mask is None:
        return None
    return mask[b if mask.shape[0] > 1 else 0]


def head_probabilities(q_h, k_h, scale, mask_b, mask_kind, causal, q_offset, window=0):
    """P [Sq, Sk], LSE [Sq] and the row-has-a-visible-key flag for one head."""
    Sq, Sk = q_h.shape[0], k_h.shape[0]
    vis = visibility(Sq, Sk, mask_b, mask_kind, causal, q_offset, window)
    s = scale * (q_h @ k_h.T) + _bias(mask_b, mask_kind, vis)
    s = np.where(vis, s, -np.inf)
    alive = vis.any(axis=1)
    row_max = np.where(alive, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(vis, np.exp(s - row_max[:, None]), 0.0)
    row_sum = e.sum(axis=1)
    safe_sum = np.where(alive, row_sum, 1.0)
    p = e / safe_sum[:, None]
    lse = np.where(alive, row_max + np.log(safe_sum), 0.0)
    return p, lse, alive


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def dequantize_q8_0(q, d) -> np.ndarray:
    """Values of a q8_0-style K/V cache (llama.cpp PR #57, commit 2394a4c: a q8_0 cache is read in
    place): feature f of a row is d[f // 32] * q[f], q int8 [..., D], d float16 [..., D / 32]."""
    q = np.asarray(q, dtype=np.float64)
    d = np.asarray(d, dtype=np.float16).astype(np.float64)
    return q * np.repeat(d, 32, axis=-1)


def forward(q, k, v, scale, mask=None, mask_kind="none", causal=False, q_offset=0, window=0):
    """Return O [B,Hq,Sq,D] and LSE [B,Hq,Sq], both float64."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        mb = _mask_for_batch(mask, b)
        for h in range(Hq):
            kv = h // G
            p, lse[b, h], _ = head_probabilities(q[b, h], k[b, kv], scale, mb, mask_kind, causal, q_offset, window)
            o[b, h] = p @ v[b, kv]
    return o, lse


def backward(q, k, v, do, scale, mask=None, mask_kind="none", causal=False, q_offset=0, window=0):
    """Return dict with o, lse, d (= rowsum(dO*O)), dq, dk, dv (float64).

    P is rebuilt from its definition, not from a stored LSE, so the backward
    depends on nothing the forward of the GPU path produced.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Sq))
    dsum = np.zeros((B, Hq, Sq))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        mb = _mask_for_batch(mask, b)
        for h in range(Hq):
            kv = h // G
            p, lse[b, h], _ = head_probabilities(q[b, h], k[b, kv], scale, mb, mask_kind, causal, q_offset, window)
            o[b, h] = p @ v[b, kv]
            dsum[b, h] = (do[b, h] * o[b, h]).sum(axis=1)
            dp = do[b, h] @ v[b, kv].T
            ds = p * (dp - dsum[b, h][:, None])
            dq[b, h] = scale * (ds @ k[b, kv])
            dk[b, kv] += scale * (ds.T @ q[b, h])
            dv[b, kv] += p.T @ do[b, h]
    return {"o": o, "lse": lse, "d": dsum, "dq": dq, "dk": dk, "dv": dv}


def probabilities(q, k, scale, mask=None, mask_kind="none", causal=False, q_offset=0, window=0):
    """P [B,Hq,Sq,Sk] (float64): exposed so tests can check its invariants."""
    q, k = _as64(q), _as64(k)
    B, Hq, Sq, _ = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, Sq, Sk))
    for b in range(B):
        mb = _mask_for_batch(mask, b)
        for h in range(Hq):
            out[b, h], _, _ = head_probabilities(q[b, h], k[b, h // G], scale, mb, mask_kind, causal, q_offset,
                                                 window)
    return out


def backward_accumulate(q, k, v, do, dk_acc, dv_acc, scale, mask=None, mask_kind="none", causal=False,
                        q_offset=0, window=0):
    """Accumulating backward: dK/dV are added to caller-owned buffers.

    llama.cpp PR #57, commit 86c140d (ggml_opt_accumulate_grad): the backward
    adds a node's gradient into an existing tensor. Sums are taken in float64.
    """
    r = backward(q, k, v, do, scale, mask, mask_kind, causal, q_offset, window)
    r["dk"] = _as64(dk_acc) + r["dk"]
    r["dv"] = _as64(dv_acc) + r["dv"]
    return r
