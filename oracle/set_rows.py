"""fp64 / exact CPU oracle of the SET_ROWS backward.

TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
does, and shares no code with it.

llama.cpp PR #57, commit 2394a4c ("the training graph is the serving graph"):
a chunk writes its K/V into the cache with SET_ROWS and attention reads the
cache in place; SET_ROWS gets a backward in which the written source's
gradient is the result's gradient at the written rows, and the destination (a
cache) carries none. With the window gradient accumulated in `acc`, the
chunk's own K/V gradient is read back from the written rows:

    out[b, h, r, :] = acc[b, h, idx[r], :]

A repeated index gives each of its source rows the same gradient row.
Converting to bf16 rounds to the nearest representable value, ties to even.
"""
from __future__ import annotations

import numpy as np


def to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns the float32 values it represents.

    Written from the definition: keep the top 16 bits of the float32 pattern, and round up when
    the dropped 16 bits exceed half an ulp, or equal it and the kept pattern is odd (a carry into
    the exponent is the correct overflow to the next binade or to infinity); NaN stays NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    keep = u >> 16
    dropped = u & 0xFFFF
    round_up = (dropped > 0x8000) | ((dropped == 0x8000) & ((keep & 1) == 1))
    out = ((keep + round_up.astype(np.uint64)) << 16).astype(np.uint32)
    out = np.where(np.isnan(x), np.uint32(0x7FC00000), out)   # a NaN stays a NaN
    return out.view(np.float32).reshape(x.shape)


def set_rows_backward(acc, idx, out_dtype: str = "f32") -> np.ndarray:
    """Gradient of the source rows of SET_ROWS: the accumulator's rows at idx (float64 or bf16 values)."""
    acc = np.asarray(acc)
    idx = np.asarray(idx, dtype=np.int64)
    out = acc[:, :, idx, :]
    if out_dtype == "bf16":
        return to_bf16_bits(out.astype(np.float32)).astype(np.float64)
    return out.astype(np.float64)
