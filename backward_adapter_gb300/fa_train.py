"""Thin Python binding of the C-ABI library libfa_train.so (include/fa_train.h).

Argument marshalling only: PyTorch supplies device memory and the current
CUDA stream, ctypes passes raw pointers and sizes, and every step of the op
runs in the library's CUDA kernels. There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_train.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE, FA_ERR_CUDA = range(5)
FA_F32, FA_BF16 = 0, 1
FA_MASK_NONE, FA_MASK_ADD_F32, FA_MASK_BOOL_U8 = 0, 1, 2
FA_KV_DTYPE, FA_KV_Q8_0, FA_KV_F16 = 0, 1, 2
FA_LAYOUT_BHSD, FA_LAYOUT_BSHD = 0, 1

EXPORTED = ("fa_train_fwd_workspace_size", "fa_train_bwd_workspace_size", "fa_train_fwd", "fa_train_bwd",
            "fa_train_bwd_accum", "fa_status_str", "fa_last_error", "fa_profile_set_events",
            "fa_profile_launch_count", "fa_device_status", "fa_train_bwd_noalloc", "fa_train_selftest_wait",
            "fa_set_rows_backward", "fa_train_bwd_accum_rows", "fa_train_fwd_q8", "fa_train_bwd_q8",
            "fa_train_bwd_accum_q8", "fa_train_bwd_plan", "fa_train_fwd_plan")
FA_KERNEL_FWD, FA_KERNEL_BWD_MAIN, FA_KERNEL_BWD_DSUM, FA_KERNEL_BWD_DQ_CONVERT, FA_KERNEL_MASK_CLASSIFY = range(5)


class FaParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("Sq", ctypes.c_int32), ("Sk", ctypes.c_int32), ("D", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("mask_kind", ctypes.c_int32), ("mask_batch", ctypes.c_int32), ("window", ctypes.c_int32),
                ("q_offset", ctypes.c_int64), ("deterministic", ctypes.c_int32), ("kv_format", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class FaKvQ8(ctypes.Structure):
    """fa_kv_q8: device pointers of a q8_0 K/V cache (int8 values, fp16 scales per 32 features)."""
    _fields_ = [("k_q", ctypes.c_void_p), ("k_d", ctypes.c_void_p), ("v_q", ctypes.c_void_p),
                ("v_d", ctypes.c_void_p)]


class FaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"fa_train: {_status_name(status)} ({status}): {detail}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfa_train.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with backward_adapter_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(FaParams)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.fa_train_fwd_workspace_size.argtypes = [P]
    lib.fa_train_fwd_workspace_size.restype = sz
    lib.fa_train_bwd_workspace_size.argtypes = [P]
    lib.fa_train_bwd_workspace_size.restype = sz
    lib.fa_train_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_train_fwd.restype = st
    lib.fa_train_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_train_bwd.restype = st
    lib.fa_train_bwd_accum.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_train_bwd_accum.restype = st
    lib.fa_status_str.argtypes = [st]
    lib.fa_status_str.restype = ctypes.c_char_p
    lib.fa_last_error.argtypes = []
    lib.fa_last_error.restype = ctypes.c_char_p
    lib.fa_profile_set_events.argtypes = [st, vp, vp]
    lib.fa_profile_set_events.restype = st
    lib.fa_profile_launch_count.argtypes = []
    lib.fa_profile_launch_count.restype = ctypes.c_uint64
    lib.fa_train_bwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.fa_train_bwd_noalloc.restype = st
    lib.fa_train_selftest_wait.argtypes = [ctypes.c_uint32, vp]
    lib.fa_train_selftest_wait.restype = st
    lib.fa_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.fa_device_status.restype = st
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.fa_set_rows_backward.argtypes = [vp, i32, i32, i32, i32, vp, i32, vp, i32, vp]
    lib.fa_set_rows_backward.restype = st
    lib.fa_train_bwd_accum_rows.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, vp, vp, vp, sz, vp]
    lib.fa_train_bwd_accum_rows.restype = st
    KV = ctypes.POINTER(FaKvQ8)
    lib.fa_train_fwd_q8.argtypes = [P, vp, KV, vp, vp, vp, vp, sz, vp]
    lib.fa_train_fwd_q8.restype = st
    lib.fa_train_bwd_q8.argtypes = [P, vp, KV, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_train_bwd_q8.restype = st
    lib.fa_train_bwd_accum_q8.argtypes = [P, vp, KV, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.fa_train_bwd_accum_q8.restype = st
    lib.fa_train_bwd_plan.argtypes = [P, ctypes.POINTER(i32), i32, ctypes.POINTER(i32)]
    lib.fa_train_bwd_plan.restype = st
    lib.fa_train_fwd_plan.argtypes = [P, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.fa_train_fwd_plan.restype = st
    _lib = lib
    return lib


def _status_name(s: int) -> str:
    try:
        return load_library().fa_status_str(s).decode()
    except Exception:  # library not loadable while formatting an error
        return str(s)


def _check(status: int) -> None:
    if status != FA_OK:
        raise FaError(status, load_library().fa_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _mask_view(mask: Optional[torch.Tensor]):
    if mask is None:
        return None, FA_MASK_NONE, 1
    if mask.dim() != 3:
        raise ValueError("mask must be [mask_batch, Sq, Sk]")
    if mask.dtype == torch.float32:
        return mask, FA_MASK_ADD_F32, mask.shape[0]
    if mask.dtype == torch.bool:
        return mask.view(torch.uint8), FA_MASK_BOOL_U8, mask.shape[0]
    if mask.dtype == torch.uint8:
        return mask, FA_MASK_BOOL_U8, mask.shape[0]
    raise TypeError(f"mask dtype {mask.dtype}: float32 (additive) or uint8/bool (1 = attend)")


def _kv_format(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> int:
    """K/V in q's dtype, or an fp16 cache under bf16 queries (rounded to bf16 by the library)."""
    if k.dtype != v.dtype:
        raise TypeError(f"k ({k.dtype}) and v ({v.dtype}) must have one dtype")
    if k.dtype == q.dtype:
        return FA_KV_DTYPE
    if k.dtype == torch.float16 and q.dtype == torch.bfloat16:
        return FA_KV_F16
    raise TypeError(f"k/v dtype {k.dtype} with q dtype {q.dtype}: same as q, or float16 under bfloat16 q")


def make_params(q: torch.Tensor, k: torch.Tensor, mask: Optional[torch.Tensor] = None, *,
                scale: Optional[float] = None, causal: bool = False,
                q_offset: Optional[int] = None, window: int = 0, deterministic: bool = False,
                kv_format: int = FA_KV_DTYPE, layout: str = "bhsd") -> FaParams:
    """Fill fa_params from tensor shapes. q: [B,Hq,Sq,D], k: [B,Hkv,Sk,D] (layout "bhsd"), or
    q: [B,Sq,Hq,D], k: [B,Sk,Hkv,D] (layout "bshd": PyTorch's activations, no transpose copy).

    q_offset (causal or windowed) defaults to Sk - Sq: the query rows are the last Sq
    key positions. window is the sliding-window half-width (0 = none). deterministic makes
    the backward's dQ bitwise reproducible.
    """
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError(f"q and k must be 4-D (got {q.dim()}-D and {k.dim()}-D)")
    if layout == "bhsd":
        B, Hq, Sq, D = q.shape
        Hkv, Sk = k.shape[1], k.shape[2]
    elif layout == "bshd":
        B, Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
    else:
        raise ValueError(f"layout {layout!r}: 'bhsd' or 'bshd'")
    _, kind, mb = _mask_view(mask)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if q_offset is None:
        q_offset = Sk - Sq if (causal or window > 0) else 0
    return FaParams(B, Hq, Hkv, Sq, Sk, D, _dtype_code(q), float(scale), int(bool(causal)), kind, mb,
                    int(window), int(q_offset), int(bool(deterministic)), int(kv_format),
                    FA_LAYOUT_BSHD if layout == "bshd" else FA_LAYOUT_BHSD, 0)


def fwd_workspace_size(p: FaParams) -> int:
    return int(load_library().fa_train_fwd_workspace_size(ctypes.byref(p)))


def bwd_workspace_size(p: FaParams) -> int:
    return int(load_library().fa_train_bwd_workspace_size(ctypes.byref(p)))


def bwd_plan(p: FaParams) -> "list[tuple[int, int, int, int, int, int]]":
    """The backward's CTAs in launch order (host only): (key tile, batch * Hkv + kv head, part,
    parts, first query row, end query row) each; see fa_train_bwd_plan."""
    lib = load_library()
    n = ctypes.c_int32(0)
    _check(lib.fa_train_bwd_plan(ctypes.byref(p), None, 0, ctypes.byref(n)))
    rec = (ctypes.c_int32 * (6 * max(n.value, 1)))()
    _check(lib.fa_train_bwd_plan(ctypes.byref(p), rec, n.value, ctypes.byref(n)))
    return [tuple(rec[6 * i:6 * i + 6]) for i in range(n.value)]


def fwd_plan(p: FaParams) -> "tuple[int, int, bool]":
    """The forward's launch (host only): (CTAs, key splits per unit, persistent); see
    fa_train_fwd_plan."""
    lib = load_library()
    ctas, splits, pers = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.fa_train_fwd_plan(ctypes.byref(p), ctypes.byref(ctas), ctypes.byref(splits), ctypes.byref(pers)))
    return ctas.value, splits.value, bool(pers.value)


def _on_device(t: torch.Tensor):
    """The library launches on, and keeps its per-device state for, the current CUDA device:
    make it the device the call's tensors live on."""
    return torch.cuda.device(t.device)


def _stream(device: torch.device, stream) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return ws
    if ws is not None and ws.numel() * ws.element_size() >= nbytes:
        return ws
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("every tensor must be a contiguous CUDA tensor")


def _q_shape(p: FaParams, layout: str):
    return (p.B, p.Hq, p.Sq, p.D) if layout == "bhsd" else (p.B, p.Sq, p.Hq, p.D)


def _kv_shape(p: FaParams, layout: str, rows: Optional[int] = None):
    S = p.Sk if rows is None else rows
    return (p.B, p.Hkv, S, p.D) if layout == "bhsd" else (p.B, S, p.Hkv, p.D)


def _check_tensors(q: torch.Tensor, **expect) -> None:
    """Every tensor the library will read or write has the shape (and dtype) the parameters imply
    and lives on q's device: the C ABI receives bare pointers, so a wrong shape would reach the
    kernels as out-of-bounds accesses. expect maps a name to (tensor or None, shape, dtype or None)."""
    for name, (t, shape, dtype) in expect.items():
        if t is None:
            continue
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")


def _common_expect(p: FaParams, layout: str, q, k=None, v=None, mask=None, o=None, lse=None, do=None, dq=None):
    qs, ks = _q_shape(p, layout), _kv_shape(p, layout)
    e = {"k": (k, ks, None), "v": (v, ks, None), "o": (o, qs, q.dtype), "lse": (lse, (p.B, p.Hq, p.Sq), torch.float32),
         "do": (do, qs, q.dtype), "dq": (dq, qs, q.dtype)}
    if mask is not None:
        e["mask"] = (mask, (mask.shape[0], p.Sq, p.Sk), None)
    return e


def fwd(q, k, v, mask=None, *, scale=None, causal=False, q_offset=None, window=0, deterministic=False, layout="bhsd",
        out=None, lse=None, workspace=None, stream=None):
    """Forward: returns (O [B,Hq,Sq,D] in q's dtype, LSE [B,Hq,Sq] fp32). k and v are in q's dtype,
    or float16 (an fp16 cache) under bfloat16 q."""
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    p = make_params(q, k, mask, scale=scale, causal=causal, q_offset=q_offset, window=window,
                    deterministic=deterministic, kv_format=_kv_format(q, k, v), layout=layout)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device=q.device)
    _check_tensors(q, **_common_expect(p, layout, q, k, v, mask, o=out, lse=lse))
    _need_cuda(q, k, v, mview, out, lse)
    ws_bytes = fwd_workspace_size(p)
    ws = _workspace(ws_bytes, q.device, workspace)
    with _on_device(q):
        _check(lib.fa_train_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(mview), _ptr(out), _ptr(lse),
                                _ptr(ws), ws_bytes, _stream(q.device, stream)))
    return out, lse


def bwd(q, k, v, o, lse, do, mask=None, *, scale=None, causal=False, q_offset=None, window=0, deterministic=False,
        layout="bhsd", dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward: returns (dQ, dK, dV) in q's dtype (overwriting any given buffers); k and v as in fwd."""
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    p = make_params(q, k, mask, scale=scale, causal=causal, q_offset=q_offset, window=window,
                    deterministic=deterministic, kv_format=_kv_format(q, k, v), layout=layout)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k, dtype=q.dtype) if dk is None else dk   # q's dtype for an fp16 cache too
    dv = torch.empty_like(v, dtype=q.dtype) if dv is None else dv
    ks = _kv_shape(p, layout)
    _check_tensors(q, **_common_expect(p, layout, q, k, v, mask, o, lse, do, dq), dk=(dk, ks, q.dtype),
                   dv=(dv, ks, q.dtype))
    _need_cuda(q, k, v, o, lse, do, mview, dq, dk, dv)
    ws_bytes = bwd_workspace_size(p)
    ws = _workspace(ws_bytes, q.device, workspace)
    with _on_device(q):
        _check(lib.fa_train_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(mview), _ptr(o), _ptr(lse),
                                _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws_bytes,
                                _stream(q.device, stream)))
    return dq, dk, dv


def bwd_accum(q, k, v, o, lse, do, dk_acc, dv_acc, mask=None, *, scale=None, causal=False, q_offset=None, window=0,
              deterministic=False, layout="bhsd", dq=None, workspace=None, stream=None):
    """Accumulating backward: dK/dV are added into fp32 dk_acc/dv_acc in place; returns dQ."""
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    if dk_acc.dtype != torch.float32 or dv_acc.dtype != torch.float32:
        raise TypeError("dk_acc and dv_acc must be float32")
    p = make_params(q, k, mask, scale=scale, causal=causal, q_offset=q_offset, window=window,
                    deterministic=deterministic, kv_format=_kv_format(q, k, v), layout=layout)
    dq = torch.empty_like(q) if dq is None else dq
    ks = _kv_shape(p, layout)
    _check_tensors(q, **_common_expect(p, layout, q, k, v, mask, o, lse, do, dq),
                   dk_acc=(dk_acc, ks, torch.float32), dv_acc=(dv_acc, ks, torch.float32))
    _need_cuda(q, k, v, o, lse, do, dk_acc, dv_acc, mview, dq)
    ws_bytes = bwd_workspace_size(p)
    ws = _workspace(ws_bytes, q.device, workspace)
    with _on_device(q):
        _check(lib.fa_train_bwd_accum(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(mview), _ptr(o), _ptr(lse),
                                      _ptr(do), _ptr(dq), _ptr(dk_acc), _ptr(dv_acc), _ptr(ws), ws_bytes,
                                      _stream(q.device, stream)))
    return dq


def bwd_accum_rows(q, k, v, o, lse, do, dk_acc, dv_acc, rows_begin: int, n_rows: int, mask=None, *, scale=None,
                   causal=False, q_offset=None, window=0, deterministic=False, layout="bhsd", dq=None, dk_rows=None,
                   dv_rows=None, workspace=None, stream=None):
    """Accumulating backward fused with the SET_ROWS backward of keys [rows_begin, rows_begin + n_rows).

    Adds dK/dV into dk_acc/dv_acc and also returns those keys' finished sums, read back in q's
    dtype: (dQ, dK_rows [B, Hkv, n_rows, D], dV_rows [B, Hkv, n_rows, D]), or [B, n_rows, Hkv, D]
    with layout "bshd".
    """
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    if dk_acc.dtype != torch.float32 or dv_acc.dtype != torch.float32:
        raise TypeError("dk_acc and dv_acc must be float32")
    p = make_params(q, k, mask, scale=scale, causal=causal, q_offset=q_offset, window=window,
                    deterministic=deterministic, kv_format=_kv_format(q, k, v), layout=layout)
    dq = torch.empty_like(q) if dq is None else dq
    shape = _kv_shape(p, layout, rows=int(n_rows))
    dk_rows = torch.empty(shape, dtype=q.dtype, device=q.device) if dk_rows is None else dk_rows
    dv_rows = torch.empty(shape, dtype=q.dtype, device=q.device) if dv_rows is None else dv_rows
    ks = _kv_shape(p, layout)
    _check_tensors(q, **_common_expect(p, layout, q, k, v, mask, o, lse, do, dq),
                   dk_acc=(dk_acc, ks, torch.float32), dv_acc=(dv_acc, ks, torch.float32),
                   dk_rows=(dk_rows, shape, q.dtype), dv_rows=(dv_rows, shape, q.dtype))
    _need_cuda(q, k, v, o, lse, do, dk_acc, dv_acc, mview, dq, dk_rows, dv_rows)
    ws_bytes = bwd_workspace_size(p)
    ws = _workspace(ws_bytes, q.device, workspace)
    with _on_device(q):
        _check(lib.fa_train_bwd_accum_rows(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(mview), _ptr(o), _ptr(lse),
                                           _ptr(do), _ptr(dq), _ptr(dk_acc), _ptr(dv_acc), int(rows_begin), int(n_rows),
                                           _ptr(dk_rows), _ptr(dv_rows), _ptr(ws), ws_bytes, _stream(q.device, stream)))
    return dq, dk_rows, dv_rows


def _kv_q8(k_q, k_d, v_q, v_d) -> FaKvQ8:
    if k_q.dtype != torch.int8 or v_q.dtype != torch.int8:
        raise TypeError("k_q and v_q must be int8 [B, Hkv, Sk, D]")
    if k_d.dtype != torch.float16 or v_d.dtype != torch.float16:
        raise TypeError("k_d and v_d must be float16 [B, Hkv, Sk, D / 32]")
    return FaKvQ8(k_q.data_ptr(), k_d.data_ptr(), v_q.data_ptr(), v_d.data_ptr())


def _cache_shape_view(k_q, layout):
    """The cache planes are [B, Hkv, Sk, ...] whatever the layout of Q: a view for the shapes only."""
    return k_q if layout == "bhsd" else k_q.transpose(1, 2)


def _q8_expect(p: FaParams, k_q, k_d, v_q, v_d):
    planes, scales = (p.B, p.Hkv, p.Sk, p.D), (p.B, p.Hkv, p.Sk, p.D // 32)
    return {"k_q": (k_q, planes, torch.int8), "v_q": (v_q, planes, torch.int8),
            "k_d": (k_d, scales, torch.float16), "v_d": (v_d, scales, torch.float16)}


def fwd_q8(q, k_q, k_d, v_q, v_d, mask=None, *, scale=None, causal=False, q_offset=None, window=0, layout="bhsd",
           out=None, lse=None, workspace=None, stream=None):
    """Forward over a q8_0 K/V cache (int8 values k_q/v_q, fp16 scales k_d/v_d per 32 features)."""
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    kv = _kv_q8(k_q, k_d, v_q, v_d)
    p = make_params(q, _cache_shape_view(k_q, layout), mask, scale=scale, causal=causal, q_offset=q_offset,
                    window=window, kv_format=FA_KV_Q8_0, layout=layout)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensors(q, **_common_expect(p, layout, q, mask=mask, o=out, lse=lse), **_q8_expect(p, k_q, k_d, v_q, v_d))
    _need_cuda(q, mview, out, lse, k_q, k_d, v_q, v_d)
    ws_bytes = fwd_workspace_size(p)
    ws = _workspace(ws_bytes, q.device, workspace)
    with _on_device(q):
        _check(lib.fa_train_fwd_q8(ctypes.byref(p), _ptr(q), ctypes.byref(kv), _ptr(mview), _ptr(out), _ptr(lse),
                                   _ptr(ws), ws_bytes, _stream(q.device, stream)))
    return out, lse


def bwd_q8(q, k_q, k_d, v_q, v_d, o, lse, do, mask=None, *, scale=None, causal=False, q_offset=None, window=0,
           deterministic=False, layout="bhsd", dq=None, dk=None, dv=None, dk_acc=None, dv_acc=None, workspace=None,
           stream=None):
    """Backward over a q8_0 K/V cache. With dk_acc/dv_acc (fp32) the gradients of the dequantized
    K/V are added into them (returns dQ); otherwise returns (dQ, dK, dV) in q's dtype."""
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    kv = _kv_q8(k_q, k_d, v_q, v_d)
    p = make_params(q, _cache_shape_view(k_q, layout), mask, scale=scale, causal=causal, q_offset=q_offset,
                    window=window, deterministic=deterministic, kv_format=FA_KV_Q8_0, layout=layout)
    dq = torch.empty_like(q) if dq is None else dq
    if (dk_acc is None) != (dv_acc is None):
        raise ValueError("give both dk_acc and dv_acc, or neither")
    ks = _kv_shape(p, layout)
    _check_tensors(q, **_common_expect(p, layout, q, mask=mask, o=o, lse=lse, do=do, dq=dq),
                   **_q8_expect(p, k_q, k_d, v_q, v_d), dk_acc=(dk_acc, ks, torch.float32),
                   dv_acc=(dv_acc, ks, torch.float32), dk=(dk, ks, q.dtype), dv=(dv, ks, q.dtype))
    _need_cuda(q, o, lse, do, mview, dq, dk_acc, dv_acc, dk, dv, k_q, k_d, v_q, v_d)
    ws_bytes = bwd_workspace_size(p)
    ws = _workspace(ws_bytes, q.device, workspace)
    if dk_acc is not None:
        with _on_device(q):
            _check(lib.fa_train_bwd_accum_q8(ctypes.byref(p), _ptr(q), ctypes.byref(kv), _ptr(mview), _ptr(o), _ptr(lse),
                                             _ptr(do), _ptr(dq), _ptr(dk_acc), _ptr(dv_acc), _ptr(ws), ws_bytes,
                                             _stream(q.device, stream)))
        return dq
    shape = tuple(_cache_shape_view(k_q, layout).shape)   # dK / dV in the call's layout
    dk = torch.empty(shape, dtype=q.dtype, device=q.device) if dk is None else dk
    dv = torch.empty(shape, dtype=q.dtype, device=q.device) if dv is None else dv
    with _on_device(q):
        _check(lib.fa_train_bwd_q8(ctypes.byref(p), _ptr(q), ctypes.byref(kv), _ptr(mview), _ptr(o), _ptr(lse),
                                   _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws_bytes, _stream(q.device, stream)))
    return dq, dk, dv


def set_rows_backward(acc: torch.Tensor, idx: torch.Tensor, out_dtype=torch.bfloat16, out=None, stream=None):
    """SET_ROWS backward: out[b, h, r] = acc[b, h, idx[r]] (acc fp32 [B, H, S, D], idx int64 [n])."""
    if acc.dtype != torch.float32 or acc.dim() != 4:
        raise TypeError("acc must be float32 [B, H, S, D]")
    if idx.dtype != torch.int64 or idx.dim() != 1:
        raise TypeError("idx must be int64 [n_rows]")
    B, H, S, D = acc.shape
    if out is None:
        out = torch.empty((B, H, idx.shape[0], D), dtype=out_dtype, device=acc.device)
    if tuple(out.shape) != (B, H, idx.shape[0], D):
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {(B, H, idx.shape[0], D)}")
    _need_cuda(acc, idx, out)
    with _on_device(acc):
        _check(load_library().fa_set_rows_backward(_ptr(acc), B, H, S, D, _ptr(idx), idx.shape[0], _ptr(out),
                                                   _dtype_code(out), _stream(acc.device, stream)))
    return out


def profile_set_events(kernel: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event start/stop around a kernel family on later calls (None clears)."""
    _check(load_library().fa_profile_set_events(kernel, None if start is None else start.cuda_event,
                                                None if stop is None else stop.cuda_event))


def profile_launch_count() -> int:
    """Kernels the library has launched from this thread so far."""
    return int(load_library().fa_profile_launch_count())


WAIT_SELFTEST_SITE = 900


def selftest_wait(limit_ms: int = 50, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait nothing ever satisfies); see device_status()."""
    import torch as _torch
    dev = _torch.device("cuda", _torch.cuda.current_device())
    _check(load_library().fa_train_selftest_wait(int(limit_ms), _stream(dev, stream)))


def device_status() -> int:
    """Read and clear the kernels' status word (0 = every bounded wait completed)."""
    v = ctypes.c_uint32(0)
    _check(load_library().fa_device_status(ctypes.byref(v)))
    return int(v.value)


NOALLOC_SCRATCH_BYTES = 16 << 20


def bwd_noalloc(q, k, v, o, lse, do, mask=None, *, scale=None, causal=False, q_offset=None, window=0,
                deterministic=False, layout="bhsd", dq=None, dk=None, dv=None, stream=None):
    """Backward through fa_train_bwd_noalloc: no workspace is allocated or passed.

    For callers that cannot allocate device memory (their memory is owned by another
    allocator, or allocation is not allowed where they run). The library keeps the scratch in
    a fixed 16 MiB device array; larger shapes raise FaError (FA_ERR_WORKSPACE). Calls that
    overlap on the GPU share that array and race.
    """
    lib = load_library()
    mview, _, _ = _mask_view(mask)
    p = make_params(q, k, mask, scale=scale, causal=causal, q_offset=q_offset, window=window,
                    deterministic=deterministic, kv_format=_kv_format(q, k, v), layout=layout)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k, dtype=q.dtype) if dk is None else dk   # q's dtype for an fp16 cache too
    dv = torch.empty_like(v, dtype=q.dtype) if dv is None else dv
    ks = _kv_shape(p, layout)
    _check_tensors(q, **_common_expect(p, layout, q, k, v, mask, o, lse, do, dq), dk=(dk, ks, q.dtype),
                   dv=(dv, ks, q.dtype))
    _need_cuda(q, k, v, o, lse, do, mview, dq, dk, dv)
    # the library finds its static scratch, and launches, on the current device: make it q's
    with _on_device(q):
        _check(lib.fa_train_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(mview), _ptr(o),
                                        _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _stream(q.device, stream)))
    return dq, dk, dv
