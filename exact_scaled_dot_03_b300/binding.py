"""Thin Python binding over the C ABI in ``include/attn.h``.

Argument marshalling only: PyTorch tensors supply device memory and the
current CUDA stream; every step of the computation runs in the CUDA library.
If the library has not been built, or a call fails, this raises instead of
computing anything another way.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_NAME = "libattn_sm103.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_ARG = range(6)

# name -> (restype, argtypes): the exported surface of include/attn.h
_vp, _i, _f, _sz, _i64, _u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                                ctypes.c_int64, ctypes.c_uint64)
SIGNATURES = {
    "attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "attn_fwd_window": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "attn_fwd_host_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "attn_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "attn_fwd_rope_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "attn_fwd_rope": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _f, _vp, _sz, _vp]),
    "attn_bwd_workspace_size": (_sz, [_i, _i, _i]),
    "attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "attn_decode_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "attn_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "attn_device_status": (_i, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "attn_status_string": (ctypes.c_char_p, [_i]),
    "attn_score_bytes": (_u64, [_i64, _i64, _i]),
    "attn_kv_cache_bytes": (_u64, [_i64, _i64, _i64, _i64, _i]),
    "attn_version": (ctypes.c_char_p, []),
    "attn_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "attn_test_arm_stall": (_i, [_i]),
    "attn_decode_paged_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "attn_decode_paged": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                               _vp, _sz, _vp]),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code) if _lib is not None else code} (status {code})")


def lib() -> ctypes.CDLL:
    """Load the CUDA library (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_NAME} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().attn_status_string(code).decode()


def _check(code: int, where: str):
    if code != OK:
        raise AttnError(code, where)


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16, dims=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")


def default_scale(d: int) -> float:
    """1/sqrt(d) rounded to fp32 (the pages' score scaling)."""
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def fwd(q, k, v, causal: bool, scale: float | None = None, out=None, lse=None, want_lse: bool = True,
        stream=None, window: int = 0):
    """Exact attention forward: returns (o, lse); see ``attn_fwd`` / ``attn_fwd_window``
    (window > 0: local window) in include/attn.h.

    q: [B, Hq, Nq, d], k/v: [B, Hkv, Nk, d], bf16 CUDA tensors.
    """
    _need(q, "q", dims=4)
    _need(k, "k", dims=4)
    _need(v, "v", dims=4)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("q/k/v shapes disagree")
    o = torch.empty_like(q) if out is None else out
    _need(o, "out", dims=4)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", dtype=torch.float32, dims=3)
    s = default_scale(d) if scale is None else float(scale)
    code = lib().attn_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr() if lse is not None else None,
                                 B, Hq, Hkv, Nq, Nk, d, s, int(bool(causal)), int(window), _stream_handle(stream))
    _check(code, "attn_fwd_window")
    return o, lse


def _need_host(t: torch.Tensor, name: str, dtype=torch.bfloat16, dims=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")


def fwd_host_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    return int(lib().attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d))


def fwd_host(q, k, v, causal: bool, scale: float | None = None, out=None, lse=None, want_lse: bool = True,
             workspace=None, stream=None, device=None):
    """Prefill on host tensors: returns (o, lse) in host memory; see ``attn_fwd_host``
    in include/attn.h. Pinned tensors (``pin_memory()``) let the copies overlap
    the kernels. The results are complete once ``stream`` has passed the call
    (``stream.synchronize()``); the call itself returns as soon as the work is queued.

    q: [B, Hq, Nq, d], k/v: [B, Hkv, Nk, d], bf16 host tensors; workspace: a uint8
    CUDA tensor of at least ``fwd_host_workspace_size`` bytes (allocated here if None).
    """
    _need_host(q, "q", dims=4)
    _need_host(k, "k", dims=4)
    _need_host(v, "v", dims=4)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("q/k/v shapes disagree")
    pin = q.is_pinned()
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin) if out is None else out
    _need_host(o, "out", dims=4)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=pin)
    if lse is not None:
        _need_host(lse, "lse", dtype=torch.float32, dims=3)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    need = fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", dtype=torch.uint8)
    s = default_scale(d) if scale is None else float(scale)
    with torch.cuda.device(workspace.device):
        code = lib().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, B, Hq, Hkv, Nq, Nk, d, s,
                                   int(bool(causal)), workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(code, "attn_fwd_host")
    return o, lse


def fwd_rope(q, k, v, causal: bool, scale: float | None = None, window: int = 0, base: float = 10000.0,
             workspace=None, out=None, lse=None, want_lse: bool = True, stream=None):
    """Prefill with RoPE on Q and K: returns (o, lse); see ``attn_fwd_rope`` in include/attn.h."""
    _need(q, "q", dims=4)
    _need(k, "k", dims=4)
    _need(v, "v", dims=4)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if workspace is None:
        n = int(lib().attn_fwd_rope_workspace_size(B, Hkv, Nq, Nk, d))
        if n == 0:
            raise AttnError(ERR_UNSUPPORTED, "attn_fwd_rope_workspace_size")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    s = default_scale(d) if scale is None else float(scale)
    code = lib().attn_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr() if lse is not None else None, B, Hq, Hkv, Nq, Nk, d, s,
                               int(bool(causal)), int(window), float(base), workspace.data_ptr(), workspace.numel(),
                               _stream_handle(stream))
    _check(code, "attn_fwd_rope")
    return o, lse


def bwd(q, k, v, o, lse, dout, causal: bool, scale: float | None = None, workspace=None, dq=None, dk=None, dv=None,
        stream=None):
    """Backward of ``fwd``: returns (dq, dk, dv); see ``attn_bwd`` in include/attn.h."""
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, name, dims=4)
    _need(lse, "lse", dtype=torch.float32, dims=3)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if workspace is None:
        n = int(lib().attn_bwd_workspace_size(B, Hq, Nq))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    s = default_scale(d) if scale is None else float(scale)
    code = lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Nq, Nk, d, s, int(bool(causal)),
                          workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(code, "attn_bwd")
    return dq, dk, dv


def decode_workspace_size(B: int, Hq: int, Hkv: int, Lmax: int, d: int) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, Hkv, Lmax, d))


def decode_workspace(B: int, Hq: int, Hkv: int, Lmax: int, d: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (the library keeps it zeroed between calls)."""
    n = decode_workspace_size(B, Hq, Hkv, Lmax, d)
    if n == 0:
        raise AttnError(ERR_UNSUPPORTED, "attn_decode_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def decode(q, k_cache, v_cache, seqlens, scale: float | None = None, workspace=None, out=None, lse=None,
           want_lse: bool = True, stream=None):
    """KV-cache decode: returns (o, lse); see ``attn_decode`` in include/attn.h.

    q: [B, Hq, d]; caches: [B, Hkv, Lmax, d] bf16; seqlens: [B] int32 (all CUDA).
    """
    _need(q, "q", dims=3)
    _need(k_cache, "k_cache", dims=4)
    _need(v_cache, "v_cache", dims=4)
    _need(seqlens, "seqlens", dtype=torch.int32, dims=1)
    B, Hq, d = q.shape
    _, Hkv, Lmax, _ = k_cache.shape
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, Lmax, d, device=q.device)
    _need(workspace, "workspace", dtype=torch.uint8, dims=1)
    o = torch.empty_like(q) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    s = default_scale(d) if scale is None else float(scale)
    code = lib().attn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seqlens.data_ptr(),
                             o.data_ptr(), lse.data_ptr() if lse is not None else None,
                             B, Hq, Hkv, Lmax, d, s, workspace.data_ptr(), workspace.numel(),
                             _stream_handle(stream))
    _check(code, "attn_decode")
    return o, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, k_new=None, v_new=None, scale: float | None = None,
                 workspace=None, out=None, lse=None, want_lse: bool = True, stream=None):
    """Paged KV-cache decode with optional fused append: returns (o, lse); see
    ``attn_decode_paged`` in include/attn.h.

    q: [B, Hq, d]; pages: [num_pages, Hkv, page_size, d] bf16; block_table:
    [B, max_pages] int32; seqlens: [B] int32 (tokens already cached); k_new,
    v_new: [B, Hkv, d] bf16 or None. The appended rows are written into the pages.
    """
    _need(q, "q", dims=3)
    _need(k_pages, "k_pages", dims=4)
    _need(v_pages, "v_pages", dims=4)
    _need(block_table, "block_table", dtype=torch.int32, dims=2)
    _need(seqlens, "seqlens", dtype=torch.int32, dims=1)
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        _need(k_new, "k_new", dims=3)
        _need(v_new, "v_new", dims=3)
    B, Hq, d = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    max_pages = block_table.shape[1]
    if workspace is None:
        n = int(lib().attn_decode_paged_workspace_size(B, Hq, Hkv, max_pages, page_size, d))
        if n == 0:
            raise AttnError(ERR_UNSUPPORTED, "attn_decode_paged_workspace_size")
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    _need(workspace, "workspace", dtype=torch.uint8, dims=1)
    o = torch.empty_like(q) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    s = default_scale(d) if scale is None else float(scale)
    code = lib().attn_decode_paged(q.data_ptr(), k_new.data_ptr() if k_new is not None else None,
                                   v_new.data_ptr() if v_new is not None else None, k_pages.data_ptr(),
                                   v_pages.data_ptr(), block_table.data_ptr(), seqlens.data_ptr(), o.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, B, Hq, Hkv, num_pages, page_size,
                                   max_pages, d, s, workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(code, "attn_decode_paged")
    return o, lse


def device_status(stream=None):
    """Synchronise the stream and read/clear the device status: (code, [flags, site, block])."""
    detail = (ctypes.c_uint * 3)()
    code = lib().attn_device_status(_stream_handle(stream), detail)
    return code, list(detail)
