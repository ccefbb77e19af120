"""Python entry points: ``fwd`` and ``bwd`` over torch CUDA tensors.

Thin wrappers: validate tensor metadata, allocate outputs / workspace with
torch (device memory is PyTorch's job here), and call the C ABI on the
current torch stream.  All arithmetic happens inside libfa.so.
"""

from __future__ import annotations

import math
from typing import Optional, Tuple

import torch

from . import _native


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


_DTYPES = (torch.float16, torch.bfloat16)


def _check_input(name: str, t: torch.Tensor, shape=None, dtype=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if t.dtype not in _DTYPES:
        raise ValueError(f"{name} must be float16 or bfloat16, got {t.dtype}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} is {t.dtype}, expected {dtype} like q")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [Z, H, N, D] tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: Optional[float] = None, out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
        stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Exact attention forward.  Returns ``(o, lse)``: o [Z,H,N,D] in q's dtype
    (float16 or bfloat16), lse fp32 [Z,H,N] (natural-log log-sum-exp of each
    row of scale*Q K^T)."""
    _check_input("q", q)
    Z, H, N, D = q.shape
    _check_input("k", k, q.shape, q.dtype)
    _check_input("v", v, q.shape, q.dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((Z, H, N), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    fn = "fa_fwd_bf16" if q.dtype == torch.bfloat16 else "fa_fwd"
    rc = getattr(_native.lib(), fn)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    Z, H, N, D, int(bool(causal)), float(scale), _stream_handle(stream))
    _native.check(rc, fn)
    return o, lse


def bwd_workspace_size(Z: int, H: int, N: int, D: int, causal: bool) -> int:
    return int(_native.lib().fa_bwd_workspace_size(Z, H, N, D, int(bool(causal))))


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, do: torch.Tensor,
        lse: torch.Tensor, causal: bool = False, scale: Optional[float] = None,
        workspace: Optional[torch.Tensor] = None, out=None,
        stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Exact attention backward.  Returns ``(dq, dk, dv)`` [Z,H,N,D] in q's
    dtype (float16 or bfloat16)."""
    _check_input("q", q)
    Z, H, N, D = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check_input(name, t, q.shape, q.dtype)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (Z, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [Z, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = bwd_workspace_size(Z, H, N, D, causal)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    fn = "fa_bwd_bf16" if q.dtype == torch.bfloat16 else "fa_bwd"
    rc = getattr(_native.lib(), fn)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                    workspace.data_ptr(), workspace.numel(), Z, H, N, D, int(bool(causal)),
                                    float(scale), _stream_handle(stream))
    _native.check(rc, fn)
    return dq, dk, dv


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream; return and clear the library's device status."""
    import ctypes
    raw = ctypes.c_int(0)
    rc = _native.lib().fa_device_status_raw(_stream_handle(stream), ctypes.byref(raw))
    return rc if rc != _native.FA_OK else 0


def fwd_flops(Z, H, N, D, causal) -> float:
    return float(_native.lib().fa_fwd_flops(Z, H, N, D, int(bool(causal))))


def bwd_flops(Z, H, N, D, causal) -> float:
    return float(_native.lib().fa_bwd_flops(Z, H, N, D, int(bool(causal))))
