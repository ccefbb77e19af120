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


def _check_input(name: str, t: torch.Tensor, dtype=None) -> None:
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


def _shape(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    """(Z, H, Hkv, Nq, Nk, D) of q [Z,H,Nq,D] and k, v [Z,Hkv,Nk,D]."""
    _check_input("q", q)
    _check_input("k", k, q.dtype)
    _check_input("v", v, q.dtype)
    Z, H, Nq, D = q.shape
    Zk, Hkv, Nk, Dk = k.shape
    if Zk != Z or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k {tuple(k.shape)} and v {tuple(v.shape)} must be [Z, Hkv, Nk, D] with q's Z and D")
    if H % Hkv != 0:
        raise ValueError(f"q's {H} heads are not a multiple of k's {Hkv} heads")
    return Z, H, Hkv, Nq, Nk, D


def _dtype_code(t: torch.Tensor) -> int:
    return _native.FA_DTYPE_BF16 if t.dtype == torch.bfloat16 else _native.FA_DTYPE_F16


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: Optional[float] = None, out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
        stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Exact attention forward.  q [Z,H,Nq,D], k and v [Z,Hkv,Nk,D] (H a
    multiple of Hkv; query head h reads K/V head h // (H // Hkv)), all
    float16 or all bfloat16.  Returns ``(o, lse)``: o like q, lse fp32
    [Z,H,Nq] (natural-log log-sum-exp of each row of scale*Q K^T).  Causal:
    query i sees key j iff j <= i + Nk - Nq (needs Nq <= Nk)."""
    Z, H, Hkv, Nq, Nk, D = _shape(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((Z, H, Nq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
        _check_input("o", o, q.dtype)
        if tuple(o.shape) != tuple(q.shape) or lse.dtype != torch.float32 or tuple(lse.shape) != (Z, H, Nq):
            raise ValueError("out must be (o like q, float32 lse [Z, H, Nq])")
    rc = _native.lib().fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 Z, H, Hkv, Nq, Nk, D, int(bool(causal)), float(scale), _dtype_code(q),
                                 _stream_handle(stream))
    _native.check(rc, "fa_fwd_ex")
    return o, lse


def reshape_and_cache(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write new tokens' K and V ([T, Hkv, D]) into the paged caches
    ([num_pages, page_size, Hkv, D]) at the slots of ``slot_mapping`` (int64
    [T]); negative slots are skipped."""
    for name, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        if not t.is_cuda or t.dtype not in _DTYPES or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float16/bfloat16 CUDA tensor")
        if t.dtype != k_cache.dtype:
            raise ValueError(f"{name} is {t.dtype}, expected {k_cache.dtype} like k_cache")
    T, Hkv, D = k_new.shape
    num_pages, page_size, Hkv_c, Dc = k_cache.shape
    if tuple(v_new.shape) != (T, Hkv, D) or (Hkv_c, Dc) != (Hkv, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_new, v_new must be [T, Hkv, D] and the caches [num_pages, page_size, Hkv, D]")
    if not slot_mapping.is_cuda or slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != (T,):
        raise ValueError("slot_mapping must be an int64 CUDA tensor [T]")
    rc = _native.lib().fa_reshape_and_cache(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(),
                                            k_cache.data_ptr(), v_cache.data_ptr(), T, Hkv, D, num_pages,
                                            page_size, _stream_handle(stream))
    _native.check(rc, "fa_reshape_and_cache")


def fwd_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
              context_lens: torch.Tensor, causal: bool = False, scale: Optional[float] = None,
              out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
              stream: Optional[torch.cuda.Stream] = None, splits: int = 1,
              workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention forward over a paged K/V cache.  q [B,H,Nq,D]; k_cache,
    v_cache [num_pages, page_size, Hkv, D] (q's dtype); block_table int32
    [B, max_pages] (sequence b's key p is in page block_table[b, p //
    page_size]); context_lens int32 [B].  Causal: the queries are the last
    Nq of each sequence's context.  Returns ``(o, lse)`` like :func:`fwd`.

    ``splits`` > 1 cuts each sequence's key range into that many slices
    (``fa_fwd_paged_split``, for batches too small to fill the GPU); 0 lets
    the library choose (``fa_fwd_paged_split_count``).  ``workspace`` is an
    optional uint8 CUDA tensor of at least
    ``fa_fwd_paged_split_workspace_size`` bytes; one is allocated if None."""
    _check_input("q", q)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check_input(name, t, q.dtype)
    B, H, Nq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must be [num_pages, page_size, Hkv, D] with q's D")
    if H % Hkv != 0:
        raise ValueError(f"q's {H} heads are not a multiple of the cache's {Hkv} heads")
    for name, t in (("block_table", block_table), ("context_lens", context_lens)):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and context_lens [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    lib = _native.lib()
    max_pages = block_table.shape[1]
    if splits == 0:
        splits = lib.fa_fwd_paged_split_count(B, H, Hkv, Nq, D, page_size, max_pages, int(bool(causal)))
    if splits == 1:
        rc = lib.fa_fwd_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                              context_lens.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq, D, num_pages,
                              page_size, max_pages, int(bool(causal)), float(scale), _dtype_code(q),
                              _stream_handle(stream))
        _native.check(rc, "fa_fwd_paged")
        return o, lse
    need = lib.fa_fwd_paged_split_workspace_size(B, H, Nq, D, int(splits))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.fa_fwd_paged_split(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                                context_lens.data_ptr(), o.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), B, H, Hkv, Nq, D, num_pages, page_size,
                                max_pages, int(splits), int(bool(causal)), float(scale), _dtype_code(q),
                                _stream_handle(stream))
    _native.check(rc, "fa_fwd_paged_split")
    return o, lse


def paged_split_count(B: int, H: int, Hkv: int, Nq: int, D: int, page_size: int, max_pages: int,
                      causal: bool = False) -> int:
    """The slice count ``fwd_paged(splits=0)`` would use on the current device."""
    return _native.lib().fa_fwd_paged_split_count(B, H, Hkv, Nq, D, page_size, max_pages, int(bool(causal)))


def fwd_sparse(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, sel_pages: torch.Tensor,
               sel_blocks: torch.Tensor, sel_count: torch.Tensor, context_lens: torch.Tensor, causal: bool = False,
               scale: Optional[float] = None, stream: Optional[torch.cuda.Stream] = None
               ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention forward over selected blocks of a paged cache.  q
    [B,H,Nq,D]; caches as for :func:`fwd_paged`; sel_pages, sel_blocks int32
    [B, Hkv, max_sel] (physical page and logical block of each selected
    entry), sel_count int32 [B, Hkv], context_lens int32 [B].  Returns
    ``(o, lse)``; rows with no visible selected token get o = 0, lse = -inf."""
    _check_input("q", q)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check_input(name, t, q.dtype)
    B, H, Nq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape) or H % Hkv != 0:
        raise ValueError("caches must be [num_pages, page_size, Hkv, D] with q's D and Hkv dividing H")
    for name, t in (("sel_pages", sel_pages), ("sel_blocks", sel_blocks), ("sel_count", sel_count),
                    ("context_lens", context_lens)):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if sel_pages.dim() != 3 or tuple(sel_pages.shape[:2]) != (B, Hkv) or tuple(sel_blocks.shape) != tuple(sel_pages.shape):
        raise ValueError("sel_pages and sel_blocks must be [B, Hkv, max_sel]")
    if tuple(sel_count.shape) != (B, Hkv) or tuple(context_lens.shape) != (B,):
        raise ValueError("sel_count must be [B, Hkv] and context_lens [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    rc = _native.lib().fa_fwd_sparse(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), sel_pages.data_ptr(),
                                     sel_blocks.data_ptr(), sel_count.data_ptr(), context_lens.data_ptr(),
                                     o.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq, D, num_pages, page_size,
                                     sel_pages.shape[2], int(bool(causal)), float(scale), _dtype_code(q),
                                     _stream_handle(stream))
    _native.check(rc, "fa_fwd_sparse")
    return o, lse


def bwd_workspace_size(Z: int, H: int, N: int, D: int, causal: bool, Hkv: Optional[int] = None,
                       Nk: Optional[int] = None) -> int:
    """Workspace bytes of a backward call; N is the query length."""
    Hkv = H if Hkv is None else Hkv
    Nk = N if Nk is None else Nk
    return int(_native.lib().fa_bwd_ex_workspace_size(Z, H, Hkv, N, Nk, D, int(bool(causal))))


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, do: torch.Tensor,
        lse: torch.Tensor, causal: bool = False, scale: Optional[float] = None,
        workspace: Optional[torch.Tensor] = None, out=None,
        stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Exact attention backward.  Shapes as for :func:`fwd`; o and do like q.
    Returns ``(dq, dk, dv)`` shaped like q, k, v; dk and dv of a shared K/V
    head sum over the query heads that read it."""
    Z, H, Hkv, Nq, Nk, D = _shape(q, k, v)
    for name, t in (("o", o), ("do", do)):
        _check_input(name, t, q.dtype)
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(q.shape)}")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (Z, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [Z, H, Nq] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = bwd_workspace_size(Z, H, Nq, D, causal, Hkv, Nk)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    rc = _native.lib().fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                 lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), Z, H, Hkv, Nq, Nk, D,
                                 int(bool(causal)), float(scale), _dtype_code(q), _stream_handle(stream))
    _native.check(rc, "fa_bwd_ex")
    return dq, dk, dv


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream; return and clear the library's device status."""
    import ctypes
    raw = ctypes.c_int(0)
    rc = _native.lib().fa_device_status_raw(_stream_handle(stream), ctypes.byref(raw))
    return rc if rc != _native.FA_OK else 0


def fwd_flops(Z, H, N, D, causal, Nk=None) -> float:
    Nk = N if Nk is None else Nk
    return float(_native.lib().fa_fwd_ex_flops(Z, H, N, Nk, D, int(bool(causal))))


def bwd_flops(Z, H, N, D, causal, Nk=None) -> float:
    Nk = N if Nk is None else Nk
    return float(_native.lib().fa_bwd_ex_flops(Z, H, N, Nk, D, int(bool(causal))))
