"""HSTU attention for GB300 (sm_103a).

A thin Python binding over the C ABI of ``libhstu_attn.so``
(``include/hstu_attn.h``).  Every step of the computation runs in the
library's CUDA kernels; this module only checks tensor metadata, allocates
outputs and the workspace with torch, and passes pointers, strides and the
current CUDA stream.  There is no CPU fallback: if the library is missing or
the device is not sm_103, calls raise.

Operation ("HSTU Attention (Blackwell SM100/SM103)", Overview): per packed
sequence and head, O = (1/L_scale) (M (.) SiLU(alpha Q K^T)) V, no softmax.
``hstu_attn_fwd`` / ``hstu_attn_bwd`` mirror the page's
``hstu_attention_forward`` / ``hstu_attention_backward`` ("High-level
functions"): THD tensors, int32 cumulative lengths, ``scaling_seqlen=None``
meaning ``max_seqlen_q``, ``window_size=(left, right)`` the token-window mask
(-1: no bound on that side; ``(-1, 0)`` causal, ``(-1, -1)`` full); without
``window_size`` the ``causal`` flag picks one of those two.
"""
from __future__ import annotations

from typing import Optional, Tuple

from ._lib import (HstuError, HSTU_BF16, HSTU_FP16, library, library_path,
                   workspace_size, workspace_size_func, plan_workspace_size, last_device_status,
                   selftest_timeout, CTen, Ten)

__all__ = ["hstu_attn_fwd", "hstu_attn_bwd", "hstu_attn_fwd_paged", "hstu_attn_plan",
           "HstuPlan", "workspace_size", "plan_workspace_size", "last_device_status",
           "selftest_timeout", "HstuError", "library", "library_path"]


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return HSTU_BF16
    if t.dtype == torch.float16:
        return HSTU_FP16
    raise TypeError(f"HSTU attention takes fp16 or bf16 tensors, got {t.dtype}")


def _check_thd(name, t, T, H, D, dtype, device):
    if t.dim() != 3 or tuple(t.shape) != (T, H, D):
        raise ValueError(f"{name}: expected shape {(T, H, D)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype} differs from q's {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if T > 0 and t.stride(2) != 1:
        raise ValueError(f"{name}: the last (head_dim) dimension must be contiguous")


def _cten(t):
    return CTen(t.data_ptr(), t.stride(0), t.stride(1))


def _ten(t):
    return Ten(t.data_ptr(), t.stride(0), t.stride(1))


def _window(causal, window_size):
    """(left, right) of the mask: ``window_size`` when given, else causal
    (-1, 0) or full (-1, -1)."""
    if window_size is None:
        return (-1, 0) if bool(causal) else (-1, -1)
    w = tuple(int(x) for x in window_size)
    if len(w) != 2 or w[0] < -1 or w[1] < -1:
        raise ValueError(f"window_size {window_size}: two bounds, each -1 (none) or >= 0")
    return w


def _func_args(func, T_q, device):
    """(pointer, N, L) of an arbitrary-mask endpoint tensor: int32, (1, N, L)
    or (N, L), contiguous, N odd, L >= T_q, on the device."""
    import torch
    f = func[0] if func.dim() == 3 else func
    if func.dtype != torch.int32 or f.dim() != 2 or func.device != device:
        raise ValueError(f"func: int32 (1, N, L) or (N, L) on {device}")
    if not func.is_contiguous() or f.shape[0] % 2 != 1 or f.shape[1] < T_q:
        raise ValueError("func: contiguous, N odd, L >= total_q")
    return func.data_ptr(), int(f.shape[0]), int(f.shape[1])


def _scaling(scaling_seqlen):
    if scaling_seqlen is None:
        return 0
    s = int(scaling_seqlen)
    if s <= 0:
        raise ValueError("scaling_seqlen must be positive")
    return s


def _meta(cu_seqlens_q, cu_seqlens_k, device):
    import torch
    for n, c in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if c.dtype != torch.int32 or c.dim() != 1 or c.device != device:
            raise ValueError(f"{n}: expected a 1-D int32 tensor on {device}")
        if not c.is_contiguous():
            raise ValueError(f"{n}: must be contiguous")
    if cu_seqlens_q.shape != cu_seqlens_k.shape:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be (B + 1,)")
    return cu_seqlens_q.shape[0] - 1


def _workspace(workspace, nbytes, device):
    import torch
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return workspace


def _event_array(events):
    import ctypes
    handles = [e.cuda_event for e in events]   # torch creates the event lazily
    if any(h == 0 for h in handles):
        raise ValueError("events must have been created on the device (record them once first)")
    arr = (ctypes.c_void_p * len(handles))(*handles)
    return arr, len(handles)


def _stream(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


class HstuPlan:
    """The schedule of one batch layout (``hstu_attn_plan``): the forward's
    and the backward's work lists, built in one launch and shared by any
    number of ``plan=`` calls in stream order.  ``workspace`` holds it and
    also serves as the backward's workspace."""

    def __init__(self, workspace, key):
        self.workspace = workspace
        self.key = key

    def check(self, key):
        if key != self.key:
            raise ValueError(f"call sizes {key} differ from the plan's {self.key}")


def hstu_attn_plan(cu_seqlens_q, cu_seqlens_k, total_q: int, total_k: int, num_heads: int,
                   head_dim: int, max_seqlen_q: int, max_seqlen_k: int, causal: bool = True,
                   window_size=None, workspace=None) -> HstuPlan:
    """Builds the schedule of one batch layout for planned calls (no host
    synchronization: cu_seqlens are read on the device)."""
    lib = library()
    dev = cu_seqlens_q.device
    B = _meta(cu_seqlens_q, cu_seqlens_k, dev)
    win = _window(causal, window_size)
    key = (B, int(total_q), int(total_k), int(num_heads), int(head_dim), int(max_seqlen_q),
           int(max_seqlen_k), win)
    ws = _workspace(workspace, plan_workspace_size(*key[:7]), dev)
    st = lib.hstu_attn_plan(cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), *key[:7],
                            win[0], win[1], ws.data_ptr(), ws.numel(), _stream(dev))
    if st != 0:
        raise HstuError(st)
    return HstuPlan(ws, key)


def hstu_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  scaling_seqlen: Optional[int] = None, causal: bool = True,
                  alpha: float = 1.0, out=None, workspace=None, window_size=None,
                  events=None, func=None, plan: Optional[HstuPlan] = None):
    """Forward HSTU attention; returns ``out`` of shape ``q.shape``.

    ``plan``: an ``HstuPlan`` of this batch layout; the call then uses its
    schedule (and ignores ``workspace``).

    q: (T_q, H, D); k, v: (T_k, H, D); fp16 or bf16 on a CUDA device.
    cu_seqlens_q/k: int32 (B + 1,) on the same device (values are trusted and
    never copied to the host).  ``out`` may be supplied (overwritten).
    ``events``: optional list of 3 torch.cuda.Event recorded before the
    scheduler, after it and after the forward kernel (profiling).
    ``func``: optional arbitrary-mask endpoints (the page's func_tensor, int32
    (1, N, L)); it replaces ``causal`` / ``window_size``.
    """
    import torch
    lib = library()
    T_q, H, D = q.shape
    T_k = k.shape[0]
    dev = q.device
    _check_thd("k", k, T_k, H, D, q.dtype, dev)
    _check_thd("v", v, T_k, H, D, q.dtype, dev)
    _check_thd("q", q, T_q, H, D, q.dtype, dev)
    B = _meta(cu_seqlens_q, cu_seqlens_k, dev)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    _check_thd("out", out, T_q, H, D, q.dtype, dev)
    win = _window(causal, window_size)
    if func is not None:
        if plan is not None:
            raise ValueError("arbitrary (func) masks are not planned")
        fp, fn, fl = _func_args(func, T_q, dev)
        ws = _workspace(workspace, workspace_size_func(B, T_q, T_k, H, D, max_seqlen_q,
                                                       max_seqlen_k, False), dev)
        st = lib.hstu_attn_fwd_func(_cten(q), _cten(k), _cten(v), _ten(out),
                                    cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, T_q, T_k,
                                    H, D, _dtype_code(q), int(max_seqlen_q), int(max_seqlen_k),
                                    float(alpha), _scaling(scaling_seqlen), fp, fn, fl,
                                    ws.data_ptr(), ws.numel(), _stream(dev))
        if st != 0:
            raise HstuError(st)
        return out
    if plan is not None:
        if events is not None:
            raise ValueError("events are not recorded by planned calls")
        plan.check((B, T_q, T_k, H, D, int(max_seqlen_q), int(max_seqlen_k), win))
        ws = plan.workspace
    else:
        ws = _workspace(workspace, workspace_size(B, T_q, T_k, H, D, max_seqlen_q,
                                                  max_seqlen_k, False), dev)
    args = (_cten(q), _cten(k), _cten(v), _ten(out), cu_seqlens_q.data_ptr(),
            cu_seqlens_k.data_ptr(), B, T_q, T_k, H, D, _dtype_code(q), int(max_seqlen_q),
            int(max_seqlen_k), float(alpha), _scaling(scaling_seqlen), win[0], win[1],
            ws.data_ptr(), ws.numel(), _stream(dev))
    if plan is not None:
        st = lib.hstu_attn_fwd_planned(*args)
    elif events is None:
        st = lib.hstu_attn_fwd(*args)
    else:
        arr, n = _event_array(events)
        st = lib.hstu_attn_fwd_profiled(*args, arr, n)
    if st != 0:
        raise HstuError(st)
    return out


def hstu_attn_fwd_paged(q, paged_kv, page_ids, page_indptrs, cu_seqlens_q, cu_seqlens_k,
                        max_seqlen_q: int, max_seqlen_k: int,
                        scaling_seqlen: Optional[int] = None, alpha: float = 1.0, out=None,
                        workspace=None):
    """Causal forward over a paged K/V cache; returns ``out`` (shape of q).

    paged_kv: contiguous (num_pages, 2, 128, H, D), K at [:, 0] and V at [:, 1];
    page_ids: int32 physical page of each 128-key block, per sequence the
    slice page_indptrs[b] : page_indptrs[b + 1]; page_indptrs: int32 (B + 1,).
    cu_seqlens_k gives the key counts.  Values are trusted, never copied to
    the host.  Rows of a page past its sequence's keys must be finite.
    """
    import torch
    lib = library()
    T_q, H, D = q.shape
    dev = q.device
    _check_thd("q", q, T_q, H, D, q.dtype, dev)
    if (paged_kv.dim() != 5 or paged_kv.shape[1] != 2 or paged_kv.shape[2] != 128
            or paged_kv.shape[3] != H or paged_kv.shape[4] != D):
        raise ValueError(f"paged_kv: shape {tuple(paged_kv.shape)}, expected (P, 2, 128, {H}, {D})")
    if paged_kv.dtype != q.dtype or paged_kv.device != dev or not paged_kv.is_contiguous():
        raise ValueError("paged_kv: q's dtype and device, contiguous")
    for name, t in (("page_ids", page_ids), ("page_indptrs", page_indptrs)):
        if t.dtype != torch.int32 or t.device != dev or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name}: contiguous 1-D int32 on {dev}")
    B = _meta(cu_seqlens_q, cu_seqlens_k, dev)
    if page_indptrs.shape[0] != B + 1:
        raise ValueError("page_indptrs: shape (B + 1,)")
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    _check_thd("out", out, T_q, H, D, q.dtype, dev)
    ws = _workspace(workspace, workspace_size(B, T_q, 0, H, D, max_seqlen_q, max_seqlen_k,
                                              False), dev)
    st = lib.hstu_attn_fwd_paged(_cten(q), paged_kv.data_ptr(), paged_kv.shape[0],
                                 page_ids.data_ptr(), page_indptrs.data_ptr(), _ten(out),
                                 cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, T_q, H, D,
                                 _dtype_code(q), int(max_seqlen_q), int(max_seqlen_k),
                                 float(alpha), _scaling(scaling_seqlen), ws.data_ptr(),
                                 ws.numel(), _stream(dev))
    if st != 0:
        raise HstuError(st)
    return out


def hstu_attn_bwd(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, scaling_seqlen: Optional[int] = None,
                  causal: bool = True, alpha: float = 1.0, dq=None, dk=None, dv=None,
                  workspace=None, window_size=None, events=None, func=None,
                  plan: Optional[HstuPlan] = None) -> Tuple:
    """Backward HSTU attention; returns ``(dq, dk, dv)``.

    Same arguments as the forward plus ``dout`` (shape of q).  Caller-owned
    ``dq``/``dk``/``dv`` may be supplied (overwritten); dk and dv may be
    disjoint views of one packed KV buffer.  ``events``: optional list of 4
    torch.cuda.Event (before the scheduler, after it, and twice after the
    backward kernel, which runs the dK/dV units and then the dQ units).
    """
    import torch
    lib = library()
    T_q, H, D = q.shape
    T_k = k.shape[0]
    dev = q.device
    _check_thd("q", q, T_q, H, D, q.dtype, dev)
    _check_thd("dout", dout, T_q, H, D, q.dtype, dev)
    _check_thd("k", k, T_k, H, D, q.dtype, dev)
    _check_thd("v", v, T_k, H, D, q.dtype, dev)
    B = _meta(cu_seqlens_q, cu_seqlens_k, dev)
    if dq is None:
        dq = torch.empty_like(q, memory_format=torch.contiguous_format)
    if dk is None:
        dk = torch.empty_like(k, memory_format=torch.contiguous_format)
    if dv is None:
        dv = torch.empty_like(v, memory_format=torch.contiguous_format)
    _check_thd("dq", dq, T_q, H, D, q.dtype, dev)
    _check_thd("dk", dk, T_k, H, D, q.dtype, dev)
    _check_thd("dv", dv, T_k, H, D, q.dtype, dev)
    win = _window(causal, window_size)
    if func is not None:
        if plan is not None:
            raise ValueError("arbitrary (func) masks are not planned")
        fp, fn, fl = _func_args(func, T_q, dev)
        ws = _workspace(workspace, workspace_size_func(B, T_q, T_k, H, D, max_seqlen_q,
                                                       max_seqlen_k, True), dev)
        st = lib.hstu_attn_bwd_func(_cten(dout), _cten(q), _cten(k), _cten(v), _ten(dq),
                                    _ten(dk), _ten(dv), cu_seqlens_q.data_ptr(),
                                    cu_seqlens_k.data_ptr(), B, T_q, T_k, H, D, _dtype_code(q),
                                    int(max_seqlen_q), int(max_seqlen_k), float(alpha),
                                    _scaling(scaling_seqlen), fp, fn, fl, ws.data_ptr(),
                                    ws.numel(), _stream(dev))
        if st != 0:
            raise HstuError(st)
        return dq, dk, dv
    if plan is not None:
        if events is not None:
            raise ValueError("events are not recorded by planned calls")
        plan.check((B, T_q, T_k, H, D, int(max_seqlen_q), int(max_seqlen_k), win))
        ws = plan.workspace
    else:
        ws = _workspace(workspace, workspace_size(B, T_q, T_k, H, D, max_seqlen_q,
                                                  max_seqlen_k, True), dev)
    args = (_cten(dout), _cten(q), _cten(k), _cten(v), _ten(dq), _ten(dk), _ten(dv),
            cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, T_q, T_k, H, D, _dtype_code(q),
            int(max_seqlen_q), int(max_seqlen_k), float(alpha), _scaling(scaling_seqlen),
            win[0], win[1], ws.data_ptr(), ws.numel(), _stream(dev))
    if plan is not None:
        st = lib.hstu_attn_bwd_planned(*args)
    elif events is None:
        st = lib.hstu_attn_bwd(*args)
    else:
        arr, n = _event_array(events)
        st = lib.hstu_attn_bwd_profiled(*args, arr, n)
    if st != 0:
        raise HstuError(st)
    return dq, dk, dv
