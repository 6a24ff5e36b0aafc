"""ctypes view of the C ABI in ``include/hstu_attn.h``.

Loads ``libhstu_attn.so`` from this package directory (built in-tree by
``build.py``).  A missing library raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libhstu_attn.so")
_lock = threading.Lock()
_lib = None

HSTU_FP16 = 0
HSTU_BF16 = 1

STATUS = {0: "HSTU_OK", 1: "HSTU_ERR_INVALID_ARG", 2: "HSTU_ERR_UNSUPPORTED",
          3: "HSTU_ERR_MISALIGNED", 4: "HSTU_ERR_CUDA", 5: "HSTU_ERR_DEVICE_TIMEOUT"}

# Every symbol include/hstu_attn.h declares.
EXPORTS = ("hstu_attn_fwd", "hstu_attn_bwd", "hstu_attn_fwd_profiled", "hstu_attn_bwd_profiled",
           "hstu_attn_workspace_size",
           "hstu_attn_status_string", "hstu_attn_last_device_status",
           "hstu_attn_selftest_timeout", "hstu_attn_version", "hstu_attn_fwd_noalloc",
           "hstu_attn_noalloc_last_device_status",
           "hstu_attn_fwd_paged", "hstu_attn_fwd_func", "hstu_attn_bwd_func",
           "hstu_attn_workspace_size_func", "hstu_attn_plan_workspace_size", "hstu_attn_plan",
           "hstu_attn_fwd_planned", "hstu_attn_bwd_planned", "hstu_lmsd_fwd", "hstu_lmsd_bwd",
           "hstu_lmsd_bwd_workspace_size")


class CTen(ctypes.Structure):
    """hstu_cten_t: read-only THD tensor (pointer, token and head strides in elements)."""
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_t", ctypes.c_int64),
                ("stride_h", ctypes.c_int64)]


class Ten(ctypes.Structure):
    """hstu_ten_t: writable THD tensor."""
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_t", ctypes.c_int64),
                ("stride_h", ctypes.c_int64)]


class HstuError(RuntimeError):
    def __init__(self, status: int):
        self.status = int(status)
        text = STATUS.get(self.status, "unknown")
        try:
            text += ": " + library().hstu_attn_status_string(self.status).decode()
        except Exception:
            pass
        super().__init__(f"hstu_attn failed with {text}")


def library_path() -> str:
    return _LIB_PATH


def _declare(lib):
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    P, S = ctypes.c_void_p, ctypes.c_size_t
    # ..., scaling_seqlen, window_left, window_right, workspace, bytes, stream
    scal = [P, P, i32, i64, i64, i32, i32, ctypes.c_int, i32, i32, f32, i32, i32, i32, P, S, P]
    lib.hstu_attn_fwd.argtypes = [CTen, CTen, CTen, Ten] + scal
    lib.hstu_attn_fwd.restype = ctypes.c_int
    lib.hstu_attn_bwd.argtypes = [CTen, CTen, CTen, CTen, Ten, Ten, Ten] + scal
    lib.hstu_attn_bwd.restype = ctypes.c_int
    lib.hstu_attn_fwd_profiled.argtypes = lib.hstu_attn_fwd.argtypes + [P, i32]
    lib.hstu_attn_fwd_profiled.restype = ctypes.c_int
    lib.hstu_attn_bwd_profiled.argtypes = lib.hstu_attn_bwd.argtypes + [P, i32]
    lib.hstu_attn_bwd_profiled.restype = ctypes.c_int
    lib.hstu_attn_workspace_size.argtypes = [i32, i64, i64, i32, i32, i32, i32, i32]
    lib.hstu_attn_workspace_size.restype = S
    lib.hstu_attn_status_string.argtypes = [ctypes.c_int]
    lib.hstu_attn_status_string.restype = ctypes.c_char_p
    lib.hstu_attn_last_device_status.argtypes = [P, P]
    lib.hstu_attn_last_device_status.restype = ctypes.c_int
    lib.hstu_attn_selftest_timeout.argtypes = [P, ctypes.c_uint32, P]
    lib.hstu_attn_selftest_timeout.restype = ctypes.c_int
    lib.hstu_attn_fwd_noalloc.argtypes = [CTen, CTen, CTen, Ten] + scal[:14] + [P]
    lib.hstu_attn_fwd_noalloc.restype = ctypes.c_int
    lib.hstu_attn_noalloc_last_device_status.argtypes = [P]
    lib.hstu_attn_noalloc_last_device_status.restype = ctypes.c_int
    # q, paged_kv, num_pages, page_ids, page_indptrs, out, cu_q, cu_k, B, T_q, H, D, dtype,
    # max_q, max_k, alpha, scaling_seqlen, workspace, bytes, stream
    lib.hstu_attn_fwd_paged.argtypes = [CTen, P, i64, P, P, Ten, P, P, i32, i64, i32, i32,
                                        ctypes.c_int, i32, i32, f32, i32, P, S, P]
    lib.hstu_attn_fwd_paged.restype = ctypes.c_int
    # the window pair of the regular calls replaced by func, func_n, func_len
    fscal = scal[:12] + [P, i32, i64] + scal[14:]
    lib.hstu_attn_fwd_func.argtypes = [CTen, CTen, CTen, Ten] + fscal
    lib.hstu_attn_fwd_func.restype = ctypes.c_int
    lib.hstu_attn_bwd_func.argtypes = [CTen, CTen, CTen, CTen, Ten, Ten, Ten] + fscal
    lib.hstu_attn_bwd_func.restype = ctypes.c_int
    lib.hstu_attn_workspace_size_func.argtypes = lib.hstu_attn_workspace_size.argtypes
    lib.hstu_attn_plan_workspace_size.argtypes = [i32, i64, i64, i32, i32, i32, i32]
    lib.hstu_attn_plan_workspace_size.restype = ctypes.c_size_t
    lib.hstu_attn_plan.argtypes = [P, P, i32, i64, i64, i32, i32, i32, i32, i32, i32, P, S, P]
    lib.hstu_attn_plan.restype = ctypes.c_int
    lib.hstu_attn_fwd_planned.argtypes = lib.hstu_attn_fwd.argtypes
    lib.hstu_attn_fwd_planned.restype = ctypes.c_int
    lib.hstu_attn_bwd_planned.argtypes = lib.hstu_attn_bwd.argtypes
    lib.hstu_attn_bwd_planned.restype = ctypes.c_int
    lib.hstu_attn_workspace_size_func.restype = S
    # LMSD (include/hstu_lmsd.h)
    i8p = P
    lib.hstu_lmsd_fwd.argtypes = [P, i64, P, i64, P, P, i64, i32, f32, f32, i32, i32, i32, i64,
                                  P, P, P, i8p, P]
    lib.hstu_lmsd_fwd.restype = ctypes.c_int
    lib.hstu_lmsd_bwd_workspace_size.argtypes = [i64, i32]
    lib.hstu_lmsd_bwd_workspace_size.restype = S
    lib.hstu_lmsd_bwd.argtypes = [P, i64, P, i64, P, i64, P, P, P, P, i8p, i64, i32, f32, i32, i32,
                                  i32, i32, P, i64, P, i64, P, P, P, S, P]
    lib.hstu_lmsd_bwd.restype = ctypes.c_int
    lib.hstu_attn_version.argtypes = []
    lib.hstu_attn_version.restype = i32


def library():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "(no CPU fallback exists)")
            lib = ctypes.CDLL(_LIB_PATH)
            _declare(lib)
            _lib = lib
        return _lib


def workspace_size(batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, max_seqlen_k,
                   is_bwd) -> int:
    n = library().hstu_attn_workspace_size(int(batch), int(total_q), int(total_k),
                                           int(num_heads), int(head_dim), int(max_seqlen_q),
                                           int(max_seqlen_k), int(bool(is_bwd)))
    if n == 0:
        raise ValueError("invalid sizes for hstu_attn_workspace_size")
    return int(n)


def workspace_size_func(batch, total_q, total_k, num_heads, head_dim, max_seqlen_q,
                        max_seqlen_k, is_bwd) -> int:
    """Workspace bytes of a call with an arbitrary (func) mask."""
    n = library().hstu_attn_workspace_size_func(int(batch), int(total_q), int(total_k),
                                                int(num_heads), int(head_dim),
                                                int(max_seqlen_q), int(max_seqlen_k),
                                                int(bool(is_bwd)))
    if n == 0:
        raise ValueError("invalid sizes for hstu_attn_workspace_size_func")
    return int(n)


def plan_workspace_size(batch, total_q, total_k, num_heads, head_dim, max_seqlen_q,
                        max_seqlen_k) -> int:
    """Bytes of a plan (the schedule shared by planned forward and backward calls)."""
    n = library().hstu_attn_plan_workspace_size(int(batch), int(total_q), int(total_k),
                                                int(num_heads), int(head_dim),
                                                int(max_seqlen_q), int(max_seqlen_k))
    if n == 0:
        raise ValueError("invalid sizes for hstu_attn_plan_workspace_size")
    return int(n)


def last_device_status(workspace, stream=None) -> int:
    """Device-side status the last call that used ``workspace`` recorded (syncs)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device).cuda_stream
    return int(library().hstu_attn_last_device_status(workspace.data_ptr(), stream))


def selftest_timeout(workspace, timeout_us: int, stream=None) -> int:
    """Launch the bounded-wait self-test; returns the launch status."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device).cuda_stream
    return int(library().hstu_attn_selftest_timeout(workspace.data_ptr(), int(timeout_us), stream))
