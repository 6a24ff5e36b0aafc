"""HSTU attention fp64 CPU oracle (Python entry points).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The CUDA
library never imports, links or calls it, and this package shares no code with
the CUDA path.

The arithmetic lives in ``hstu_oracle.c`` (plain C, fp64, optional OpenMP);
this module only builds it, widens the caller's bf16/fp16 tensors to fp64
exactly, and marshals arguments.  ``naive.py`` holds a pure-Python restatement
used as a brute-force check on tiny inputs.

Method ("HSTU Attention (Blackwell SM100/SM103)", Overview): per packed
sequence and head, O = (1/L_scale) (M (.) SiLU(alpha Q K^T)) V, no softmax.
``scaling_seqlen`` None or 0 means max_seqlen_q (same page, Overview and
"High-level functions").  The mask argument ``causal`` of every entry point is
either a bool (True: window (-1, 0), False: window (-1, -1)) or a window pair
(left, right) as in the page's section "Mask support", -1 meaning unbounded,
or ``{"func": F}`` for the arbitrary mask of the same section: F an int32
array (N, L), N odd, whose column t holds query token t's endpoints
F0, F1, ..., valid keys [0, F0) U [F1, F2) U ... (local key indices).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hstu_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libhstu_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libhstu_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c99", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the oracle still works, single-threaded.
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        common = [i64, i64, i32, f64, f64, i32, i32, P, i32, i64, P, P, i64]
        lib.hstu_oracle_fwd_rows.argtypes = [P, P, P, P, P] + common + [P, i32]
        lib.hstu_oracle_dq_rows.argtypes = [P, P, P, P, P, P] + common + [P, i32]
        lib.hstu_oracle_dkdv_rows.argtypes = [P, P, P, P, P, P] + common + [P, P, i32]
        lib.hstu_oracle_threads.argtypes = [i32]
        for f in (lib.hstu_oracle_fwd_rows, lib.hstu_oracle_dq_rows,
                  lib.hstu_oracle_dkdv_rows, lib.hstu_oracle_threads):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def threads(n: int = 0) -> int:
    """Set (n > 0) and return the OpenMP thread count the oracle uses."""
    return int(_load().hstu_oracle_threads(int(n)))


def _f64(x) -> np.ndarray:
    """Exact widening of a (T, H, D) tensor/array to contiguous fp64 numpy."""
    if hasattr(x, "detach"):  # torch tensor: bf16/fp16 -> fp64 is exact
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def resolve_scaling(scaling_seqlen, max_seqlen_q) -> float:
    """L_scale: ``scaling_seqlen`` when positive, else ``max_seqlen_q``."""
    if scaling_seqlen is None or int(scaling_seqlen) == 0:
        return float(max_seqlen_q)
    if int(scaling_seqlen) < 0:
        raise ValueError("scaling_seqlen must be positive")
    return float(scaling_seqlen)


def _func(mask):
    """(pointer-keeping array, N, L) of an arbitrary mask, or (None, 0, 0)."""
    if isinstance(mask, dict):
        f = _i32(mask["func"])
        if f.ndim == 3:
            f = f[0]
        if f.ndim != 2 or f.shape[0] % 2 != 1:
            raise ValueError("func: (N, L) int32 endpoints with N odd")
        f = np.ascontiguousarray(f)
        return f, int(f.shape[0]), int(f.shape[1])
    return None, 0, 0


def _mask_args(mask):
    """C arguments (left, right, func, func_n, func_len) of a mask; the
    array is returned too so that it stays alive during the call."""
    f, n, L = _func(mask)
    left, right = window(mask)
    return (left, right, _ptr(f) if f is not None else None, n, L), f


def window(mask):
    """(left, right) of a mask given as a bool (causal / full) or a pair;
    an arbitrary (func) mask has no window: (-1, -1)."""
    if isinstance(mask, dict):
        return -1, -1
    if isinstance(mask, (tuple, list)):
        left, right = (int(x) for x in mask)
        if left < -1 or right < -1:
            raise ValueError("window bounds are -1 (none) or >= 0")
        return left, right
    return (-1, 0) if bool(mask) else (-1, -1)


def _rows_all(T: int, H: int):
    tok = np.repeat(np.arange(T, dtype=np.int64), H)
    head = np.tile(np.arange(H, dtype=np.int64), T)
    return tok, head


def fwd_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale, causal,
             tokens, heads, n_threads: int = 0) -> np.ndarray:
    """O[tokens[r], heads[r], :] for each r, shape (n, D), fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    hd = np.ascontiguousarray(heads, dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    out = np.zeros((tok.shape[0], D), dtype=np.float64)
    margs, keep = _mask_args(causal)
    _load().hstu_oracle_fwd_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck), cq.shape[0] - 1, H, D,
        float(alpha), float(L_scale), *margs, _ptr(tok), _ptr(hd),
        tok.shape[0], _ptr(out), int(n_threads))
    del keep
    return out


def dq_rows(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale, causal,
            tokens, heads, n_threads: int = 0) -> np.ndarray:
    """dQ[tokens[r], heads[r], :] for each r, shape (n, D), fp64."""
    do, q, k, v = _f64(dout), _f64(q), _f64(k), _f64(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    hd = np.ascontiguousarray(heads, dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    out = np.zeros((tok.shape[0], D), dtype=np.float64)
    margs, keep = _mask_args(causal)
    _load().hstu_oracle_dq_rows(
        _ptr(do), _ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck),
        cq.shape[0] - 1, H, D, float(alpha), float(L_scale),
        *margs, _ptr(tok), _ptr(hd), tok.shape[0], _ptr(out),
        int(n_threads))
    del keep
    return out


def dkdv_rows(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale,
              causal, tokens, heads, n_threads: int = 0):
    """(dK, dV) rows at key-side (tokens[r], heads[r]), each (n, D), fp64."""
    do, q, k, v = _f64(dout), _f64(q), _f64(k), _f64(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    tok = np.ascontiguousarray(tokens, dtype=np.int64)
    hd = np.ascontiguousarray(heads, dtype=np.int64)
    H, D = k.shape[1], k.shape[2]
    dk = np.zeros((tok.shape[0], D), dtype=np.float64)
    dv = np.zeros((tok.shape[0], D), dtype=np.float64)
    margs, keep = _mask_args(causal)
    _load().hstu_oracle_dkdv_rows(
        _ptr(do), _ptr(q), _ptr(k), _ptr(v), _ptr(cq), _ptr(ck),
        cq.shape[0] - 1, H, D, float(alpha), float(L_scale),
        *margs, _ptr(tok), _ptr(hd), tok.shape[0], _ptr(dk),
        _ptr(dv), int(n_threads))
    del keep
    return dk, dv


def fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale, causal,
        n_threads: int = 0) -> np.ndarray:
    """Full O, shape (T_q, H, D), fp64."""
    T, H, D = q.shape
    tok, hd = _rows_all(T, H)
    return fwd_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale,
                    causal, tok, hd, n_threads).reshape(T, H, D)


def gather_paged(paged_kv, page_ids, page_indptrs, cu_seqlens_k):
    """Contiguous (T_k, H, D) K and V of a paged cache ("HSTU Attention
    (Blackwell SM100/SM103)", Mask support: paged_kv is (num_pages, 2, 128,
    H, D), K/V selected by the second index; page_ids[page_indptrs[b] + p] is
    the page holding keys 128 p .. 128 p + 127 of sequence b).  Key j of
    sequence b lands at row cu_seqlens_k[b] + j.  Values are copied, exactly."""
    kv = _f64(paged_kv)
    ids, ptr, ck = _i32(page_ids), _i32(page_indptrs), _i32(cu_seqlens_k)
    T = int(ck[-1])
    H, D = kv.shape[3], kv.shape[4]
    k = np.zeros((T, H, D))
    v = np.zeros((T, H, D))
    for b in range(ck.shape[0] - 1):
        for j in range(int(ck[b + 1] - ck[b])):
            page = int(ids[int(ptr[b]) + j // 128])
            k[ck[b] + j] = kv[page, 0, j % 128]
            v[ck[b] + j] = kv[page, 1, j % 128]
    return k, v


def fwd_paged(q, paged_kv, page_ids, page_indptrs, cu_seqlens_q, cu_seqlens_k, alpha,
              L_scale, n_threads: int = 0) -> np.ndarray:
    """Forward over a paged K/V cache, causal (the page's paged path is causal
    only): the keys are gathered into contiguous storage and the ordinary
    forward runs on them."""
    k, v = gather_paged(paged_kv, page_ids, page_indptrs, cu_seqlens_k)
    return fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale, True, n_threads)


def bwd(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale, causal,
        n_threads: int = 0):
    """Full (dQ, dK, dV), shapes of q, k, v, fp64."""
    Tq, H, D = q.shape
    Tk = k.shape[0]
    tq, hq = _rows_all(Tq, H)
    tk, hk = _rows_all(Tk, H)
    dq = dq_rows(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, alpha, L_scale,
                 causal, tq, hq, n_threads).reshape(Tq, H, D)
    dk, dv = dkdv_rows(dout, q, k, v, cu_seqlens_q, cu_seqlens_k, alpha,
                       L_scale, causal, tk, hk, n_threads)
    return dq, dk.reshape(Tk, H, D), dv.reshape(Tk, H, D)
