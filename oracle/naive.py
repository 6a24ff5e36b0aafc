"""Pure-Python brute force of HSTU attention, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It restates the
forward equations of "HSTU Attention (Blackwell SM100/SM103)", Overview, and
the chain-rule backward, one scalar at a time, with Python floats and
``math.exp``.  It is used to brute-force check the C oracle's indexing
(packed offsets, heads, masks) on inputs of a few tokens; it uses no numpy
arithmetic, no C and nothing from the C oracle.

Inputs are nested Python lists indexed [t][h][d]; cu_seqlens are lists of
ints.  ``causal`` is True for the top-left aligned causal mask (key j valid
iff j <= i and j < Lk), False for the full mask (j < Lk), or a window pair
(left, right): key j valid iff j < Lk, i - left <= j unless left == -1, and
j <= i + right unless right == -1; or {"func": F} with F a list of N rows
(N odd) of per-query-token endpoints: key j valid for query token t iff
j < Lk and j lies in [0, F[0][t]) or in one of [F[1][t], F[2][t]),
[F[3][t], F[4][t]), ...
"""
from __future__ import annotations

import math


def _sigma(x: float) -> float:
    if x < -700.0:
        return 0.0
    return 1.0 / (1.0 + math.exp(-x))


def _silu(x: float) -> float:
    return x * _sigma(x)


def _silu_grad(x: float) -> float:
    s = _sigma(x)
    return s * (1.0 + x * (1.0 - s))


def _zeros(T, H, D):
    return [[[0.0] * D for _ in range(H)] for _ in range(T)]


def _valid(i, j, Lk, causal, t=None):
    if j >= Lk:
        return False
    if isinstance(causal, dict):
        F = causal["func"]
        if j < F[0][t]:
            return True
        return any(F[m][t] <= j < F[m + 1][t] for m in range(1, len(F) - 1, 2))
    if isinstance(causal, (tuple, list)):
        left, right = causal
        lo_ok = left == -1 or i - j <= left
        hi_ok = right == -1 or j - i <= right
        return lo_ok and hi_ok
    return not causal or j <= i


def forward(q, k, v, cu_q, cu_k, alpha, L_scale, causal):
    T, H, D = len(q), len(q[0]), len(q[0][0])
    out = _zeros(T, H, D)
    for b in range(len(cu_q) - 1):
        oq, ok = cu_q[b], cu_k[b]
        Lq, Lk = cu_q[b + 1] - oq, cu_k[b + 1] - ok
        for h in range(H):
            for i in range(Lq):
                for j in range(Lk):
                    if not _valid(i, j, Lk, causal, oq + i):
                        continue
                    s = 0.0
                    for d in range(D):
                        s += q[oq + i][h][d] * k[ok + j][h][d]
                    a = _silu(alpha * s) / L_scale
                    for d in range(D):
                        out[oq + i][h][d] += a * v[ok + j][h][d]
    return out


def backward(dout, q, k, v, cu_q, cu_k, alpha, L_scale, causal):
    Tq, H, D = len(q), len(q[0]), len(q[0][0])
    Tk = len(k)
    dq, dk, dv = _zeros(Tq, H, D), _zeros(Tk, H, D), _zeros(Tk, H, D)
    for b in range(len(cu_q) - 1):
        oq, ok = cu_q[b], cu_k[b]
        Lq, Lk = cu_q[b + 1] - oq, cu_k[b + 1] - ok
        for h in range(H):
            for i in range(Lq):
                for j in range(Lk):
                    if not _valid(i, j, Lk, causal, oq + i):
                        continue
                    s = 0.0
                    da = 0.0
                    for d in range(D):
                        s += q[oq + i][h][d] * k[ok + j][h][d]
                        da += dout[oq + i][h][d] * v[ok + j][h][d]
                    x = alpha * s
                    a = _silu(x) / L_scale
                    ds = da * _silu_grad(x) / L_scale
                    for d in range(D):
                        dv[ok + j][h][d] += a * dout[oq + i][h][d]
                        dq[oq + i][h][d] += alpha * ds * k[ok + j][h][d]
                        dk[ok + j][h][d] += alpha * ds * q[oq + i][h][d]
    return dq, dk, dv
