"""HSTU LayerNorm-Multiply-SiLU-Dropout (LMSD): plain fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only the tests, the
smoke check and the benchmark's CPU legs may use it; it shares no code with
the CUDA library.

What it computes (page "HSTU LayerNorm-Multiply-SiLU-Dropout (LMSD)",
Overview), for every row of x (N, D):
    xhat = (x - mean(x)) rstd(x),  rstd = 1 / sqrt(var(x) + eps)  (biased var)
    l    = xhat * weight + bias
    a    = SiLU(u) if apply_u_silu else u
    y    = [dropout(a) if concat_u, dropout(x) if concat_x, dropout(l * a)]
Inverted dropout keeps an element with probability 1 - p and scales it by
1 / (1 - p).  The int8 mask holds one bit per segment: bit 0 the mandatory
l * a result, bit 1 the x segment, bit 2 the activated-u segment; a set bit
means kept; disabled segments leave their bits clear; p = 0 keeps everything
and returns no mask.

The random decisions come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC 2011), written here from
that definition.  The pages do not say how counters map to elements; the
reading taken here (and in the CUDA library, written separately): one
Philox call decides 8 elements.  The element at flat index e = row * D + col
of segment k (0 main, 1 x, 2 u) uses the 16-bit half e % 2 (0 = low) of
output word (e % 8) // 2 of Philox(counter = (g mod 2^32, g >> 32, k, 0),
key = (seed mod 2^32, (seed >> 32) mod 2^32)) with g = e // 8, and is kept
iff that half >= floor(p * 2^16) (p taken as fp32, then exactly).

Backward (chain rule of the forward; the page gives the API, not the
formulas): with s_k = mask bit k / (1 - p) (1 when p = 0),
    dm  = dy_main s_0;   dl = dm a;   da = dm l + (dy_u s_2 if concat_u)
    du  = da SiLU'(u) if apply_u_silu else da
    dxh = dl * weight
    dx  = rstd (dxh - mean(dxh) - xhat mean(dxh xhat)) + (dy_x s_1 if concat_x)
    dweight = sum_rows dl xhat,  dbias = sum_rows dl.
"""
from __future__ import annotations

import numpy as np

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)   # round multipliers
_W0, _W1 = np.uint64(0x9E3779B9), np.uint64(0xBB67AE85)   # key (Weyl) increments
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on uint32 counter words (arrays) and a key;
    returns the four output words as uint64 arrays holding 32-bit values."""
    c = [np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3)]
    k0, k1 = np.uint64(int(k0) & 0xFFFFFFFF), np.uint64(int(k1) & 0xFFFFFFFF)
    for r in range(10):
        p0 = _M0 * c[0]               # < 2^64: both factors are below 2^32
        p1 = _M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        if r < 9:
            k0 = (k0 + _W0) & _MASK32
            k1 = (k1 + _W1) & _MASK32
    return c


def keep_halves(n, d, segment, seed):
    """The 16-bit Philox half deciding each element of an (n, d) segment."""
    e = np.arange(n * d, dtype=np.uint64)
    g = e // np.uint64(8)
    s = int(seed) & 0xFFFFFFFFFFFFFFFF
    words = philox4x32_10(g & _MASK32, g >> np.uint64(32), np.full_like(g, segment),
                          np.zeros_like(g), s & 0xFFFFFFFF, s >> 32)
    word = np.choose(((e % np.uint64(8)) // np.uint64(2)).astype(np.int64), words)
    half = (word >> (np.uint64(16) * (e % np.uint64(2)))) & np.uint64(0xFFFF)
    return half.reshape(n, d)


def threshold(p):
    """Keep iff half >= floor(p * 2^16), with p rounded to fp32 first."""
    return int(np.floor(float(np.float32(p)) * 65536.0))


def _silu(u):
    return u / (1.0 + np.exp(-u))


def _silu_grad(u):
    s = 1.0 / (1.0 + np.exp(-u))
    return s * (1.0 + u * (1.0 - s))


def _f64(t):
    if hasattr(t, "detach"):
        t = t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def forward(x, u, weight, bias, eps, dropout_ratio, seed, apply_u_silu=True, concat_u=True,
            concat_x=True):
    """Returns (y, mean, rstd, mask) with y (N, S*D) fp64, mean/rstd (N,),
    mask int8 (N, D) or None when dropout_ratio == 0."""
    x, u, w, b = _f64(x), _f64(u), _f64(weight), _f64(bias)
    n, d = x.shape
    mean = x.mean(axis=1)
    var = ((x - mean[:, None]) ** 2).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    ell = xhat * w + b
    a = _silu(u) if apply_u_silu else u
    p = float(np.float32(dropout_ratio))
    segs = []
    mask = None
    if p > 0.0:
        t = threshold(p)
        scale = 1.0 / (1.0 - p)
        keep = {k: keep_halves(n, d, k, seed) >= np.uint64(t) for k in (0, 1, 2)}
        mask = keep[0].astype(np.int8)
        if concat_x:
            mask |= (keep[1].astype(np.int8) << 1)
        if concat_u:
            mask |= (keep[2].astype(np.int8) << 2)
        drop = lambda v, k: np.where(keep[k], v * scale, 0.0)  # noqa: E731
    else:
        drop = lambda v, k: v  # noqa: E731
    if concat_u:
        segs.append(drop(a, 2))
    if concat_x:
        segs.append(drop(x, 1))
    segs.append(drop(ell * a, 0))
    return np.concatenate(segs, axis=1), mean, rstd, mask


def backward(dy, x, u, weight, bias, mean, rstd, mask, dropout_ratio, apply_u_silu=True,
             concat_u=True, concat_x=True):
    """Returns (dx, du, dweight, dbias), fp64."""
    dy, x, u, w, b = _f64(dy), _f64(x), _f64(u), _f64(weight), _f64(bias)
    mean, rstd = _f64(mean), _f64(rstd)
    n, d = x.shape
    p = float(np.float32(dropout_ratio))
    if p > 0.0:
        m = np.asarray(mask.detach().cpu().numpy() if hasattr(mask, "detach") else mask)
        m = m.astype(np.int64)
        s = [((m >> k) & 1) / (1.0 - p) for k in (0, 1, 2)]
    else:
        s = [np.ones((n, d))] * 3
    seg = 0
    dy_u = dy_x = None
    if concat_u:
        dy_u = dy[:, seg * d:(seg + 1) * d]
        seg += 1
    if concat_x:
        dy_x = dy[:, seg * d:(seg + 1) * d]
        seg += 1
    dy_m = dy[:, seg * d:(seg + 1) * d]
    xhat = (x - mean[:, None]) * rstd[:, None]
    ell = xhat * w + b
    a = _silu(u) if apply_u_silu else u
    dm = dy_m * s[0]
    dl = dm * a
    da = dm * ell + (dy_u * s[2] if concat_u else 0.0)
    du = da * _silu_grad(u) if apply_u_silu else da
    dxh = dl * w
    dx = rstd[:, None] * (dxh - dxh.mean(axis=1, keepdims=True)
                          - xhat * (dxh * xhat).mean(axis=1, keepdims=True))
    if concat_x:
        dx = dx + dy_x * s[1]
    return dx, du, (dl * xhat).sum(axis=0), dl.sum(axis=0)
