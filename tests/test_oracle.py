"""Pins for the fp64 CPU oracle.

The pages print no numeric results for HSTU attention, so the oracle is pinned
to mathematics it does not share code with:

* a hand-worked example with exact closed-form outputs (tests/golden);
* brute force: a pure-Python scalar restatement on tiny inputs;
* closed forms: length-1 sequences, Q = 0 (SiLU(0) = 0, SiLU'(0) = 1/2),
  V = 0, K = 0;
* special cases that reduce to a library matmul: scores far above zero make
  SiLU the identity (linear attention), scores far below zero make it zero;
* invariants: linearity in V and dO, O proportional to 1/L_scale, causal rows
  blind to future keys, causal row i equal to the full mask on the prefix,
  packing invariance, head independence;
* gradients: central finite differences of <dO, O>, and torch.autograd on a
  dense masked fp64 formulation built from torch primitives;
* limits: no NaN at |score| = 1e4;
* arbitrary masks ("Mask support", func_tensor): brute force with random
  endpoints, the func masks that equal causal, full and window masks, and
  inclusion-exclusion over a union of two intervals;
* windows ("Mask support", window_size = (left, right)): brute force with
  random windows, the degenerate windows that equal the causal and full
  masks, the diagonal-only window (0, 0) in closed form, the band built with
  numpy's tril/triu in the linear regime, band additivity, finite
  differences and autograd with a band mask.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a wrong mask offset) fails it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import naive
from generative_recommender_attention_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(lq, lk, H, D, seed, std=1.0, dtype=torch.float64):
    r = workloads.random_inputs(lq, lk, H, D, torch.float32, seed, std)
    return {k: (v.to(dtype) if isinstance(v, torch.Tensor) and v.is_floating_point() else v)
            for k, v in r.items()}


def _fwd(x, alpha, L, causal):
    return oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                      alpha, L, causal)


def _bwd(x, alpha, L, causal):
    return oracle.bwd(x["do"], x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                      x["cu_seqlens_k"], alpha, L, causal)


def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"L3": math.log(3.0)}))


# --------------------------------------------------------------------------
# hand-worked closed form
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["causal", "full"])
def test_hand_worked_example(case):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_ln3.json")))
    inp = g["inputs"]
    t = {n: torch.tensor(inp[n], dtype=torch.float64) for n in ("q", "k", "v", "do")}
    cu = torch.tensor(inp["cu_seqlens"], dtype=torch.int32)
    alpha = _eval(inp["alpha"])
    L = float(inp["scaling_seqlen"])
    causal = case == "causal"
    exp = g["cases"][case]
    o = oracle.fwd(t["q"], t["k"], t["v"], cu, cu, alpha, L, causal)
    dq, dk, dv = oracle.bwd(t["do"], t["q"], t["k"], t["v"], cu, cu, alpha, L, causal)
    for name, got in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        want = np.vectorize(_eval)(np.array(exp[name], dtype=object)).astype(np.float64)
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14, err_msg=name)


# --------------------------------------------------------------------------
# brute force vs pure-Python restatement
# --------------------------------------------------------------------------
WINDOWS = [(0, 0), (2, 1), (3, -1), (-1, 2), (1, 0), (0, 3)]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [True, False] + WINDOWS)
def test_brute_force_tiny(seed, causal):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    lq = [int(x) for x in rng.integers(0, 9, size=B)]
    # q lengths <= k lengths per sequence, k sometimes longer
    lk = [L + int(rng.integers(0, 3)) * (seed % 2) for L in lq]
    H, D = int(rng.integers(1, 3)), int(rng.integers(1, 9))
    x = _rand(lq, lk, H, D, seed)
    alpha = float(rng.uniform(-1.5, 1.5))
    L = float(rng.integers(1, 12))
    o = _fwd(x, alpha, L, causal)
    dq, dk, dv = _bwd(x, alpha, L, causal)
    lst = {k: x[k].tolist() for k in ("q", "k", "v", "do")}
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    o_n = np.array(naive.forward(lst["q"], lst["k"], lst["v"], cq, ck, alpha, L, causal))
    dq_n, dk_n, dv_n = (np.array(a) for a in
                        naive.backward(lst["do"], lst["q"], lst["k"], lst["v"], cq, ck,
                                       alpha, L, causal))
    for got, want in ((o, o_n), (dq, dq_n), (dk, dk_n), (dv, dv_n)):
        np.testing.assert_allclose(got.reshape(want.shape), want, rtol=1e-12, atol=1e-12)


def test_tiny_workload_matches_brute_force():
    """The 4-sequence tiny workload (lengths 17, 64, 100, 128) on one head."""
    w = workloads.WORKLOADS["tiny"]
    x = workloads.make_inputs(w, seed=0)
    # restrict to head 0 and D = 8 to keep the pure-Python loops quick
    q, k, v, do = (x[n][:, :1, :8].double() for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens_q"]
    o = oracle.fwd(q, k, v, cu, cu, w.alpha, 128.0, True)
    o_n = np.array(naive.forward(q.tolist(), k.tolist(), v.tolist(), cu.tolist(),
                                 cu.tolist(), w.alpha, 128.0, True))
    np.testing.assert_allclose(o, o_n, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def _silu(x):
    return x / (1.0 + np.exp(-x))


def _silu_grad(x):
    s = 1.0 / (1.0 + np.exp(-x))
    return s * (1.0 + x * (1.0 - s))


def test_length_one_sequences():
    lens = [1, 1, 1, 1, 1]
    x = _rand(lens, lens, 3, 7, seed=11)
    alpha, L = 0.7, 3.0
    o = _fwd(x, alpha, L, True)
    dq, dk, dv = _bwd(x, alpha, L, True)
    q, k, v, do = (x[n].numpy() for n in ("q", "k", "v", "do"))
    s = alpha * np.einsum("thd,thd->th", q, k)
    np.testing.assert_allclose(o, (_silu(s) / L)[..., None] * v, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dv, (_silu(s) / L)[..., None] * do, rtol=1e-13, atol=1e-15)
    da = np.einsum("thd,thd->th", do, v)
    ds = da * _silu_grad(s) / L
    np.testing.assert_allclose(dq, alpha * ds[..., None] * k, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dk, alpha * ds[..., None] * q, rtol=1e-12, atol=1e-15)


def _dense_mask(Lq, Lk, causal):
    """Dense 0/1 mask: bool (causal / full) by index comparison; a window
    (left, right) as a band from numpy's tril (j <= i + right) and triu
    (j >= i - left)."""
    if isinstance(causal, tuple):
        left, right = causal
        m = np.ones((Lq, Lk))
        if right >= 0:
            m = np.tril(m, right)
        if left >= 0:
            m = np.triu(m, -left)
        return m
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    m = j < Lk
    if causal:
        m = m & (j <= i)
    return m.astype(np.float64)


@pytest.mark.parametrize("causal", [True, False])
def test_q_zero(causal):
    """Q = 0: SiLU(0) = 0 gives O = dV = dK = 0; SiLU'(0) = 1/2 gives
    dQ = (alpha / 2L) (M (.) dO V^T) K."""
    lens = [5, 9, 3]
    x = _rand(lens, lens, 2, 6, seed=3)
    x["q"] = torch.zeros_like(x["q"])
    alpha, L = 1.3, 4.0
    o = _fwd(x, alpha, L, causal)
    dq, dk, dv = _bwd(x, alpha, L, causal)
    assert np.all(o == 0) and np.all(dk == 0) and np.all(dv == 0)
    cu = x["cu_seqlens_q"].tolist()
    for b in range(len(lens)):
        s0, s1 = cu[b], cu[b + 1]
        for h in range(2):
            do = x["do"][s0:s1, h].numpy()
            v = x["v"][s0:s1, h].numpy()
            k = x["k"][s0:s1, h].numpy()
            M = _dense_mask(s1 - s0, s1 - s0, causal)
            want = alpha / (2 * L) * (M * (do @ v.T)) @ k
            np.testing.assert_allclose(dq[s0:s1, h], want, rtol=1e-12, atol=1e-14)


def test_v_zero_and_k_zero():
    lens = [6, 4]
    x = _rand(lens, lens, 2, 5, seed=5)
    alpha, L = 0.9, 6.0
    xv = dict(x, v=torch.zeros_like(x["v"]))
    o = _fwd(xv, alpha, L, True)
    dq, dk, dv = _bwd(xv, alpha, L, True)
    assert np.all(o == 0) and np.all(dq == 0) and np.all(dk == 0)
    assert np.any(dv != 0)
    xk = dict(x, k=torch.zeros_like(x["k"]))
    o = _fwd(xk, alpha, L, True)
    dq, dk, dv = _bwd(xk, alpha, L, True)
    assert np.all(o == 0) and np.all(dq == 0) and np.all(dv == 0)


# --------------------------------------------------------------------------
# special cases reducing to a library matmul
# --------------------------------------------------------------------------
def _aligned_inputs(lens, H, D, sign, seed):
    """q_i = c u + small noise, k_j = sign (c u + small noise): every score is
    about sign * alpha * c^2 = +/-40 or beyond."""
    rng = np.random.default_rng(seed)
    T = sum(lens)
    u = np.ones(D) / math.sqrt(D)
    c = 8.0
    q = c * u + 0.05 * rng.standard_normal((T, H, D))
    k = sign * (c * u + 0.05 * rng.standard_normal((T, H, D)))
    v = rng.standard_normal((T, H, D))
    do = rng.standard_normal((T, H, D))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return {n: torch.tensor(a) for n, a in (("q", q), ("k", k), ("v", v), ("do", do))}, cu


@pytest.mark.parametrize("causal", [True, False, (2, 1), (0, 0), (4, -1), (-1, 3)])
def test_linear_regime_matches_matmul(causal):
    """Scores >= 40: sigma = 1 to fp64 precision, SiLU(x) = x and SiLU'(x) = 1,
    so HSTU is masked linear attention, computed here with numpy matmuls."""
    lens = [7, 12, 3]
    H, D = 2, 8
    t, cu = _aligned_inputs(lens, H, D, +1.0, seed=1)
    alpha, L = 0.7, 5.0
    o = oracle.fwd(t["q"], t["k"], t["v"], cu, cu, alpha, L, causal)
    dq, dk, dv = oracle.bwd(t["do"], t["q"], t["k"], t["v"], cu, cu, alpha, L, causal)
    c = cu.tolist()
    for b in range(len(lens)):
        s0, s1 = c[b], c[b + 1]
        for h in range(H):
            q, k, v, do = (t[n][s0:s1, h].numpy() for n in ("q", "k", "v", "do"))
            S = alpha * q @ k.T
            assert S.min() > 36.0
            M = _dense_mask(s1 - s0, s1 - s0, causal)
            A = M * S / L
            np.testing.assert_allclose(o[s0:s1, h], A @ v, rtol=1e-12)
            np.testing.assert_allclose(dv[s0:s1, h], A.T @ do, rtol=1e-12)
            dS = M * (do @ v.T) / L
            np.testing.assert_allclose(dq[s0:s1, h], alpha * dS @ k, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(dk[s0:s1, h], alpha * dS.T @ q, rtol=1e-11, atol=1e-12)


def test_negative_regime_is_zero():
    lens = [9, 4]
    t, cu = _aligned_inputs(lens, 1, 8, -1.0, seed=2)
    o = oracle.fwd(t["q"], t["k"], t["v"], cu, cu, 2.0, 3.0, False)
    assert np.abs(o).max() < 1e-20


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_linearity_in_v_and_do():
    lens = [8, 5]
    x = _rand(lens, lens, 2, 6, seed=7)
    y = _rand(lens, lens, 2, 6, seed=8)
    alpha, L = 0.8, 7.0
    a, b = 1.7, -0.6
    xv = dict(x, v=a * x["v"] + b * y["v"])
    np.testing.assert_allclose(
        _fwd(xv, alpha, L, True),
        a * _fwd(x, alpha, L, True) + b * _fwd(dict(x, v=y["v"]), alpha, L, True),
        rtol=1e-12, atol=1e-13)
    xd = dict(x, do=a * x["do"] + b * y["do"])
    g = _bwd(xd, alpha, L, True)
    g1 = _bwd(x, alpha, L, True)
    g2 = _bwd(dict(x, do=y["do"]), alpha, L, True)
    for u, w1, w2 in zip(g, g1, g2):
        np.testing.assert_allclose(u, a * w1 + b * w2, rtol=1e-12, atol=1e-13)


def test_inverse_proportional_to_scaling():
    lens = [6, 10]
    x = _rand(lens, lens, 1, 4, seed=9)
    o1 = _fwd(x, 0.5, 1.0, True)
    o7 = _fwd(x, 0.5, 7.0, True)
    np.testing.assert_allclose(o7 * 7.0, o1, rtol=1e-13)


def test_causal_rows_ignore_future_keys():
    lens = [10]
    x = _rand(lens, lens, 2, 5, seed=12)
    o = _fwd(x, 0.9, 3.0, True)
    y = dict(x)
    y["k"] = x["k"].clone()
    y["v"] = x["v"].clone()
    y["k"][6:] += 3.0
    y["v"][6:] -= 2.0
    o2 = _fwd(y, 0.9, 3.0, True)
    np.testing.assert_array_equal(o[:6], o2[:6])
    assert np.abs(o[6:] - o2[6:]).max() > 1e-3


def test_causal_row_equals_full_on_prefix():
    L = 9
    x = _rand([L], [L], 2, 4, seed=13)
    o = _fwd(x, 1.1, 5.0, True)
    for i in range(L):
        cu = torch.tensor([0, i + 1], dtype=torch.int32)
        of = oracle.fwd(x["q"][: i + 1], x["k"][: i + 1], x["v"][: i + 1], cu, cu,
                        1.1, 5.0, False)
        np.testing.assert_allclose(o[i], of[i], rtol=1e-13, atol=1e-15)


def test_packing_invariance():
    lens = [4, 0, 7, 3]
    x = _rand(lens, lens, 2, 5, seed=14)
    o = _fwd(x, 0.6, 4.0, True)
    g = _bwd(x, 0.6, 4.0, True)
    cu = x["cu_seqlens_q"].tolist()
    for b in range(len(lens)):
        s0, s1 = cu[b], cu[b + 1]
        if s1 == s0:
            continue
        c1 = torch.tensor([0, s1 - s0], dtype=torch.int32)
        sub = {n: x[n][s0:s1] for n in ("q", "k", "v", "do")}
        np.testing.assert_array_equal(
            o[s0:s1], oracle.fwd(sub["q"], sub["k"], sub["v"], c1, c1, 0.6, 4.0, True))
        gs = oracle.bwd(sub["do"], sub["q"], sub["k"], sub["v"], c1, c1, 0.6, 4.0, True)
        for a, bb in zip(g, gs):
            np.testing.assert_array_equal(a[s0:s1], bb)


def test_heads_independent():
    lens = [5, 6]
    x = _rand(lens, lens, 3, 4, seed=15)
    perm = [2, 0, 1]
    o = _fwd(x, 0.7, 2.0, True)
    xp = {n: (x[n][:, perm] if n in ("q", "k", "v", "do") else x[n]) for n in x}
    op = _fwd(xp, 0.7, 2.0, True)
    np.testing.assert_array_equal(o[:, perm], op)


# --------------------------------------------------------------------------
# gradients
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False, (1, 1), (2, -1)])
def test_finite_differences(causal):
    lens = [4, 3]
    lk = [5, 3]
    x = _rand(lens, lk, 2, 3, seed=21)
    alpha, L = 0.9, 3.0
    dq, dk, dv = _bwd(x, alpha, L, causal)
    do = x["do"].numpy()
    rng = np.random.default_rng(0)
    eps = 1e-6

    def loss(y):
        return float(np.sum(_fwd(y, alpha, L, causal) * do))

    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        for _ in range(8):
            idx = tuple(int(rng.integers(0, s)) for s in x[name].shape)
            p = x[name].clone()
            p[idx] += eps
            m = x[name].clone()
            m[idx] -= eps
            fd = (loss(dict(x, **{name: p})) - loss(dict(x, **{name: m}))) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7 + 1e-6 * abs(fd), (name, idx, fd, grad[idx])


def test_adjoint_identity_on_q():
    lens = [6, 5]
    x = _rand(lens, lens, 2, 4, seed=22)
    alpha, L = 1.2, 4.0
    dq, _, _ = _bwd(x, alpha, L, True)
    rng = np.random.default_rng(1)
    dQ = torch.tensor(rng.standard_normal(x["q"].shape))
    eps = 1e-6
    do = x["do"].numpy()
    fp = np.sum(_fwd(dict(x, q=x["q"] + eps * dQ), alpha, L, True) * do)
    fm = np.sum(_fwd(dict(x, q=x["q"] - eps * dQ), alpha, L, True) * do)
    assert abs((fp - fm) / (2 * eps) - np.sum(dq * dQ.numpy())) < 1e-6


@pytest.mark.parametrize("causal", [True, False, (2, 1), (0, 0), (-1, 2)])
def test_torch_autograd_dense(causal):
    """Dense masked fp64 formulation built from torch primitives
    (torch.nn.functional.silu, matmul), differentiated by autograd."""
    lens_q = [5, 8, 1]
    lens_k = [7, 8, 2]
    H, D = 2, 6
    x = _rand(lens_q, lens_k, H, D, seed=31)
    alpha, L = 0.75, 6.0
    o = _fwd(x, alpha, L, causal)
    dq, dk, dv = _bwd(x, alpha, L, causal)
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    for b in range(len(lens_q)):
        q = x["q"][cq[b]:cq[b + 1]].clone().requires_grad_(True)
        k = x["k"][ck[b]:ck[b + 1]].clone().requires_grad_(True)
        v = x["v"][ck[b]:ck[b + 1]].clone().requires_grad_(True)
        do = x["do"][cq[b]:cq[b + 1]]
        M = torch.tensor(_dense_mask(q.shape[0], k.shape[0], causal))
        S = alpha * torch.einsum("ihd,jhd->hij", q, k)
        A = torch.nn.functional.silu(S) * M / L
        O = torch.einsum("hij,jhd->ihd", A, v)
        (O * do).sum().backward()
        np.testing.assert_allclose(o[cq[b]:cq[b + 1]], O.detach().numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dq[cq[b]:cq[b + 1]], q.grad.numpy(), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dk[ck[b]:ck[b + 1]], k.grad.numpy(), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dv[ck[b]:ck[b + 1]], v.grad.numpy(), rtol=1e-11, atol=1e-13)


# --------------------------------------------------------------------------
# windows
# --------------------------------------------------------------------------
def test_degenerate_windows_equal_causal_and_full():
    """(-1, 0) is causal and (-1, -1) full; bounds at least as long as every
    sequence remove nothing on their side."""
    lq, lk = [9, 1, 14, 0, 6], [9, 3, 16, 2, 6]
    x = _rand(lq, lk, 2, 5, seed=41)
    alpha, L = 0.8, 7.0
    big = 40
    pairs = [((-1, 0), True), ((-1, -1), False), ((big, 0), True), ((big, big), False),
             ((big, -1), False), ((-1, big), False)]
    for win, ref in pairs:
        np.testing.assert_array_equal(_fwd(x, alpha, L, win), _fwd(x, alpha, L, ref))
        for g, h in zip(_bwd(x, alpha, L, win), _bwd(x, alpha, L, ref)):
            np.testing.assert_array_equal(g, h)


def test_diagonal_window_closed_form():
    """Window (0, 0) keeps only key j = i: O_i = SiLU(x_ii) v_i / L,
    dV_i = SiLU(x_ii) dO_i / L, dQ_i = alpha SiLU'(x_ii) <dO_i, v_i> k_i / L,
    dK_i = alpha SiLU'(x_ii) <dO_i, v_i> q_i / L (rows past the other side's
    length get nothing)."""
    lq, lk = [5, 7, 2], [6, 4, 2]
    H, D = 2, 4
    x = _rand(lq, lk, H, D, seed=42)
    alpha, L = 1.1, 3.0
    o = _fwd(x, alpha, L, (0, 0))
    dq, dk, dv = _bwd(x, alpha, L, (0, 0))
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    for b in range(len(lq)):
        n = min(lq[b], lk[b])
        qs, ks = slice(cq[b], cq[b] + n), slice(ck[b], ck[b] + n)
        q, k, v, do = x["q"][qs].numpy(), x["k"][ks].numpy(), x["v"][ks].numpy(), x["do"][qs].numpy()
        s = alpha * np.sum(q * k, axis=-1)
        da = np.sum(do * v, axis=-1)
        np.testing.assert_allclose(o[qs], _silu(s)[..., None] * v / L, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dv[ks], _silu(s)[..., None] * do / L, rtol=1e-12, atol=1e-15)
        g = alpha * _silu_grad(s) * da / L
        np.testing.assert_allclose(dq[qs], g[..., None] * k, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dk[ks], g[..., None] * q, rtol=1e-12, atol=1e-15)
        assert np.all(o[cq[b] + n:cq[b + 1]] == 0) and np.all(dq[cq[b] + n:cq[b + 1]] == 0)
        assert np.all(dk[ck[b] + n:ck[b + 1]] == 0) and np.all(dv[ck[b] + n:ck[b + 1]] == 0)


@pytest.mark.parametrize("left,right", [(0, 2), (3, 1), (2, 4)])
def test_band_additivity(left, right):
    """Every output is a sum of per-pair terms over the valid pairs, so the
    pairs that a right bound adds past the diagonal are the same with or
    without a left bound: F(l, r) - F(l, 0) = F(-1, r) - F(-1, 0)."""
    lens = [10, 13]
    x = _rand(lens, lens, 2, 4, seed=43)
    alpha, L = 0.6, 5.0
    f = lambda w: [_fwd(x, alpha, L, w)] + list(_bwd(x, alpha, L, w))  # noqa: E731
    a, b, c, d = f((left, right)), f((left, 0)), f((-1, right)), f((-1, 0))
    for ta, tb, tc, td in zip(a, b, c, d):
        np.testing.assert_allclose(ta - tb, tc - td, rtol=1e-11, atol=1e-13)
    # and the band really excludes something on each side
    assert np.abs(a[0] - f((-1, -1))[0]).max() > 1e-3


# --------------------------------------------------------------------------
# arbitrary (func) masks
# --------------------------------------------------------------------------
def _local_rows(x):
    """Local query index and its sequence's key count for every query token."""
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    T = cq[-1]
    i = np.zeros(T, np.int64)
    lk = np.zeros(T, np.int64)
    for b in range(len(cq) - 1):
        i[cq[b]:cq[b + 1]] = np.arange(cq[b + 1] - cq[b])
        lk[cq[b]:cq[b + 1]] = ck[b + 1] - ck[b]
    return i, lk


def _func(*rows):
    return {"func": np.stack([np.asarray(r, dtype=np.int32) for r in rows])}


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("n", [1, 3, 5])
def test_func_brute_force_tiny(seed, n):
    """Random endpoints (overlapping, unordered, negative, past the
    sequence) against the pure-Python restatement."""
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 4))
    lq = [int(v) for v in rng.integers(0, 9, size=B)]
    lk = [L + int(rng.integers(0, 3)) for L in lq]
    H, D = int(rng.integers(1, 3)), int(rng.integers(1, 6))
    x = _rand(lq, lk, H, D, seed)
    T = sum(lq)
    F = rng.integers(-2, 12, size=(n, T + 3)).astype(np.int32)
    mask = {"func": F}
    alpha, L = float(rng.uniform(-1.5, 1.5)), float(rng.integers(1, 12))
    o = _fwd(x, alpha, L, mask)
    dq, dk, dv = _bwd(x, alpha, L, mask)
    lst = {k: x[k].tolist() for k in ("q", "k", "v", "do")}
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    nm = {"func": F.tolist()}
    o_n = np.array(naive.forward(lst["q"], lst["k"], lst["v"], cq, ck, alpha, L, nm))
    dq_n, dk_n, dv_n = (np.array(a) for a in
                        naive.backward(lst["do"], lst["q"], lst["k"], lst["v"], cq, ck, alpha, L, nm))
    for got, want in ((o, o_n), (dq, dq_n), (dk, dk_n), (dv, dv_n)):
        np.testing.assert_allclose(got.reshape(want.shape), want, rtol=1e-12, atol=1e-12)


def test_func_masks_that_are_windows():
    """F0 = i + 1 is the causal mask, F0 >= Lk the full mask, and
    [0, 0) U [i - l, i + r + 1) the window (l, r), exactly."""
    lq, lk = [9, 1, 14, 0, 6], [9, 3, 16, 2, 6]
    x = _rand(lq, lk, 2, 5, seed=61)
    i, klen = _local_rows(x)
    alpha, L = 0.8, 7.0
    cases = [(_func(i + 1), True), (_func(klen + 5), False),
             (_func(np.zeros_like(i), i - 2, i + 2), (2, 1)),
             (_func(np.zeros_like(i), np.maximum(0, i - 3), i + 1), (3, 0))]
    for fm, ref in cases:
        np.testing.assert_array_equal(_fwd(x, alpha, L, fm), _fwd(x, alpha, L, ref))
        for g, h in zip(_bwd(x, alpha, L, fm), _bwd(x, alpha, L, ref)):
            np.testing.assert_array_equal(g, h)


def test_func_union_inclusion_exclusion():
    """Outputs are sums over valid pairs, so for A = [0, F0), B = [F1, F2):
    F(A u B) + F(A n B) = F(A) + F(B); and [0, 5) u [3, 8) = [0, 8)."""
    lens = [12, 7, 10]
    x = _rand(lens, lens, 2, 4, seed=62)
    i, klen = _local_rows(x)
    alpha, L = 0.7, 6.0
    f0, f1, f2 = i + 1, np.maximum(0, klen - 4), klen
    zero = np.zeros_like(i)
    masks = [_func(f0, f1, f2), _func(zero, np.maximum(zero, f1), np.minimum(f0, f2)),
             _func(f0), _func(zero, f1, f2)]
    out = [[_fwd(x, alpha, L, m)] + list(_bwd(x, alpha, L, m)) for m in masks]
    for a, b, c, d in zip(*out):
        np.testing.assert_allclose(a + b, c + d, rtol=1e-11, atol=1e-13)
    assert np.abs(out[0][0] - out[2][0]).max() > 1e-3  # B adds keys past the diagonal
    five = np.full_like(i, 5)
    np.testing.assert_array_equal(_fwd(x, alpha, L, _func(five, five - 2, five + 3)),
                                  _fwd(x, alpha, L, _func(five + 3)))


# --------------------------------------------------------------------------
# paged K/V
# --------------------------------------------------------------------------
def test_paged_gather_is_the_contiguous_forward():
    """Keys scattered over shuffled 128-row pages (with unused pages and
    garbage past each sequence's last key) give exactly the forward of the
    contiguous keys; a page holding keys of the wrong offset would not."""
    lens_q, lens_k = [130, 1, 300, 0, 256], [200, 1, 300, 5, 256]
    H, D = 2, 8
    x = _rand(lens_q, lens_k, H, D, seed=51)
    rng = np.random.default_rng(5)
    ck = x["cu_seqlens_k"].tolist()
    n_pages = [-(-L // 128) for L in lens_k]
    total_pages = sum(n_pages) + 3
    perm = rng.permutation(total_pages)
    kv = rng.standard_normal((total_pages, 2, 128, H, D)) * 100.0   # finite garbage
    ids, ptr, used = [], [0], 0
    for b, L in enumerate(lens_k):
        for p in range(n_pages[b]):
            page = int(perm[used]); used += 1
            ids.append(page)
            rows = slice(ck[b] + 128 * p, ck[b] + min(L, 128 * p + 128))
            n = rows.stop - rows.start
            kv[page, 0, :n] = x["k"][rows].numpy()
            kv[page, 1, :n] = x["v"][rows].numpy()
        ptr.append(len(ids))
    alpha, L = 0.7, 9.0
    got = oracle.fwd_paged(x["q"], kv, np.array(ids, np.int32), np.array(ptr, np.int32),
                           x["cu_seqlens_q"], x["cu_seqlens_k"], alpha, L)
    want = _fwd(x, alpha, L, True)
    np.testing.assert_array_equal(got, want)
    # swapping two pages of one sequence changes the result
    ids2 = list(ids)
    ids2[ptr[2]], ids2[ptr[2] + 1] = ids2[ptr[2] + 1], ids2[ptr[2]]
    bad = oracle.fwd_paged(x["q"], kv, np.array(ids2, np.int32), np.array(ptr, np.int32),
                           x["cu_seqlens_q"], x["cu_seqlens_k"], alpha, L)
    assert np.abs(bad - want).max() > 1e-3


# --------------------------------------------------------------------------
# limits, empty and ragged cases, row entry points
# --------------------------------------------------------------------------
def test_huge_scores_no_nan():
    lens = [3]
    q = torch.zeros(3, 1, 2, dtype=torch.float64)
    k = torch.zeros(3, 1, 2, dtype=torch.float64)
    q[:, 0, 0] = 100.0
    k[0, 0, 0] = 1.0
    k[1, 0, 0] = -1.0
    k[2, 0, 0] = 0.5
    v = torch.ones(3, 1, 2, dtype=torch.float64)
    cu = torch.tensor([0, 3], dtype=torch.int32)
    o = oracle.fwd(q, k, v, cu, cu, 100.0, 1.0, False)  # scores +-1e4, 5e3
    dq, dk, dv = oracle.bwd(v, q, k, v, cu, cu, 100.0, 1.0, False)
    for a in (o, dq, dk, dv):
        assert np.all(np.isfinite(a))
    # SiLU(1e4) = 1e4, SiLU(-1e4) = 0, SiLU(5e3) = 5e3
    np.testing.assert_allclose(o[0, 0], [15000.0, 15000.0], rtol=1e-15)


def test_empty_and_keyless_rows():
    lq = [0, 3, 2]
    lk = [0, 3, 0]   # third sequence has queries but no keys -> zero rows
    x = _rand(lq, lk, 1, 4, seed=41)
    o = _fwd(x, 1.0, 2.0, True)
    dq, dk, dv = _bwd(x, 1.0, 2.0, True)
    assert np.all(o[3:5] == 0) and np.all(dq[3:5] == 0)
    assert np.any(o[:3] != 0)


def test_row_entry_points_match_full():
    lens = [9, 14, 2]
    x = _rand(lens, lens, 2, 5, seed=51)
    o = _fwd(x, 0.8, 9.0, True)
    dq, dk, dv = _bwd(x, 0.8, 9.0, True)
    tok = np.array([0, 8, 9, 22, 24, 13])
    hd = np.array([1, 0, 1, 0, 1, 0])
    np.testing.assert_array_equal(
        oracle.fwd_rows(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                        0.8, 9.0, True, tok, hd), o[tok, hd])
    r = oracle.dq_rows(x["do"], x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                       x["cu_seqlens_k"], 0.8, 9.0, True, tok, hd)
    np.testing.assert_array_equal(r, dq[tok, hd])
    rk, rv = oracle.dkdv_rows(x["do"], x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                              x["cu_seqlens_k"], 0.8, 9.0, True, tok, hd)
    np.testing.assert_array_equal(rk, dk[tok, hd])
    np.testing.assert_array_equal(rv, dv[tok, hd])


def test_resolve_scaling():
    assert oracle.resolve_scaling(None, 37) == 37.0
    assert oracle.resolve_scaling(0, 37) == 37.0
    assert oracle.resolve_scaling(5, 37) == 5.0
    with pytest.raises(ValueError):
        oracle.resolve_scaling(-1, 37)
