"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same 16-bit inputs, compare.

Tolerance (fixed for this operation): max |gpu - ref| over a tensor must be
at most 1e-2 * max |ref| for the forward output and 2e-2 * max |ref| for
each of dQ, dK, dV.  When only sampled rows are checked, max |ref| is taken
over the sample, which can only make the bound tighter.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import generative_recommender_attention_gb300 as hstu

TOL_FWD = 1e-2
TOL_BWD = 2e-2


def to_dev(x, device="cuda"):
    out = {}
    for k, v in x.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def mask_kwargs(causal):
    """Binding keywords of a mask given as a bool, a (left, right) window or
    {"func": (N, L) int32 endpoints} (an arbitrary mask)."""
    if isinstance(causal, dict):
        f = torch.as_tensor(np.ascontiguousarray(causal["func"]), dtype=torch.int32)
        return {"func": f[None].contiguous().cuda()}
    if isinstance(causal, tuple):
        return {"window_size": causal}
    return {"causal": bool(causal)}


def gpu_fwd_bwd(xd, scaling, causal, alpha, **kw):
    o = hstu.hstu_attn_fwd(xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"], xd["cu_seqlens_k"],
                           xd["max_seqlen_q"], xd["max_seqlen_k"], scaling_seqlen=scaling,
                           alpha=alpha, **mask_kwargs(causal), **kw.get("fwd", {}))
    dq, dk, dv = hstu.hstu_attn_bwd(xd["do"], xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"],
                                    xd["cu_seqlens_k"], xd["max_seqlen_q"], xd["max_seqlen_k"],
                                    scaling_seqlen=scaling, alpha=alpha, **mask_kwargs(causal),
                                    **kw.get("bwd", {}))
    torch.cuda.synchronize()
    return o, dq, dk, dv


def max_err(got: torch.Tensor, ref: np.ndarray):
    g = got.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "non-finite values in GPU output"
    return float(np.max(np.abs(g - ref))) if ref.size else 0.0, float(np.max(np.abs(ref))) if ref.size else 0.0


def check(name, got, ref, tol):
    err, mx = max_err(got, ref)
    bound = tol * mx
    assert err <= bound or (mx == 0.0 and err == 0.0), \
        f"{name}: max abs err {err:.3e} > {tol} * max|ref| = {bound:.3e}"
    return err, mx


def full_compare(x, scaling, causal, alpha, n_threads=0):
    """Full fwd+bwd on the GPU vs the full oracle."""
    L = oracle.resolve_scaling(scaling, x["max_seqlen_q"])
    xd = to_dev(x)
    o, dq, dk, dv = gpu_fwd_bwd(xd, scaling, causal, alpha)
    ro = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], alpha, L,
                    causal, n_threads)
    rdq, rdk, rdv = oracle.bwd(x["do"], x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                               x["cu_seqlens_k"], alpha, L, causal, n_threads)
    res = {"o": check("O", o, ro, TOL_FWD), "dq": check("dQ", dq, rdq, TOL_BWD),
           "dk": check("dK", dk, rdk, TOL_BWD), "dv": check("dV", dv, rdv, TOL_BWD)}
    return res


def sample_rows(cu: torch.Tensor, H: int, n_random: int, seed: int):
    """(token, head) pairs covering sequence starts and ends, tile boundaries
    and random rows, for sampled comparisons at full size."""
    rng = np.random.default_rng(seed)
    c = cu.tolist()
    B = len(c) - 1
    toks = []
    nonempty = [b for b in range(B) if c[b + 1] > c[b]]
    pick = nonempty[:3] + nonempty[-3:] + list(rng.choice(nonempty, size=min(6, len(nonempty)),
                                                             replace=False))
    for b in pick:
        L = c[b + 1] - c[b]
        for i in (0, 1, 63, 64, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1):
            if 0 <= i < L:
                toks.append(c[b] + i)
    T = c[-1]
    if T > 0:
        toks += list(rng.integers(0, T, size=n_random))
    toks = np.array(sorted(set(int(t) for t in toks)), dtype=np.int64)
    heads = rng.integers(0, H, size=toks.shape[0]).astype(np.int64)
    return toks, heads


def sampled_compare(x, scaling, causal, alpha, n_random=160, seed=0, gpu_out=None):
    """Full-size GPU fwd+bwd, checked on sampled rows against the oracle."""
    L = oracle.resolve_scaling(scaling, x["max_seqlen_q"])
    if gpu_out is None:
        xd = to_dev(x)
        gpu_out = gpu_fwd_bwd(xd, scaling, causal, alpha)
    o, dq, dk, dv = gpu_out
    H = x["q"].shape[1]
    tq, hq = sample_rows(x["cu_seqlens_q"], H, n_random, seed)
    tk, hk = sample_rows(x["cu_seqlens_k"], H, n_random, seed + 1)
    args = (x["cu_seqlens_q"], x["cu_seqlens_k"], alpha, L, causal)
    ro = oracle.fwd_rows(x["q"], x["k"], x["v"], *args, tq, hq)
    rdq = oracle.dq_rows(x["do"], x["q"], x["k"], x["v"], *args, tq, hq)
    rdk, rdv = oracle.dkdv_rows(x["do"], x["q"], x["k"], x["v"], *args, tk, hk)
    tqt, hqt = torch.from_numpy(tq), torch.from_numpy(hq)
    tkt, hkt = torch.from_numpy(tk), torch.from_numpy(hk)
    sel = lambda t, a, b: t.cpu()[a, b]  # noqa: E731
    return {"o": check("O", sel(o, tqt, hqt), ro, TOL_FWD),
            "dq": check("dQ", sel(dq, tqt, hqt), rdq, TOL_BWD),
            "dk": check("dK", sel(dk, tkt, hkt), rdk, TOL_BWD),
            "dv": check("dV", sel(dv, tkt, hkt), rdv, TOL_BWD)}
