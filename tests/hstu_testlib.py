"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same 16-bit inputs, compare.

Tolerance (fixed for this operation): max |gpu - ref| over a whole tensor
must be at most 1e-2 * max |ref| for the forward output and 2e-2 * max |ref|
for each of dQ, dK, dV.
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
