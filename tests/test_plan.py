"""GPU tests of plans (hstu_attn_plan + the planned forward and backward):
one scheduling launch shared by any number of calls on one batch layout.

A planned call must give the unplanned call's results bit for bit (the
kernels and their per-unit arithmetic are the same; only who builds the work
lists differs), the unplanned results are held to the oracle elsewhere, and
one case here is checked against the oracle directly.  A plan must survive
reuse (each kernel leaves its unit counter at zero for the next call) and a
call whose sizes differ from the plan's must write nothing and report
HSTU_ERR_INVALID_ARG on the device."""
import math

import pytest
import torch

import oracle
from generative_recommender_attention_gb300 import workloads
import generative_recommender_attention_gb300 as hstu

from hstu_testlib import TOL_BWD, TOL_FWD, check, to_dev

pytestmark = pytest.mark.gpu

LENS = [300, 1, 129, 517, 0, 64, 256, 1000]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _mask(window):
    return {"causal": True} if window == "causal" else \
        {"causal": False} if window == "full" else {"window_size": window}


def _calls(xd, D, mask, plan=None):
    alpha = 1.0 / math.sqrt(D)
    T_q, T_k = xd["q"].shape[0], xd["k"].shape[0]
    kw = dict(alpha=alpha, **_mask(mask))
    o = hstu.hstu_attn_fwd(xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"], xd["cu_seqlens_k"],
                           xd["max_seqlen_q"], xd["max_seqlen_k"], plan=plan, **kw)
    g = hstu.hstu_attn_bwd(xd["do"], xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"],
                           xd["cu_seqlens_k"], xd["max_seqlen_q"], xd["max_seqlen_k"], plan=plan,
                           **kw)
    return (o,) + tuple(g)


def _plan(xd, H, D, mask, workspace=None, max_q=None):
    mq = xd["max_seqlen_q"] if max_q is None else max_q
    mk = xd["max_seqlen_k"] if max_q is None else max(max_q, xd["max_seqlen_k"])
    return hstu.hstu_attn_plan(xd["cu_seqlens_q"], xd["cu_seqlens_k"], xd["q"].shape[0],
                               xd["k"].shape[0], H, D, mq, mk, workspace=workspace, **_mask(mask))


@pytest.mark.parametrize("D,dtype,mask", [(128, torch.bfloat16, "causal"),
                                          (64, torch.float16, (64, 32)),
                                          (256, torch.float16, "full"),
                                          (32, torch.bfloat16, "causal"),
                                          (128, torch.float16, (200, 0))])
def test_planned_equals_unplanned(D, dtype, mask):
    x = workloads.random_inputs(LENS, LENS, 2, D, dtype, seed=D)
    xd = to_dev(x)
    ref = _calls(xd, D, mask)
    p = _plan(xd, 2, D, mask)
    got = _calls(xd, D, mask, plan=p)
    torch.cuda.synchronize()
    assert hstu.last_device_status(p.workspace) == 0
    for name, a, b in zip(("O", "dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name


def test_planned_against_oracle():
    D = 128
    x = workloads.random_inputs(LENS, LENS, 2, D, torch.bfloat16, seed=11)
    xd = to_dev(x)
    p = _plan(xd, 2, D, "causal")
    o, dq, dk, dv = _calls(xd, D, "causal", plan=p)
    torch.cuda.synchronize()
    alpha, L = 1.0 / math.sqrt(D), x["max_seqlen_q"]
    ro = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], alpha, L, True)
    rdq, rdk, rdv = oracle.bwd(x["do"], x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                               x["cu_seqlens_k"], alpha, L, True)
    check("O", o, ro, TOL_FWD)
    check("dQ", dq, rdq, TOL_BWD)
    check("dK", dk, rdk, TOL_BWD)
    check("dV", dv, rdv, TOL_BWD)


def test_plan_serves_many_calls():
    """One plan, several forwards and backwards in stream order (as the
    layers of a model would use it), on different inputs of one layout."""
    D = 64
    xs = [to_dev(workloads.random_inputs(LENS, LENS, 2, D, torch.bfloat16, seed=s))
          for s in range(3)]
    p = _plan(xs[0], 2, D, "causal")
    got = [_calls(xd, D, "causal", plan=p) for xd in xs + xs[:1]]
    ref = [_calls(xd, D, "causal") for xd in xs + xs[:1]]
    torch.cuda.synchronize()
    assert hstu.last_device_status(p.workspace) == 0
    for g, r in zip(got, ref):
        for a, b in zip(g, r):
            assert torch.equal(a, b)


def test_plan_of_other_sizes_is_refused_on_the_device():
    """A call whose sizes differ from the plan's (here max_seqlen_q) writes
    nothing and records HSTU_ERR_INVALID_ARG; a new plan then works."""
    D, H = 64, 2
    x = workloads.random_inputs(LENS, LENS, H, D, torch.bfloat16, seed=5)
    xd = to_dev(x)
    T = xd["q"].shape[0]
    mq = xd["max_seqlen_q"]
    big = hstu.plan_workspace_size(len(LENS), T, T, H, D, mq + 64, mq + 64)
    ws = torch.empty(big, dtype=torch.uint8, device="cuda")
    p = _plan(xd, H, D, "causal", workspace=ws)  # made for max_seqlen_q = mq
    forged = hstu.HstuPlan(ws, (len(LENS), T, T, H, D, mq + 64, mq + 64, (-1, 0)))
    out = torch.full_like(xd["q"], 7.0)
    hstu.hstu_attn_fwd(xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"], xd["cu_seqlens_k"],
                       mq + 64, mq + 64, alpha=0.125, out=out, plan=forged)
    torch.cuda.synchronize()
    assert hstu.last_device_status(ws) == 1
    assert torch.all(out == 7.0)
    p = _plan(xd, H, D, "causal", workspace=ws)
    ref = _calls(xd, D, "causal")
    got = _calls(xd, D, "causal", plan=p)
    torch.cuda.synchronize()
    assert hstu.last_device_status(ws) == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_planned_recsys_workload_equals_unplanned():
    w = workloads.WORKLOADS["recsys"]
    xd = to_dev(workloads.make_inputs(w, seed=0))
    kw = dict(alpha=w.alpha, scaling_seqlen=w.scaling_seqlen, causal=True)
    T = xd["q"].shape[0]
    p = hstu.hstu_attn_plan(xd["cu_seqlens_q"], xd["cu_seqlens_k"], T, T, w.heads, w.head_dim,
                            xd["max_seqlen_q"], xd["max_seqlen_k"])
    args = (xd["cu_seqlens_q"], xd["cu_seqlens_k"], xd["max_seqlen_q"], xd["max_seqlen_k"])
    for plan in (None, p):
        o = hstu.hstu_attn_fwd(xd["q"], xd["k"], xd["v"], *args, plan=plan, **kw)
        g = hstu.hstu_attn_bwd(xd["do"], xd["q"], xd["k"], xd["v"], *args, plan=plan, **kw)
        if plan is None:
            ref = (o,) + tuple(g)
    torch.cuda.synchronize()
    for a, b in zip((o,) + tuple(g), ref):
        assert torch.equal(a, b)
