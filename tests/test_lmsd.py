"""GPU parity of the LMSD kernels (through the C ABI via the binding) against
the fp64 oracle (oracle/lmsd.py) on the same bf16 inputs.

Tolerances: every output segment and gradient within 1e-2 * max |ref| of that
tensor (bf16 outputs, fp32 arithmetic); mean and rstd within 1e-5 relative;
the dropout mask bit for bit (both sides draw the same Philox words and
compare them with the same integer threshold)."""
import numpy as np
import pytest
import torch

from oracle import lmsd as ref
from generative_recommender_attention_gb300 import lmsd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _inputs(n, d, seed, pad=0):
    g = torch.Generator().manual_seed(seed)
    xs = (torch.randn(n, d + pad, generator=g) * 1.5 + 0.3).to(torch.bfloat16)
    us = torch.randn(n, d + 2 * pad, generator=g).to(torch.bfloat16)
    w = torch.randn(d, generator=g).to(torch.bfloat16)
    b = torch.randn(d, generator=g).to(torch.bfloat16)
    return xs[:, :d], us[:, :d], w, b


def _close(name, got, want, tol=1e-2):
    g = got.detach().float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), name
    err, mx = float(np.abs(g - want).max()), float(np.abs(want).max())
    assert err <= tol * mx + 1e-6, f"{name}: {err:.3e} > {tol} * {mx:.3e}"


CASES = [(257, 128, 0), (1000, 64, 8), (33, 1016, 0), (100, 8, 0), (64, 520, 8), (3, 256, 0)]


@pytest.mark.parametrize("n,d,pad", CASES)
@pytest.mark.parametrize("flags", [(True, True, True), (False, False, False), (True, True, False)])
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_lmsd_forward_backward(n, d, pad, flags, p):
    silu, cu, cx = flags
    x, u, w, b = _inputs(n, d, seed=n + d, pad=pad)
    xd, ud, wd, bd = (t.cuda() for t in (x, u, w, b))
    if pad:   # padded row strides, as the page allows for x and u
        xd = torch.empty(n, d + pad, dtype=torch.bfloat16, device="cuda")[:, :d]
        xd.copy_(x)
        ud = torch.empty(n, d + 2 * pad, dtype=torch.bfloat16, device="cuda")[:, :d]
        ud.copy_(u)
    out = lmsd.hstu_lmsd_forward(xd, ud, wd, bd, eps=1e-5, dropout_ratio=p, seed=17 + n,
                                 apply_u_silu=silu, concat_u=cu, concat_x=cx)
    torch.cuda.synchronize()
    y, mean, rstd, mask = ref.forward(x, u, w, b, 1e-5, p, 17 + n, silu, cu, cx)
    assert out["y_tensor"].shape == y.shape
    S = y.shape[1] // d
    for k in range(S):
        _close(f"y segment {k}", out["y_tensor"][:, k * d:(k + 1) * d], y[:, k * d:(k + 1) * d])
    np.testing.assert_allclose(out["mean_tensor"].cpu().numpy(), mean, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(out["rstd_tensor"].cpu().numpy(), rstd, rtol=1e-5)
    if p == 0:
        assert out["mask_tensor"] is None
    else:
        np.testing.assert_array_equal(out["mask_tensor"].cpu().numpy(), mask)
    dy = torch.randn(y.shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    g = lmsd.hstu_lmsd_backward(dy.cuda(), xd, ud, wd, bd, out["mean_tensor"], out["rstd_tensor"],
                                out["mask_tensor"], dropout_ratio=p, apply_u_silu=silu,
                                concat_u=cu, concat_x=cx)
    torch.cuda.synchronize()
    dx, du, dw, db = ref.backward(dy.double(), x, u, w, b, mean, rstd, mask, p, silu, cu, cx)
    _close("dx", g["dx_tensor"], dx, 2e-2)
    _close("du", g["du_tensor"], du, 2e-2)
    _close("dweight", g["dweight_tensor"], dw, 2e-2)
    _close("dbias", g["dbias_tensor"], db, 2e-2)


def test_lmsd_backward_deterministic_and_dweight_optional():
    n, d = 5000, 256
    x, u, w, b = (t.cuda() for t in _inputs(n, d, seed=3))
    out = lmsd.hstu_lmsd_forward(x, u, w, b, dropout_ratio=0.2, seed=9)
    dy = torch.randn_like(out["y_tensor"])
    args = (dy, x, u, w, b, out["mean_tensor"], out["rstd_tensor"], out["mask_tensor"])
    g1 = lmsd.hstu_lmsd_backward(*args, dropout_ratio=0.2)
    g2 = lmsd.hstu_lmsd_backward(*args, dropout_ratio=0.2)
    g3 = lmsd.hstu_lmsd_backward(*args, dropout_ratio=0.2, compute_dweight=False)
    torch.cuda.synchronize()
    for k in ("dx_tensor", "du_tensor", "dweight_tensor", "dbias_tensor"):
        assert torch.equal(g1[k], g2[k])
    assert g3["dweight_tensor"] is None and torch.equal(g3["dbias_tensor"], g1["dbias_tensor"])
    # the same seed draws the same mask; another seed another one
    o2 = lmsd.hstu_lmsd_forward(x, u, w, b, dropout_ratio=0.2, seed=9)
    o3 = lmsd.hstu_lmsd_forward(x, u, w, b, dropout_ratio=0.2, seed=10)
    torch.cuda.synchronize()
    assert torch.equal(o2["mask_tensor"], out["mask_tensor"])
    assert not torch.equal(o3["mask_tensor"], out["mask_tensor"])


@pytest.mark.parametrize("n,d,pad", [(257, 128, 8), (100, 1016, 16), (64, 256, 24)])
def test_lmsd_backward_padded_dy_and_outputs(n, d, pad):
    # dy may have a row stride larger than S * D, and dx / du row strides
    # larger than D ("Tensor shapes and layouts"): the gradients are the same
    # bit for bit as with contiguous tensors, and match the oracle.
    p = 0.1
    x, u, w, b = _inputs(n, d, seed=2 * n + d)
    xd, ud, wd, bd = (t.cuda() for t in (x, u, w, b))
    out = lmsd.hstu_lmsd_forward(xd, ud, wd, bd, eps=1e-5, dropout_ratio=p, seed=3 + n)
    y = out["y_tensor"]
    dy = torch.randn(y.shape, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    dy_pad = torch.empty(y.shape[0], y.shape[1] + pad, dtype=torch.bfloat16,
                         device="cuda")[:, :y.shape[1]]
    dy_pad.copy_(dy)
    assert dy_pad.stride(0) == y.shape[1] + pad
    dx_pad = torch.empty(n, d + pad, dtype=torch.bfloat16, device="cuda")[:, :d]
    du_pad = torch.empty(n, d + 2 * pad, dtype=torch.bfloat16, device="cuda")[:, :d]
    rest = (xd, ud, wd, bd, out["mean_tensor"], out["rstd_tensor"], out["mask_tensor"])
    g0 = lmsd.hstu_lmsd_backward(dy.cuda(), *rest, dropout_ratio=p)
    g1 = lmsd.hstu_lmsd_backward(dy_pad, *rest, dropout_ratio=p, dx=dx_pad, du=du_pad)
    torch.cuda.synchronize()
    for k in ("dx_tensor", "du_tensor", "dweight_tensor", "dbias_tensor"):
        assert torch.equal(g0[k], g1[k]), k
    _, mean, rstd, mask = ref.forward(x, u, w, b, 1e-5, p, 3 + n, True, True, True)
    dx, du, dw, db = ref.backward(dy.double(), x, u, w, b, mean, rstd, mask, p, True, True, True)
    _close("dx", g1["dx_tensor"], dx, 2e-2)
    _close("du", g1["du_tensor"], du, 2e-2)
    _close("dweight", g1["dweight_tensor"], dw, 2e-2)
    _close("dbias", g1["dbias_tensor"], db, 2e-2)
