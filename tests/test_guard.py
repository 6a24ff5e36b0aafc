"""Out-of-bounds write guard (stands in for a memory checker).

Outputs live inside sentinel-filled buffers: a padded head stride and token
stride leave gaps between logical elements, extra rows follow the last
sequence, and guard rows sit before and after the tensor.  After the forward
and backward calls, every byte outside the logical outputs must still hold the
sentinel, and every logical element must have been written."""
import numpy as np
import pytest
import torch

from generative_recommender_attention_gb300 import workloads
import generative_recommender_attention_gb300 as hstu

from hstu_testlib import mask_kwargs

pytestmark = pytest.mark.gpu

SENT = -3072.0   # exactly representable in bf16 and fp16; no output reaches it


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _guarded(T, H, D, dtype, extra_rows=3, pad_h=8, pad_t=16, guard=64):
    """A (T + extra_rows, H, D) view with padded strides inside a sentinel buffer."""
    sh = D + pad_h
    st = H * sh + pad_t
    n = guard + (T + extra_rows) * st + guard
    buf = torch.full((n,), SENT, dtype=dtype, device="cuda")
    view = buf[guard:guard + (T + extra_rows) * st].as_strided((T + extra_rows, H, D), (st, sh, 1))
    mask = torch.zeros(n, dtype=torch.bool, device="cuda")
    mview = mask[guard:guard + (T + extra_rows) * st].as_strided((T + extra_rows, H, D), (st, sh, 1))
    mview[:T] = True      # logical elements of the real rows
    return buf, view, mask


@pytest.mark.parametrize("D,dtype,causal", [(64, torch.bfloat16, True), (128, torch.float16, False),
                                            (256, torch.bfloat16, True),
                                            (128, torch.bfloat16, (100, 20)),
                                            (32, torch.float16, True), (128, torch.bfloat16, "func")])
def test_no_write_outside_logical_outputs(D, dtype, causal):
    lens = [129, 1, 300, 0, 64]
    H = 2
    T = sum(lens)
    x = workloads.random_inputs(lens, lens, H, D, dtype, seed=D)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    # inputs get the 3 extra rows too (T_q = T + 3 with cu[B] = T): rows past cu[B]
    # belong to no sequence and must never be written
    pad = lambda t: torch.cat([t, torch.zeros(3, H, D, dtype=dtype, device="cuda")])  # noqa
    q, k, v, do = pad(dev["q"]), pad(dev["k"]), pad(dev["v"]), pad(dev["do"])
    bufs = [_guarded(T, H, D, dtype) for _ in range(4)]
    if causal == "func":  # causal plus the last 5 keys of each sequence
        i = np.concatenate([np.arange(L) for L in lens] + [np.zeros(3, np.int64)])
        lk = np.concatenate([np.full(L, L) for L in lens] + [np.zeros(3, np.int64)])
        causal = {"func": np.stack([i + 1, lk - 5, lk]).astype(np.int32)}
    mk = mask_kwargs(causal)
    o = hstu.hstu_attn_fwd(q, k, v, dev["cu_seqlens_q"], dev["cu_seqlens_k"], 300, 300,
                           alpha=0.1, out=bufs[0][1], **mk)
    hstu.hstu_attn_bwd(do, q, k, v, dev["cu_seqlens_q"], dev["cu_seqlens_k"], 300, 300,
                       alpha=0.1, dq=bufs[1][1], dk=bufs[2][1], dv=bufs[3][1], **mk)
    torch.cuda.synchronize()
    for name, (buf, view, mask) in zip(("out", "dq", "dk", "dv"), bufs):
        outside = buf[~mask]
        assert torch.all(outside == SENT), f"{name}: {int((outside != SENT).sum())} bytes outside written"
        inside = buf[mask]
        assert torch.all(inside != SENT) and torch.isfinite(inside.float()).all(), \
            f"{name}: logical element not written"
    assert o.data_ptr() == bufs[0][1].data_ptr()
