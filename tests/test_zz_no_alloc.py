"""The no-allocation forward entry point against the regular one.

hstu_attn_fwd_noalloc serves callers that cannot allocate device memory when
they call in (for instance an inference-engine plugin that only receives
buffers planned ahead of time), so it keeps its schedule in a fixed array of
the library instead of a caller workspace.  This test calls it through the C
ABI twice in a row and checks each result against hstu_attn_fwd on the same
inputs, within the forward tolerance of the parity tests.  The file is named
so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from generative_recommender_attention_gb300 import _lib as L
from generative_recommender_attention_gb300 import workloads
import generative_recommender_attention_gb300 as hstu

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _noalloc(lib, x, out, causal, alpha, scaling):
    T_q, H, D = x["q"].shape
    B = x["cu_seqlens_q"].shape[0] - 1
    dt = L.HSTU_BF16 if x["q"].dtype == torch.bfloat16 else L.HSTU_FP16
    ten = lambda t: L.CTen(t.data_ptr(), t.stride(0), t.stride(1))  # noqa: E731
    return lib.hstu_attn_fwd_noalloc(
        ten(x["q"]), ten(x["k"]), ten(x["v"]), L.Ten(out.data_ptr(), out.stride(0), out.stride(1)),
        x["cu_seqlens_q"].data_ptr(), x["cu_seqlens_k"].data_ptr(), B, T_q, x["k"].shape[0], H, D,
        dt, x["max_seqlen_q"], x["max_seqlen_k"], float(alpha), int(scaling), -1,
        0 if causal else -1,
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["recsys", "tiny"])
def test_noalloc_matches_regular_forward_twice(name):
    lib = L.library()
    w = workloads.WORKLOADS[name]
    # two different inputs on the two calls: the second must not see the first's schedule
    for seed in (0, 1):
        x = workloads.make_inputs(w, seed=seed)
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        ref = hstu.hstu_attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                                 d["max_seqlen_q"], d["max_seqlen_k"],
                                 scaling_seqlen=w.scaling_seqlen, causal=w.causal, alpha=w.alpha)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(lib, d, out, w.causal, w.alpha, w.scaling_seqlen or 0)
        assert st == 0, L.STATUS.get(st)
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        bound = TOL_FWD * ref.float().abs().max().item()
        assert torch.isfinite(out.float()).all()
        assert err <= bound, (err, bound)


def test_noalloc_rejects_schedules_over_its_limit():
    lib = L.library()
    # 65,529 work units: one more than the 2 MiB array holds; rejected on the host
    fake = L.CTen(0x1000, 64, 64)
    st = lib.hstu_attn_fwd_noalloc(fake, fake, fake, L.Ten(0x1000, 64, 64), 0x2000, 0x2000, 1,
                                   128 * 65528, 128 * 65528, 1, 64, L.HSTU_BF16, 128, 128,
                                   0.125, 0, -1, 0, None)
    assert st == 1
