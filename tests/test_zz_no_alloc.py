"""The no-allocation forward entry point against the regular one.

hstu_attn_fwd_noalloc serves callers that cannot allocate device memory when
they call in (for instance an inference-engine plugin that only receives
buffers planned ahead of time), so it keeps its schedule in a fixed array of
the library instead of a caller workspace.  These tests call it through the C
ABI twice in a row, on batches of different shapes, and check each result
against hstu_attn_fwd on the same inputs within the forward tolerance of the
parity tests; that the device's free memory and torch's reserved memory do
not move across repeated calls; and that its device-side status query
reports success after good calls and bad metadata after a bad one.  The file
is named so that pytest collects it last.
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


def _check_against_regular(lib, x, w, causal=None):
    causal = w.causal if causal is None else causal
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    ref = hstu.hstu_attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                             d["max_seqlen_q"], d["max_seqlen_k"],
                             scaling_seqlen=w.scaling_seqlen, causal=causal, alpha=w.alpha)
    out = torch.full_like(ref, float("nan"))
    st = _noalloc(lib, d, out, causal, w.alpha, w.scaling_seqlen or 0)
    assert st == 0, L.STATUS.get(st)
    torch.cuda.synchronize()
    assert lib.hstu_attn_noalloc_last_device_status(torch.cuda.current_stream().cuda_stream) == 0
    err = (out.float() - ref.float()).abs().max().item()
    bound = TOL_FWD * ref.float().abs().max().item()
    assert torch.isfinite(out.float()).all()
    assert err <= bound, (err, bound)


@pytest.mark.parametrize("name", ["recsys", "tiny"])
def test_noalloc_matches_regular_forward_twice(name):
    lib = L.library()
    w = workloads.WORKLOADS[name]
    # two different inputs on the two calls: the second must not see the first's schedule
    for seed in (0, 1):
        _check_against_regular(lib, workloads.make_inputs(w, seed=seed), w)


def test_noalloc_second_call_of_another_shape():
    """A call with more work units, then one with fewer, another head count
    and head dimension and the full mask: a stale header or unit counter left
    by the first call would show in the second's output or status."""
    lib = L.library()
    w = workloads.WORKLOADS["recsys"]
    _check_against_regular(lib, workloads.make_inputs(w, seed=2), w)
    x = workloads.random_inputs([300, 1, 129, 517, 64], [300, 1, 129, 517, 64], 2, 64,
                                torch.float16, seed=3)
    import dataclasses
    w2 = dataclasses.replace(w, heads=2, head_dim=64, alpha=0.125, scaling_seqlen=None,
                             causal=False)
    _check_against_regular(lib, x, w2, causal=False)


def test_noalloc_allocates_nothing():
    """After a first call (which looks the array's address up), repeated
    calls leave the device's free memory and torch's reserved memory as they
    were."""
    lib = L.library()
    w = workloads.WORKLOADS["recsys"]
    x = workloads.make_inputs(w, seed=4)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = torch.empty_like(d["q"])
    assert _noalloc(lib, d, out, True, w.alpha, 0) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(5):
        assert _noalloc(lib, d, out, True, w.alpha, 0) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_reserved() == reserved0


def test_noalloc_status_reports_bad_metadata():
    """cu_seqlens that run past total_q: the scheduler drops the units past
    the schedule's capacity (nothing is read or written past the tensors) and
    the status query says so; a good call afterwards reports success again."""
    lib = L.library()
    H, D, T = 2, 64, 256
    q = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    cu = torch.tensor([0, 128, 100000], dtype=torch.int32, device="cuda")
    x = {"q": q, "k": q, "v": q, "cu_seqlens_q": cu, "cu_seqlens_k": cu,
         "max_seqlen_q": 128, "max_seqlen_k": 128}
    assert _noalloc(lib, x, out, True, 0.125, 0) == 0
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.hstu_attn_noalloc_last_device_status(stream) == 1   # HSTU_ERR_INVALID_ARG
    w = workloads.WORKLOADS["tiny"]
    _check_against_regular(lib, workloads.make_inputs(w, seed=0), w)


def test_noalloc_rejects_schedules_over_its_limit():
    lib = L.library()
    # 65,529 work units: one more than the 2 MiB array holds; rejected on the host
    fake = L.CTen(0x1000, 64, 64)
    st = lib.hstu_attn_fwd_noalloc(fake, fake, fake, L.Ten(0x1000, 64, 64), 0x2000, 0x2000, 1,
                                   128 * 65528, 128 * 65528, 1, 64, L.HSTU_BF16, 128, 128,
                                   0.125, 0, -1, 0, None)
    assert st == 1
