"""Failure detection without a GPU fault.

Every barrier wait in the kernels is bounded.  The self-test kernel waits on a
barrier that nothing completes, with a short limit; it must give up, record
HSTU_ERR_DEVICE_TIMEOUT in the workspace and return, leaving the context
usable.  No trap, no fault, no hang."""
import time

import pytest
import torch

from generative_recommender_attention_gb300 import workloads
import generative_recommender_attention_gb300 as hstu

pytestmark = pytest.mark.gpu

TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    t0 = time.time()
    assert hstu.selftest_timeout(ws, 200_000) == 0          # 0.2 s limit
    status = hstu.last_device_status(ws)
    elapsed = time.time() - t0
    assert status == TIMEOUT
    assert 0.15 < elapsed < 30.0
    # the context still works: a normal call on the same workspace reports OK
    lens = [100, 40]
    x = workloads.random_inputs(lens, lens, 2, 64, torch.bfloat16, seed=1)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o = hstu.hstu_attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], 100, 100,
                           workspace=ws)
    assert hstu.last_device_status(ws) == 0
    assert torch.isfinite(o.float()).all()
