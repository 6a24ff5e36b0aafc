"""GPU parity: the CUDA path (called through the C ABI via the binding)
against the fp64 oracle on the same bf16/fp16 inputs, element by element.

Tolerances: forward max-abs error <= 1e-2 * max|O_ref|, each gradient
<= 2e-2 * max|grad_ref| (see hstu_testlib)."""
import math

import numpy as np
import pytest
import torch

import oracle
from generative_recommender_attention_gb300 import workloads
import generative_recommender_attention_gb300 as hstu

from hstu_testlib import TOL_BWD, TOL_FWD, check, full_compare, gpu_fwd_bwd, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _ws(name):
    return workloads.WORKLOADS[name]


# ------------------------------------------------------------------ workloads
def test_tiny_workload_full():
    w = _ws("tiny")
    x = workloads.make_inputs(w, seed=0)
    full_compare(x, w.scaling_seqlen, w.causal, w.alpha)


@pytest.mark.parametrize("name", ["recsys", "long", "skewed", "full"])
def test_workload_full_size(name):
    """Every element of O, dQ, dK and dV at the full workload sizes, against
    the whole fp64 oracle run on all host cores (the oracle does the full
    recommender batch in about a second and the full-mask D = 256 batch in
    under a minute there)."""
    w = _ws(name)
    x = workloads.make_inputs(w, seed=0)
    full_compare(x, w.scaling_seqlen, w.causal, w.alpha)


# ------------------------------------------------------------------ medium, every variant
MEDIUM_LENS = [300, 1, 129, 517, 0, 64, 256]


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("causal", [True, False])
def test_medium_every_variant(D, dtype, causal):
    x = workloads.random_inputs(MEDIUM_LENS, MEDIUM_LENS, 2, D, dtype, seed=D + int(causal))
    alpha = 1.0 / math.sqrt(D)
    full_compare(x, None, causal, alpha)


# ------------------------------------------------------------------ windows
# Local / sliding windows ("Mask support", window_size = (left, right)).
WINDOWS = [(0, 0), (16, 0), (200, 40), (70, -1), (-1, 100), (129, 1), (1000, 0)]


@pytest.mark.parametrize("D,dtype", [(32, torch.float16), (64, torch.bfloat16),
                                     (128, torch.float16), (256, torch.bfloat16)])
@pytest.mark.parametrize("window", WINDOWS)
def test_medium_windows(D, dtype, window):
    x = workloads.random_inputs(MEDIUM_LENS, MEDIUM_LENS, 2, D, dtype, seed=D + window[0] + 7)
    full_compare(x, None, window, 1.0 / math.sqrt(D))


@pytest.mark.parametrize("window", [(256, 0), (64, 64)])
def test_window_unequal_lengths(window):
    lq = [100, 250, 7, 300, 513]
    lk = [180, 250, 40, 200, 600]
    x = workloads.random_inputs(lq, lk, 2, 128, torch.bfloat16, seed=13)
    x["max_seqlen_k"] = max(max(lk), x["max_seqlen_q"])
    full_compare(x, 96, window, 0.2)


def test_window_recsys_full():
    """The recsys workload's shapes with a 256-token look-back window, every
    element compared."""
    w = _ws("recsys")
    x = workloads.make_inputs(w, seed=0)
    full_compare(x, w.scaling_seqlen, (256, 0), w.alpha)


# ------------------------------------------------------------------ arbitrary (func) masks
def _local(x):
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_k"].tolist()
    T = cq[-1]
    i, lk = np.zeros(T, np.int64), np.zeros(T, np.int64)
    for b in range(len(cq) - 1):
        i[cq[b]:cq[b + 1]] = np.arange(cq[b + 1] - cq[b])
        lk[cq[b]:cq[b + 1]] = ck[b + 1] - ck[b]
    return i, lk


def _func_mask(kind, x, seed=0, pad=256):
    """Endpoint patterns: causal with the last 8 keys as targets; a band with
    a hole; random endpoints (N = 5)."""
    i, lk = _local(x)
    rng = np.random.default_rng(seed)
    if kind == "causal_targets":
        rows = [i + 1, lk - 8, lk]
    elif kind == "band_hole":
        rows = [np.minimum(i + 1, 64), np.maximum(0, i - 200), np.maximum(0, i - 100),
                np.maximum(0, i - 40), i + 30]
    else:
        rows = [rng.integers(-50, int(lk.max()) + 50, size=i.shape[0]) for _ in range(5)]
    F = np.stack([np.asarray(r) for r in rows]).astype(np.int32)
    return {"func": np.concatenate([F, np.zeros((F.shape[0], pad), np.int32)], axis=1)}


@pytest.mark.parametrize("D,dtype", [(32, torch.float16), (64, torch.bfloat16),
                                     (128, torch.float16), (256, torch.bfloat16)])
@pytest.mark.parametrize("kind", ["causal_targets", "band_hole", "random"])
def test_func_masks(D, dtype, kind):
    x = workloads.random_inputs(MEDIUM_LENS, MEDIUM_LENS, 2, D, dtype, seed=D + len(kind))
    full_compare(x, None, _func_mask(kind, x, seed=D), 1.0 / math.sqrt(D))


@pytest.mark.parametrize("kind", ["causal_targets", "band_hole"])
def test_func_mask_long_sequence(kind):
    """A sequence of more than 32 key tiles: the live-tile bitmaps take two
    32-bit words per query block and the scheduler walks two tile groups."""
    lens = [4500, 300, 1]
    x = workloads.random_inputs(lens, lens, 2, 64, torch.bfloat16, seed=17)
    full_compare(x, None, _func_mask(kind, x, seed=3), 0.125)


def test_func_mask_equal_to_causal_is_bitwise_causal():
    x = workloads.random_inputs(MEDIUM_LENS, MEDIUM_LENS, 2, 128, torch.bfloat16, seed=5)
    i, _ = _local(x)
    fm = {"func": np.concatenate([(i + 1)[None].astype(np.int32), np.zeros((1, 3), np.int32)], 1)}
    xd = to_dev(x)
    a = gpu_fwd_bwd(xd, None, fm, 0.09)
    b = gpu_fwd_bwd(xd, None, True, 0.09)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_func_mask_recsys_full():
    """The recsys workload with causal attention plus the last 16 keys of
    every sequence as targets, every element compared."""
    w = _ws("recsys")
    x = workloads.make_inputs(w, seed=0)
    i, lk = _local(x)
    fm = {"func": np.stack([i + 1, lk - 16, lk]).astype(np.int32)}
    full_compare(x, w.scaling_seqlen, fm, w.alpha)


# ------------------------------------------------------------------ paged K/V forward
def _paged_cache(x, n_extra, seed, garbage=1e3):
    """Scatter x's K/V into shuffled 128-row pages (plus unused pages); rows
    past each sequence's keys hold finite garbage."""
    rng = np.random.default_rng(seed)
    ck = x["cu_seqlens_k"].tolist()
    lens = [ck[b + 1] - ck[b] for b in range(len(ck) - 1)]
    n_pages = [-(-L // 128) for L in lens]
    total = sum(n_pages) + n_extra
    perm = rng.permutation(total)
    H, D = x["k"].shape[1], x["k"].shape[2]
    kv = (torch.from_numpy(rng.uniform(-garbage, garbage, (total, 2, 128, H, D)))
          .to(x["k"].dtype))
    ids, ptr, used = [], [0], 0
    for b, L in enumerate(lens):
        for p in range(n_pages[b]):
            page = int(perm[used])
            used += 1
            ids.append(page)
            lo, hi = ck[b] + 128 * p, ck[b] + min(L, 128 * p + 128)
            kv[page, 0, :hi - lo] = x["k"][lo:hi]
            kv[page, 1, :hi - lo] = x["v"][lo:hi]
        ptr.append(len(ids))
    return kv, torch.tensor(ids, dtype=torch.int32), torch.tensor(ptr, dtype=torch.int32)


@pytest.mark.parametrize("D,dtype", [(32, torch.bfloat16), (64, torch.float16),
                                     (128, torch.bfloat16), (256, torch.float16)])
def test_paged_forward(D, dtype):
    lq = [300, 1, 129, 517, 0, 64, 256]
    lk = [340, 1, 129, 600, 3, 64, 256]
    x = workloads.random_inputs(lq, lk, 2, D, dtype, seed=D + 17)
    x["max_seqlen_k"] = max(lk)
    kv, ids, ptr = _paged_cache(x, n_extra=5, seed=D)
    xd = to_dev(x)
    alpha = 1.0 / math.sqrt(D)
    o = hstu.hstu_attn_fwd_paged(xd["q"], kv.cuda(), ids.cuda(), ptr.cuda(), xd["cu_seqlens_q"],
                                 xd["cu_seqlens_k"], x["max_seqlen_q"], x["max_seqlen_k"],
                                 alpha=alpha)
    torch.cuda.synchronize()
    L = oracle.resolve_scaling(None, x["max_seqlen_q"])
    ref = oracle.fwd_paged(x["q"], kv, ids, ptr, x["cu_seqlens_q"], x["cu_seqlens_k"], alpha, L)
    check("O paged", o, ref, TOL_FWD)
    # the same kernel over the contiguous keys computes the same numbers
    oc = hstu.hstu_attn_fwd(xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"], xd["cu_seqlens_k"],
                            x["max_seqlen_q"], x["max_seqlen_k"], causal=True, alpha=alpha)
    torch.cuda.synchronize()
    assert torch.equal(o, oc)


def test_paged_forward_recsys_full():
    """The recsys workload's sequences served from a shuffled page pool, every
    output element compared."""
    w = _ws("recsys")
    x = workloads.make_inputs(w, seed=0)
    kv, ids, ptr = _paged_cache(x, n_extra=17, seed=1)
    xd = to_dev(x)
    o = hstu.hstu_attn_fwd_paged(xd["q"], kv.cuda(), ids.cuda(), ptr.cuda(), xd["cu_seqlens_q"],
                                 xd["cu_seqlens_k"], x["max_seqlen_q"], x["max_seqlen_k"],
                                 alpha=w.alpha, scaling_seqlen=w.scaling_seqlen)
    torch.cuda.synchronize()
    L = oracle.resolve_scaling(w.scaling_seqlen, x["max_seqlen_q"])
    ref = oracle.fwd_paged(x["q"], kv, ids, ptr, x["cu_seqlens_q"], x["cu_seqlens_k"], w.alpha, L)
    check("O paged", o, ref, TOL_FWD)


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("causal", [True, False])
def test_unequal_q_and_k_lengths(causal):
    # per sequence Lq <= Lk, and one sequence with Lq > Lk (max_q <= max_k still)
    lq = [100, 250, 7, 300]
    lk = [180, 250, 40, 200]
    x = workloads.random_inputs(lq, lk, 2, 64, torch.bfloat16, seed=3)
    x["max_seqlen_k"] = max(max(lk), x["max_seqlen_q"])
    full_compare(x, 96, causal, 0.2)


def test_sequences_without_keys_get_zero_rows():
    lq = [50, 130, 20]
    lk = [60, 0, 140]
    x = workloads.random_inputs(lq, lk, 2, 128, torch.bfloat16, seed=4)
    res = full_compare(x, None, True, 0.1)
    xd = to_dev(x)
    o, dq, _, _ = gpu_fwd_bwd(xd, None, True, 0.1)
    assert torch.all(o[50:180] == 0) and torch.all(dq[50:180] == 0)
    assert res["o"][1] > 0


def test_length_one_and_empty_sequences():
    lens = [1, 0, 1, 1, 0, 2, 1]
    x = workloads.random_inputs(lens, lens, 3, 64, torch.float16, seed=5)
    full_compare(x, 4, True, 0.3)


def test_single_long_sequence_ragged_tail():
    lens = [1000]
    x = workloads.random_inputs(lens, lens, 1, 128, torch.bfloat16, seed=6)
    full_compare(x, None, True, 1.0 / math.sqrt(128))


def test_explicit_scaling_and_negative_alpha():
    lens = [200, 77]
    x = workloads.random_inputs(lens, lens, 2, 64, torch.bfloat16, seed=7)
    full_compare(x, 1000, True, -0.15)


def test_strided_views_and_packed_kv_gradients():
    """q/k/v as views of one packed (T, 3, H, D) buffer, dk/dv as disjoint
    views of one packed (T, H, 2D) buffer, out with a padded token stride."""
    lens = [140, 260, 33]
    T, H, D = sum(lens), 2, 64
    g = torch.Generator().manual_seed(8)
    qkv = torch.randn(T, 3, H, D, generator=g).to(torch.bfloat16)
    do = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
    cu = workloads.cu_seqlens(lens)
    x = {"q": qkv[:, 0], "k": qkv[:, 1], "v": qkv[:, 2], "do": do, "cu_seqlens_q": cu,
         "cu_seqlens_k": cu.clone(), "max_seqlen_q": max(lens), "max_seqlen_k": max(lens)}
    qkv_d = qkv.cuda()
    xd = {"q": qkv_d[:, 0], "k": qkv_d[:, 1], "v": qkv_d[:, 2], "do": do.cuda(),
          "cu_seqlens_q": cu.cuda(), "cu_seqlens_k": cu.cuda(),
          "max_seqlen_q": max(lens), "max_seqlen_k": max(lens)}
    out_buf = torch.full((T, H, D + 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    kv_grad = torch.full((T, H, 2 * D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o, dq, dk, dv = gpu_fwd_bwd(xd, None, True, 0.125,
                                fwd={"out": out_buf[:, :, :D]},
                                bwd={"dk": kv_grad[:, :, :D], "dv": kv_grad[:, :, D:]})
    assert o.data_ptr() == out_buf.data_ptr()
    L = float(max(lens))
    ro = oracle.fwd(x["q"], x["k"], x["v"], cu, cu, 0.125, L, True)
    rdq, rdk, rdv = oracle.bwd(do, x["q"], x["k"], x["v"], cu, cu, 0.125, L, True)
    check("O", o, ro, TOL_FWD)
    check("dQ", dq, rdq, TOL_BWD)
    check("dK", kv_grad[:, :, :D], rdk, TOL_BWD)
    check("dV", kv_grad[:, :, D:], rdv, TOL_BWD)
    assert torch.isnan(out_buf[:, :, D:].float()).all()   # padding untouched


def test_backward_is_deterministic():
    w = _ws("recsys")
    x = workloads.make_inputs(w, seed=1, lengths=[700, 256, 1024, 300])
    xd = to_dev(x)
    a = gpu_fwd_bwd(xd, None, True, w.alpha)
    b = gpu_fwd_bwd(xd, None, True, w.alpha)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_outputs_fully_overwritten():
    lens = [129, 64, 300]
    x = workloads.random_inputs(lens, lens, 2, 128, torch.float16, seed=9)
    xd = to_dev(x)
    T = sum(lens)
    nan = lambda: torch.full((T, 2, 128), float("nan"), dtype=torch.float16, device="cuda")  # noqa
    o, dq, dk, dv = gpu_fwd_bwd(xd, None, False, 0.09, fwd={"out": nan()},
                                bwd={"dq": nan(), "dk": nan(), "dv": nan()})
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()


def test_device_status_ok_after_calls():
    lens = [300, 20]
    x = workloads.random_inputs(lens, lens, 2, 64, torch.bfloat16, seed=10)
    xd = to_dev(x)
    ws = torch.empty(hstu.workspace_size(2, 320, 320, 2, 64, 300, 300, True), dtype=torch.uint8,
                     device="cuda")
    hstu.hstu_attn_bwd(xd["do"], xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"],
                       xd["cu_seqlens_k"], 300, 300, workspace=ws)
    assert hstu.last_device_status(ws) == 0


def test_backward_reports_understated_max_seqlen():
    # A sequence longer than max_seqlen_q makes the dS blocks outgrow the
    # workspace, which is sized from max_seqlen_q: the stores past its end are
    # skipped (nothing outside the workspace is written) and the device status
    # reports an invalid argument.
    lens = [700, 20]
    x = workloads.random_inputs(lens, lens, 2, 64, torch.bfloat16, seed=11)
    xd = to_dev(x)
    n = hstu.workspace_size(2, 720, 720, 2, 64, 64, 64, True)
    guard = 1 << 16
    buf = torch.full((n + 2 * guard,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = buf[guard:guard + n]
    hstu.hstu_attn_bwd(xd["do"], xd["q"], xd["k"], xd["v"], xd["cu_seqlens_q"],
                       xd["cu_seqlens_k"], 64, 64, workspace=ws)
    assert hstu.last_device_status(ws) == 1   # HSTU_ERR_INVALID_ARG
    assert torch.all(buf[:guard] == 0x5A) and torch.all(buf[guard + n:] == 0x5A)
