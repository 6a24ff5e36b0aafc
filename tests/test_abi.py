"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/hstu_attn.h declares, sizes its workspace, and rejects bad arguments
on the host before anything is launched (those paths make no CUDA call)."""
import ctypes
import os
import re

import pytest

from generative_recommender_attention_gb300 import _lib as L
from generative_recommender_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("hstu_attn.h", "hstu_lmsd.h")]

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.library()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hstu_(?:attn|lmsd)_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(L.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_symbols_have_c_linkage():
    out = os.popen(f"nm -D --defined-only {L.library_path()}").read()
    names = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in names, name


def test_version_and_status_strings(lib):
    assert lib.hstu_attn_version() == 100
    for code in range(6):
        assert lib.hstu_attn_status_string(code)
    assert lib.hstu_attn_status_string(5) == b"device wait timed out"


def _bwd_bytes(B, Tq, Tk, H, D, max_q):
    # header | list A | list B (unit records of 32 bytes, units <= H * (ceil(T/128) + B),
    # twice on the key side for D = 256) | B + 1 block offsets | 1024-aligned dS blocks of
    # 128 keys x 64 queries x 2 bytes, H * ceil(max_q / 64) * (ceil(Tk / 128) + B) of them
    cdiv = lambda a, b: -(-a // b)  # noqa: E731
    capA = H * (cdiv(Tq, 128) + B)
    capB = H * (2 if D == 256 else 1) * (cdiv(Tk, 128) + B)
    ds = (256 + 32 * capA + 32 * capB + 4 * (B + 1) + 1023) // 1024 * 1024
    total = ds + H * cdiv(max_q, 64) * (cdiv(Tk, 128) + B) * 128 * 64 * 2
    return (total + 255) // 256 * 256


def test_workspace_size(lib):
    ws = lib.hstu_attn_workspace_size
    # forward: header + 32 bytes per unit record, units <= H * (ceil(T/128) + B), 256-aligned
    assert ws(4, 309, 309, 2, 64, 128, 128, 0) == (256 + 32 * 2 * (3 + 4) + 255) // 256 * 256
    fwd = ws(32, 20480, 20480, 4, 128, 1024, 1024, 0)
    bwd = ws(32, 20480, 20480, 4, 128, 1024, 1024, 1)
    assert bwd == _bwd_bytes(32, 20480, 20480, 4, 128, 1024) and fwd < bwd
    assert ws(16, 65536, 65536, 2, 256, 4096, 4096, 1) == _bwd_bytes(16, 65536, 65536, 2, 256, 4096)
    assert ws(4, 309, 309, 2, 64, 128, 128, 1) == _bwd_bytes(4, 309, 309, 2, 64, 128)
    # the dS bound grows with max_seqlen_q, not with max_seqlen_k
    assert ws(4, 309, 309, 2, 64, 64, 128, 1) < ws(4, 309, 309, 2, 64, 128, 128, 1)
    assert ws(4, 309, 309, 2, 64, 128, 256, 1) == ws(4, 309, 309, 2, 64, 128, 128, 1)
    assert ws(1, 10, 10, 1, 96, 10, 10, 0) == 0        # unsupported head_dim
    assert ws(-1, 10, 10, 1, 64, 10, 10, 0) == 0
    assert ws(1, 10, 10, 0, 64, 10, 10, 0) == 0
    assert ws(1, 10, 10, 1, 64, -1, 10, 1) == 0
    # more than 2^31 - 1 dS blocks cannot be indexed
    assert ws(1 << 20, 1 << 30, 1 << 30, 64, 64, 1 << 30, 1 << 30, 1) == 0


def _call_fwd(lib, **over):
    """hstu_attn_fwd with fake (never dereferenced) device pointers."""
    a = dict(q=(0x10000, 256, 64), k=(0x20000, 256, 64), v=(0x30000, 256, 64),
             out=(0x40000, 256, 64), cu_q=0x50000, cu_k=0x60000, batch=2, total_q=100,
             total_k=100, H=4, D=64, dtype=L.HSTU_BF16, max_q=60, max_k=60, alpha=0.125,
             scaling=0, wl=-1, wr=0, ws=0x70000, ws_bytes=1 << 20, stream=None)
    a.update(over)
    return lib.hstu_attn_fwd(L.CTen(*a["q"]), L.CTen(*a["k"]), L.CTen(*a["v"]),
                             L.Ten(*a["out"]), a["cu_q"], a["cu_k"], a["batch"], a["total_q"],
                             a["total_k"], a["H"], a["D"], a["dtype"], a["max_q"], a["max_k"],
                             a["alpha"], a["scaling"], a["wl"], a["wr"], a["ws"], a["ws_bytes"],
                             a["stream"])


def test_fwd_argument_errors(lib):
    assert _call_fwd(lib, D=96) == UNSUPPORTED
    assert _call_fwd(lib, D=16) == UNSUPPORTED
    assert _call_fwd(lib, dtype=7) == UNSUPPORTED
    assert _call_fwd(lib, max_q=61, max_k=60) == INVALID          # max_seqlen_q > max_seqlen_k
    assert _call_fwd(lib, scaling=-1) == INVALID                 # scaling_seqlen must be > 0
    assert _call_fwd(lib, alpha=float("nan")) == INVALID
    assert _call_fwd(lib, alpha=float("inf")) == INVALID
    assert _call_fwd(lib, batch=-1) == INVALID
    assert _call_fwd(lib, H=0) == INVALID
    assert _call_fwd(lib, wl=-2) == INVALID                      # window bounds are -1 or >= 0
    assert _call_fwd(lib, wr=-5) == INVALID
    assert _call_fwd(lib, total_q=-5) == INVALID
    assert _call_fwd(lib, cu_q=None) == INVALID
    assert _call_fwd(lib, q=(0, 256, 64)) == INVALID              # null with rows
    assert _call_fwd(lib, q=(0x10008, 256, 64)) == MISALIGNED     # base not 16-byte aligned
    assert _call_fwd(lib, k=(0x20000, 260, 64)) == MISALIGNED     # stride 520 bytes
    assert _call_fwd(lib, v=(0x30000, 256, 36)) == MISALIGNED     # head stride 72 bytes
    assert _call_fwd(lib, out=(0x40000, 256, 32)) == INVALID      # heads overlap (32 < 64)
    assert _call_fwd(lib, out=(0x40000, 64, 64)) == INVALID       # tokens overlap heads
    assert _call_fwd(lib, out=(0x40000, -256, 64)) == INVALID
    assert _call_fwd(lib, ws=None) == INVALID                     # workspace required
    assert _call_fwd(lib, ws_bytes=16) == INVALID                 # workspace too small
    assert _call_fwd(lib, ws=0x70010) == MISALIGNED               # workspace 256-aligned
    assert _call_fwd(lib, max_q=0, max_k=0, scaling=0) == INVALID  # L_scale would be 0


def test_fwd_empty_problems_are_noops(lib):
    # nothing to compute: returns before touching the device
    assert _call_fwd(lib, batch=0) == OK
    assert _call_fwd(lib, total_q=0, q=(0, 256, 64), out=(0, 256, 64)) == OK


def test_non_contiguous_layouts_accepted_by_validation(lib):
    # (T, H, 2D) packed KV buffer: k and v are disjoint views with stride_t = 2*H*D
    from generative_recommender_attention_gb300._lib import CTen  # noqa: F401
    st = lib.hstu_attn_workspace_size(2, 100, 100, 4, 64, 60, 60, 0)
    assert st > 0
    # validation of a padded layout passes (the call then fails only for lack
    # of a device, which the CPU test does not reach: batch = 0 short-cuts)
    assert _call_fwd(lib, k=(0x20000, 512, 128), v=(0x20080, 512, 128), batch=0) == OK


def _call_bwd(lib, **over):
    t = (0x10000, 256, 64)
    a = dict(do=t, q=t, k=t, v=t, dq=(0x80000, 256, 64), dk=(0x90000, 256, 64),
             dv=(0xA0000, 256, 64), batch=2, total_q=100, total_k=100, D=64, max_q=60,
             max_k=60, scaling=0, wl=-1, wr=-1, ws_bytes=1 << 20)
    a.update(over)
    return lib.hstu_attn_bwd(L.CTen(*a["do"]), L.CTen(*a["q"]), L.CTen(*a["k"]), L.CTen(*a["v"]),
                             L.Ten(*a["dq"]), L.Ten(*a["dk"]), L.Ten(*a["dv"]), 0x50000, 0x60000,
                             a["batch"], a["total_q"], a["total_k"], 4, a["D"], L.HSTU_FP16,
                             a["max_q"], a["max_k"], 0.5, a["scaling"], a["wl"], a["wr"],
                             0x70000, a["ws_bytes"], None)


def test_bwd_argument_errors(lib):
    assert _call_bwd(lib, D=48) == UNSUPPORTED
    assert _call_bwd(lib, max_q=70) == INVALID
    assert _call_bwd(lib, scaling=-3) == INVALID
    assert _call_bwd(lib, dk=(0x90004, 256, 64)) == MISALIGNED
    assert _call_bwd(lib, dv=(0xA0000, 8, 64)) == INVALID
    assert _call_bwd(lib, ws_bytes=100) == INVALID
    assert _call_bwd(lib, wl=-7) == INVALID
    assert _call_bwd(lib, batch=0) == OK
    assert _call_bwd(lib, batch=0, wl=5, wr=3) == OK


def test_plan_workspace_size(lib):
    cdiv = lambda a, b: -(-a // b)  # noqa: E731
    ps = lib.hstu_attn_plan_workspace_size
    for B, Tq, Tk, H, D, mq in ((32, 20480, 20480, 4, 128, 1024), (4, 309, 309, 2, 64, 128),
                                (16, 65536, 65536, 2, 256, 4096)):
        capA = H * (cdiv(Tq, 128) + B)
        want = (_bwd_bytes(B, Tq, Tk, H, D, mq) + 32 * capA + 255) // 256 * 256
        assert ps(B, Tq, Tk, H, D, mq, mq) == want
    assert ps(1, 10, 10, 1, 96, 10, 10) == 0
    assert ps(1 << 20, 1 << 30, 1 << 30, 64, 64, 1 << 30, 1 << 30) == 0


def _call_plan(lib, **over):
    a = dict(cu_q=0x50000, cu_k=0x60000, batch=2, total_q=100, total_k=100, H=4, D=64, max_q=60,
             max_k=60, wl=-1, wr=0, ws=0x70000, ws_bytes=1 << 22)
    a.update(over)
    return lib.hstu_attn_plan(a["cu_q"], a["cu_k"], a["batch"], a["total_q"], a["total_k"],
                              a["H"], a["D"], a["max_q"], a["max_k"], a["wl"], a["wr"], a["ws"],
                              a["ws_bytes"], None)


def test_plan_argument_errors(lib):
    assert _call_plan(lib, D=96) == UNSUPPORTED
    assert _call_plan(lib, max_q=61) == INVALID
    assert _call_plan(lib, wl=-2) == INVALID
    assert _call_plan(lib, cu_k=None) == INVALID
    assert _call_plan(lib, ws=None) == INVALID
    assert _call_plan(lib, ws_bytes=4096) == INVALID
    assert _call_plan(lib, ws=0x70040) == MISALIGNED
    assert _call_plan(lib, batch=0) == OK
    # planned calls need a plan-sized workspace: a forward-sized one is refused
    fwd_bytes = lib.hstu_attn_workspace_size(2, 100, 100, 4, 64, 60, 60, 0)
    t = L.CTen(0x10000, 256, 64)
    o = L.Ten(0x40000, 256, 64)
    assert lib.hstu_attn_fwd_planned(t, t, t, o, 0x50000, 0x60000, 2, 100, 100, 4, 64,
                                     L.HSTU_BF16, 60, 60, 0.125, 0, -1, 0, 0x70000, fwd_bytes,
                                     None) == INVALID
    assert lib.hstu_attn_bwd_planned(t, t, t, t, o, o, o, 0x50000, 0x60000, 2, 100, 100, 4, 64,
                                     L.HSTU_BF16, 60, 60, 0.125, 0, -1, 0, 0x70000, 1 << 10,
                                     None) == INVALID
    assert lib.hstu_attn_fwd_planned(t, t, t, o, 0x50000, 0x60000, 0, 100, 100, 4, 64,
                                     L.HSTU_BF16, 60, 60, 0.125, 0, -1, 0, None, 0, None) == OK


def _call_paged(lib, **over):
    a = dict(kv=0x20000, pages=4, ids=0x30000, ptr=0x40000, batch=2, D=64, max_q=60, max_k=60)
    a.update(over)
    return lib.hstu_attn_fwd_paged(L.CTen(0x10000, 256, 64), a["kv"], a["pages"], a["ids"],
                                   a["ptr"], L.Ten(0x50000, 256, 64), 0x60000, 0x61000,
                                   a["batch"], 100, 4, a["D"], L.HSTU_BF16, a["max_q"],
                                   a["max_k"], 0.125, 0, 0x70000, 1 << 20, None)


def test_paged_argument_errors(lib):
    assert _call_paged(lib, kv=None) == INVALID
    assert _call_paged(lib, pages=0) == INVALID
    assert _call_paged(lib, ids=None) == INVALID
    assert _call_paged(lib, ptr=None) == INVALID
    assert _call_paged(lib, kv=0x20008) == MISALIGNED
    assert _call_paged(lib, D=96) == UNSUPPORTED
    assert _call_paged(lib, max_q=70) == INVALID
    assert _call_paged(lib, batch=0) == OK


def _call_fwd_func(lib, **over):
    a = dict(func=0x80000, n=3, L=100, batch=2, D=64, ws_bytes=1 << 20)
    a.update(over)
    t = L.CTen(0x10000, 256, 64)
    return lib.hstu_attn_fwd_func(t, t, t, L.Ten(0x40000, 256, 64), 0x50000, 0x60000,
                                  a["batch"], 100, 100, 4, a["D"], L.HSTU_BF16, 60, 60, 0.125,
                                  0, a["func"], a["n"], a["L"], 0x70000, a["ws_bytes"], None)


def test_func_argument_errors(lib):
    assert _call_fwd_func(lib, n=2) == INVALID          # N must be odd
    assert _call_fwd_func(lib, n=0) == INVALID
    assert _call_fwd_func(lib, L=99) == INVALID         # L >= total_q
    assert _call_fwd_func(lib, func=None) == INVALID
    assert _call_fwd_func(lib, func=0x80002) == MISALIGNED
    assert _call_fwd_func(lib, D=48) == UNSUPPORTED
    need = lib.hstu_attn_workspace_size_func(2, 100, 100, 4, 64, 60, 60, 0)
    assert need > lib.hstu_attn_workspace_size(2, 100, 100, 4, 64, 60, 60, 0)
    assert _call_fwd_func(lib, ws_bytes=need - 1) == INVALID
    assert _call_fwd_func(lib, batch=0) == OK


def _lmsd_fwd(lib, **over):
    a = dict(x=0x10000, xs=128, u=0x20000, us=128, w=0x30000, b=0x30100, n=10, d=128, eps=1e-5,
             p=0.1, mask=0x50000, y=0x40000)
    a.update(over)
    return lib.hstu_lmsd_fwd(a["x"], a["xs"], a["u"], a["us"], a["w"], a["b"], a["n"], a["d"],
                             a["eps"], a["p"], 1, 1, 1, 7, a["y"], 0x60000, 0x61000, a["mask"],
                             None)


def test_lmsd_argument_errors(lib):
    assert _lmsd_fwd(lib, d=12) == UNSUPPORTED      # D multiple of 8
    assert _lmsd_fwd(lib, d=1024) == UNSUPPORTED    # D < 1024
    assert _lmsd_fwd(lib, p=1.0) == INVALID
    assert _lmsd_fwd(lib, p=-0.1) == INVALID
    assert _lmsd_fwd(lib, eps=0.0) == INVALID
    assert _lmsd_fwd(lib, xs=100) == INVALID        # stride < D
    assert _lmsd_fwd(lib, x=0x10008) == MISALIGNED
    assert _lmsd_fwd(lib, mask=None) == INVALID     # dropout needs the mask
    assert _lmsd_fwd(lib, n=0) == OK
    assert lib.hstu_lmsd_bwd_workspace_size(1000, 128) > 0
    assert lib.hstu_lmsd_bwd_workspace_size(1000, 7) == 0


def test_selftest_argument_errors(lib):
    assert lib.hstu_attn_selftest_timeout(None, 1000, None) == INVALID
    assert lib.hstu_attn_selftest_timeout(0x70000, 0, None) == INVALID
    assert lib.hstu_attn_selftest_timeout(0x70000, 20_000_000, None) == INVALID
    assert lib.hstu_attn_selftest_timeout(0x70008, 1000, None) == MISALIGNED
    assert lib.hstu_attn_last_device_status(None, None) == INVALID


def test_binding_rejects_bad_tensors_on_cpu():
    import torch
    import generative_recommender_attention_gb300 as g
    q = torch.zeros(8, 2, 64, dtype=torch.float32)
    cu = torch.tensor([0, 8], dtype=torch.int32)
    with pytest.raises(TypeError):
        g.hstu_attn_fwd(q, q, q, cu, cu, 8, 8)
    with pytest.raises(ValueError):
        g._window(True, (4, -3))
    with pytest.raises(ValueError):
        g._scaling(-2)
    assert g._window(False, (-1, 0)) == (-1, 0) and g._window(True, (-1, -1)) == (-1, -1)
    assert g._window(True, None) == (-1, 0) and g._window(False, None) == (-1, -1)
    assert g._window(True, (16, 3)) == (16, 3)


def _window_rules():
    """The tile-range and dS-block rules of kernels.h (query_tile_keys,
    key_tile_queries, ds_block_off), restated in Python."""
    cdiv = lambda a, b: -(-a // b)  # noqa: E731

    def query_tile_keys(t, Lq, Lk, w, bn):
        r0, r1 = 128 * t, min(128 * t + 128, Lq)
        j0 = 0 if w[0] < 0 else max(0, r0 - w[0])
        j1 = Lk if w[1] < 0 else min(Lk, r1 + w[1])
        first = j0 // bn
        return first, (cdiv(j1, bn) - first if r1 > r0 and j1 > j0 else 0)

    def key_tile_queries(s, Lq, Lk, w, bq):
        c0, c1 = 128 * s, min(128 * s + 128, Lk)
        i0 = 0 if w[1] < 0 else max(0, c0 - w[1])
        i1 = Lq if w[0] < 0 else min(Lq, c1 + w[0])
        first = i0 // bq
        return first, (cdiv(i1, bq) - first if c1 > c0 and i1 > i0 else 0)

    def ds_block_off(j, Lq, Lk, w):
        nqb = cdiv(Lq, 64)
        if w == (-1, -1):
            return j * nqb
        if w == (-1, 0):
            jj = min(j, (nqb + 1) // 2)
            return jj * nqb - jj * (jj - 1)
        return sum(key_tile_queries(t, Lq, Lk, w, 64)[1] for t in range(j))

    return cdiv, query_tile_keys, key_tile_queries, ds_block_off


def _valid(i, j, Lq, Lk, w):
    return (i < Lq and j < Lk and (w[0] < 0 or j >= i - w[0])
            and (w[1] < 0 or j <= i + w[1]))


def test_tile_ranges_cover_exactly_the_valid_pairs():
    """Brute force over the mask definition: the key tiles a query tile
    visits, and the query blocks a key tile visits, are exactly those holding
    at least one valid (query, key) pair, for random windows and ragged
    lengths; the closed forms of ds_block_off equal the summed counts."""
    import random
    cdiv, qtk, ktq, off = _window_rules()
    rng = random.Random(3)
    for _ in range(300):
        Lk = rng.randint(0, 700)
        Lq = rng.randint(0, Lk)
        w = rng.choice([(-1, 0), (-1, -1), (0, 0), (rng.randint(0, 300), rng.randint(-1, 200)),
                        (rng.randint(-1, 300), rng.randint(0, 40)), (rng.randint(0, 90), -1)])
        for bn in (64, 128):
            for t in range(cdiv(Lq, 128)):
                first, n = qtk(t, Lq, Lk, w, bn)
                need = {j // bn for i in range(128 * t, min(128 * t + 128, Lq))
                        for j in range(Lk) if _valid(i, j, Lq, Lk, w)}
                assert set(range(first, first + n)) == need, (Lq, Lk, w, bn, t)
        for s_ in range(cdiv(Lk, 128)):
            first, n = ktq(s_, Lq, Lk, w, 64)
            need = {i // 64 for j in range(128 * s_, min(128 * s_ + 128, Lk))
                    for i in range(Lq) if _valid(i, j, Lq, Lk, w)}
            assert set(range(first, first + n)) == need, (Lq, Lk, w, s_)
        if w in ((-1, 0), (-1, -1)):
            for j in range(cdiv(Lk, 128) + 1):
                assert off(j, Lq, Lk, w) == sum(ktq(t, Lq, Lk, w, 64)[1] for t in range(j))


def test_ds_block_layout_rule():
    """The dS block layout of the backward workspace (kernels.h: ds_blocks_of,
    ds_block_off, ds_blocks_head; sched.cu: ds_base), restated and checked by
    brute force on random ragged batches and windows: every block the dK/dV
    kernel writes has a unique index inside its sequence's range, the dQ
    kernel finds each block it reads where it was written (and a block it
    does not find holds no valid pair, so reading zeros there is exact), and
    the host's size bound holds."""
    import random
    cdiv, qtk, ktq, off = _window_rules()
    rng = random.Random(7)
    for _ in range(300):
        w = rng.choice([(-1, 0), (-1, -1), (0, 0), (rng.randint(0, 300), rng.randint(-1, 200)),
                        (rng.randint(-1, 300), rng.randint(0, 40))])
        B, H = rng.randint(1, 5), rng.randint(1, 3)
        Lk = [rng.randint(0, 600) for _ in range(B)]
        Lq = [rng.randint(0, l) if rng.random() < 0.3 else l for l in Lk]
        base = [0]
        for b in range(B):
            base.append(base[-1] + H * off(cdiv(Lk[b], 128), Lq[b], Lk[b], w))
        written = {}
        for b in range(B):
            head_blocks = (base[b + 1] - base[b]) // H
            for h in range(H):
                for j in range(cdiv(Lk[b], 128)):
                    first = base[b] + h * head_blocks + off(j, Lq[b], Lk[b], w)
                    m0, n = ktq(j, Lq[b], Lk[b], w, 64)      # the key tile's half-steps
                    for m in range(n):
                        k = first + m
                        assert base[b] <= k < base[b + 1] and k not in written
                        written[k] = (b, h, j, m0 + m)
        assert len(written) == base[-1]
        for b in range(B):
            nqb, head_blocks = cdiv(Lq[b], 64), (base[b + 1] - base[b]) // H
            for h in range(H):
                for i in range(cdiv(Lq[b], 128)):
                    kt0, n = qtk(i, Lq[b], Lk[b], w, 128)
                    running = off(kt0, Lq[b], Lk[b], w)
                    for j in range(kt0, kt0 + n):
                        m0, cnt = ktq(j, Lq[b], Lk[b], w, 64)
                        assert running == off(j, Lq[b], Lk[b], w)
                        for m in (2 * i, 2 * i + 1):
                            if m >= nqb:
                                continue
                            if m0 <= m < m0 + cnt:
                                blk = base[b] + h * head_blocks + running + m - m0
                                assert written[blk] == (b, h, j, m)
                            else:   # never stored: must hold no valid pair
                                assert not any(_valid(ii, jj, Lq[b], Lk[b], w)
                                               for ii in range(64 * m, 64 * m + 64)
                                               for jj in range(128 * j, 128 * j + 128))
                        running += cnt
        assert base[-1] <= H * cdiv(max(Lq), 64) * (cdiv(sum(Lk), 128) + B)


def test_plan_key_checked_by_the_binding():
    import generative_recommender_attention_gb300 as hstu
    p = hstu.HstuPlan(None, (2, 100, 100, 4, 64, 60, 60, (-1, 0)))
    p.check((2, 100, 100, 4, 64, 60, 60, (-1, 0)))
    with pytest.raises(ValueError):
        p.check((2, 100, 100, 4, 64, 61, 61, (-1, 0)))
    with pytest.raises(ValueError):
        p.check((2, 100, 100, 4, 64, 60, 60, (-1, -1)))
