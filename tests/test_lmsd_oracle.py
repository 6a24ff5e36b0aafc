"""Pins for the LMSD oracle (oracle/lmsd.py), on CPU.

* LayerNorm against torch.nn.functional.layer_norm (fp64), SiLU against
  torch.nn.functional.silu: the forward with dropout off is a composition of
  library routines;
* the segment order [dropout(a), dropout(x), dropout(l a)] and the mask bits;
* inverted dropout: dropped elements are exactly 0, kept ones exactly the
  undropped value / (1 - p), keep rates within binomial bounds;
* the backward against torch.autograd on the same formulation with the mask
  fixed;
* Philox4x32-10: full avalanche (one flipped counter or key bit changes about
  half of the output bits, which a generator with too few or broken rounds
  does not), uniform words, independent segments.
* Philox4x32-10 against the generator authors' published known-answer
  values (tests/golden/philox4x32_10_kat.txt).
The mapping of Philox words to elements is a reading (the page fixes only
the generator); the GPU and CPU implementations, written separately, must
agree on it bit for bit.
"""
import pathlib
import numpy as np
import pytest
import torch

from oracle import lmsd


def _inputs(n, d, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(n, d, generator=g) * 2 + 0.5).to(torch.bfloat16).double()
    u = torch.randn(n, d, generator=g).to(torch.bfloat16).double()
    w = torch.randn(d, generator=g).to(torch.bfloat16).double()
    b = torch.randn(d, generator=g).to(torch.bfloat16).double()
    return x, u, w, b


@pytest.mark.parametrize("silu", [True, False])
def test_no_dropout_is_layer_norm_times_activation(silu):
    x, u, w, b = _inputs(33, 40, 1)
    y, mean, rstd, mask = lmsd.forward(x, u, w, b, 1e-5, 0.0, 7, silu, True, True)
    assert mask is None and y.shape == (33, 120)
    ln = torch.nn.functional.layer_norm(x, (40,), w, b, 1e-5).numpy()
    a = torch.nn.functional.silu(u).numpy() if silu else u.numpy()
    np.testing.assert_allclose(y[:, :40], a, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(y[:, 40:80], x.numpy())
    np.testing.assert_allclose(y[:, 80:], ln * a, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(mean, x.mean(1).numpy(), rtol=1e-13)
    var = torch.var(x, dim=1, unbiased=False).numpy()
    np.testing.assert_allclose(rstd, 1 / np.sqrt(var + 1e-5), rtol=1e-13)


def test_segments_can_be_dropped_from_the_output():
    x, u, w, b = _inputs(5, 16, 2)
    y1, *_ = lmsd.forward(x, u, w, b, 1e-6, 0.0, 0, True, False, False)
    y3, *_ = lmsd.forward(x, u, w, b, 1e-6, 0.0, 0, True, True, True)
    assert y1.shape == (5, 16)
    np.testing.assert_array_equal(y1, y3[:, 32:])
    yx, *_ = lmsd.forward(x, u, w, b, 1e-6, 0.0, 0, True, False, True)   # x segment only
    np.testing.assert_array_equal(yx[:, :16], x.numpy())


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_inverted_dropout(p):
    n, d = 64, 256
    x, u, w, b = _inputs(n, d, 3)
    y, _, _, mask = lmsd.forward(x, u, w, b, 1e-5, p, 1234, True, True, True)
    y0, _, _, _ = lmsd.forward(x, u, w, b, 1e-5, 0.0, 1234, True, True, True)
    pf = float(np.float32(p))
    for k, seg in ((0, 2), (1, 1), (2, 0)):     # mask bit, output segment
        kept = ((mask >> k) & 1).astype(bool)
        got, ref = y[:, seg * d:(seg + 1) * d], y0[:, seg * d:(seg + 1) * d]
        assert np.all(got[~kept] == 0.0)
        np.testing.assert_array_equal(got[kept], ref[kept] * (1.0 / (1.0 - pf)))
        rate, m = kept.mean(), kept.size
        assert abs(rate - (1 - pf)) < 5 * np.sqrt(pf * (1 - pf) / m)
    # segments decide independently
    k0, k1 = mask & 1, (mask >> 1) & 1
    assert abs(np.corrcoef(k0.ravel(), k1.ravel())[0, 1]) < 0.05
    # disabled segments leave their bits clear
    _, _, _, m1 = lmsd.forward(x, u, w, b, 1e-5, p, 1234, True, False, False)
    assert np.all(m1 >> 1 == 0) and np.array_equal(m1 & 1, mask & 1)


@pytest.mark.parametrize("flags", [(True, True, True), (False, False, False), (True, False, True)])
@pytest.mark.parametrize("p", [0.0, 0.3])
def test_backward_matches_autograd(flags, p):
    silu, cu, cx = flags
    n, d = 9, 24
    x, u, w, b = _inputs(n, d, 4)
    y, mean, rstd, mask = lmsd.forward(x, u, w, b, 1e-5, p, 99, silu, cu, cx)
    dy = np.random.default_rng(0).standard_normal(y.shape)
    dx, du, dw, db = lmsd.backward(dy, x, u, w, b, mean, rstd, mask, p, silu, cu, cx)
    xs, us, ws, bs = (t.clone().requires_grad_(True) for t in (x, u, w, b))
    pf = float(np.float32(p))
    ms = [torch.ones(n, d, dtype=torch.float64)] * 3 if p == 0 else \
        [torch.from_numpy(((mask >> k) & 1).astype(np.float64)) / (1 - pf) for k in (0, 1, 2)]
    ln = torch.nn.functional.layer_norm(xs, (d,), ws, bs, 1e-5)
    a = torch.nn.functional.silu(us) if silu else us
    segs = ([a * ms[2]] if cu else []) + ([xs * ms[1]] if cx else []) + [ln * a * ms[0]]
    (torch.cat(segs, 1) * torch.from_numpy(dy)).sum().backward()
    np.testing.assert_allclose(dx, xs.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(du, us.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dw, ws.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(db, bs.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_philox_known_answers():
    path = pathlib.Path(__file__).parent / "golden" / "philox4x32_10_kat.txt"
    rows = [ln.split() for ln in path.read_text().splitlines() if ln and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(t, 16) for t in r]
        out = lmsd.philox4x32_10(*[[t] for t in v[:4]], v[4], v[5])
        assert [int(o[0]) for o in out] == v[6:], r


def _popcount(v):
    v = np.asarray(v, dtype=np.uint64)
    return np.array([bin(int(t)).count("1") for t in v.ravel()]).reshape(v.shape)


def test_philox_avalanche_and_uniformity():
    rng = np.random.default_rng(5)
    c = [rng.integers(0, 2**32, size=4000, dtype=np.uint64) for _ in range(4)]
    key = (0x12345678, 0x9ABCDEF0)
    base = lmsd.philox4x32_10(*c, *key)
    for word in range(4):
        for bit in (0, 17, 31):
            cc = [v.copy() for v in c]
            cc[word] ^= np.uint64(1 << bit)
            out = lmsd.philox4x32_10(*cc, *key)
            flips = sum(_popcount(o ^ b0) for o, b0 in zip(out, base)) / 4.0
            assert abs(flips.mean() - 16.0) < 0.5, (word, bit, flips.mean())
    for kk in ((key[0] ^ 1, key[1]), (key[0], key[1] ^ (1 << 20))):  # one bit of either key word
        out = lmsd.philox4x32_10(*c, *kk)
        flips = sum(_popcount(o ^ b0) for o, b0 in zip(out, base)) / 4.0
        assert abs(flips.mean() - 16.0) < 0.5
    words = np.concatenate(base).astype(np.float64) / 2**32
    assert abs(words.mean() - 0.5) < 0.01 and abs(words.var() - 1 / 12) < 0.005
    # a stream counted from zero, as the dropout uses it, is uniform too
    w0 = lmsd.keep_halves(512, 512, 0, 42).astype(np.float64) / 2**16
    hist = np.histogram(w0, bins=16, range=(0, 1))[0] / w0.size
    assert np.all(np.abs(hist - 1 / 16) < 0.003)


def test_keep_halves_layout():
    """Eight elements per Philox call: element e takes the 16-bit half e % 2
    (low first) of word (e % 8) // 2 of the call with counter e // 8."""
    n, d, seed = 3, 24, (7 << 32) | 5
    h = lmsd.keep_halves(n, d, 2, seed).ravel()
    for e in (0, 1, 6, 7, 8, 15, 40, 71):
        g = e // 8
        words = lmsd.philox4x32_10([g], [0], [2], [0], 5, 7)
        want = (int(words[(e % 8) // 2][0]) >> (16 * (e % 2))) & 0xFFFF
        assert int(h[e]) == want, e
    assert lmsd.threshold(0.5) == 32768 and lmsd.threshold(0.1) == 6553
