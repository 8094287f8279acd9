"""Pins for the fp64 oracle: each check ties it to something other than itself.

* the pages' worked example and two-tile split (golden files with citations),
* brute force in pure Python on tiny inputs (math.exp / math.log loops),
* the library routine torch.nn.functional.cross_entropy in float64 with autograd,
* central finite differences of the loss for dH and dW,
* closed forms (W = 0, V = 1, huge logits, softcap -> infinity),
* split invariance of the blockwise (m, s) merge over non-dividing chunk sizes,
* label conventions (ignored rows, all ignored, out-of-range labels),
* the bf16 -> float64 widening every parity test feeds the oracle through, checked on
  all 65536 bit patterns against a decoding of the format's sign, exponent and
  fraction fields, and on values the format fixes (1.0, -3.0, the largest finite
  value, the smallest subnormal 2^-133, the infinities).

A final group plants mistakes in the oracle (monkeypatched, CPU only) and checks
that at least one pin catches each of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.conftest import read_golden

RNG = np.random.default_rng(1234)


def _case(N, Hd, V, seed, ignore_frac=0.25, scale=1.0, bad=False):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, Hd)) * scale
    W = rng.standard_normal((V, Hd)) * scale
    y = rng.integers(0, V, N)
    y[rng.random(N) < ignore_frac] = -100
    if bad:
        y[0] = V + 3
    return H, W, y


# ------------------------------------------------------------------ pages' examples
def pin_worked_example():
    g = read_golden("worked_example.txt")
    z = np.log(np.array(g["logits_exp"], dtype=np.float64))
    # Hd = 1: H = [[1]], W[v] = z_v, so Z = H W^T reproduces the row exactly.
    f = O.forward(np.ones((1, 1)), z[:, None], np.array([g["target"]]))
    assert abs(float(f.loss) - math.log(10 / 3)) < 1e-12
    assert round(float(f.loss), g["loss_digits"]) == g["loss"]
    p = math.exp(f.target[0] - f.lse[0])
    assert abs(p - g["p_target"]) < 1e-12


def pin_two_tile_split():
    g = read_golden("two_tile_split.txt")
    z = np.log(np.array([1.0, 2.0, 3.0, 4.0]))
    a = z[np.array(g["tile_a"])][None, :]
    b = z[np.array(g["tile_b"])][None, :]
    ma, sa = O.tile_stats(a)
    mb, sb = O.tile_stats(b)
    assert abs(math.exp(ma[0]) * sa[0] - g["mass_a"]) < 1e-12
    assert abs(math.exp(mb[0]) * sb[0] - g["mass_b"]) < 1e-12
    m, s = O.merge(ma, sa, mb, sb)
    assert abs(math.exp(m[0]) * s[0] - g["mass_total"]) < 1e-12
    # first tile initialises directly: merging into an empty (-inf, 0) state is exact
    m0, s0 = O.merge(np.array([-np.inf]), np.array([0.0]), ma, sa)
    assert m0[0] == ma[0] and s0[0] == sa[0]
    # the loss with the merged denominator is ln(10/3); the tile-local one is ln(7/3)
    f = O.forward_split(np.ones((1, 1)), z[:, None], np.array([2]), [1], [2, 2])
    assert abs(float(f.loss) - math.log(10 / 3)) < 1e-12
    wrong = float(mb[0] + math.log(sb[0]) - z[2])
    assert round(wrong, g["loss_digits"]) == g["wrong_tile_local_loss"]
    assert abs(float(f.loss) - wrong) > 0.3


# ------------------------------------------------------------------ brute force
def _brute(H, W, y, ignore, c, red, g):
    N, Hd = len(H), len(H[0])
    V = len(W)
    rows = []
    for i in range(N):
        x = [sum(H[i][k] * W[v][k] for k in range(Hd)) for v in range(V)]
        z = [c * math.tanh(t / c) if c > 0 else t for t in x]
        mx = max(z)
        lse = mx + math.log(sum(math.exp(t - mx) for t in z))
        ok = y[i] != ignore and 0 <= y[i] < V
        rows.append((x, z, lse, ok))
    nv = sum(1 for r in rows if r[3])
    losses = [(r[2] - r[1][y[i]]) if r[3] else 0.0 for i, r in enumerate(rows)]
    if red == "mean":
        loss = sum(losses) / nv if nv else 0.0
    elif red == "sum":
        loss = sum(losses)
    else:
        loss = losses
    dH = [[0.0] * Hd for _ in range(N)]
    dW = [[0.0] * Hd for _ in range(V)]
    for i, (x, z, lse, ok) in enumerate(rows):
        if not ok:
            continue
        sc = g / nv if red == "mean" else (g if red == "sum" else g[i])
        for v in range(V):
            d = math.exp(z[v] - lse) - (1.0 if v == y[i] else 0.0)
            if c > 0:
                d *= 1 - math.tanh(x[v] / c) ** 2
            d *= sc
            for k in range(Hd):
                dH[i][k] += d * W[v][k]
                dW[v][k] += d * H[i][k]
    return loss, [r[2] for r in rows], np.array(dH), np.array(dW)


@pytest.mark.parametrize("softcap", [0.0, 2.5])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_brute_force(softcap, red):
    H, W, y = _case(5, 4, 7, seed=7)
    g = 0.7 if red != "none" else list(np.linspace(0.5, 1.5, 5))
    loss, lse, dH, dW = _brute(H.tolist(), W.tolist(), y.tolist(), -100, softcap, red, g)
    f = O.forward(H, W, y, softcap=softcap, reduction=red)
    np.testing.assert_allclose(f.lse, lse, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(f.loss, loss, rtol=1e-13, atol=1e-13)
    oh, ow = O.backward(H, W, y, f.lse, softcap=softcap, reduction=red, grad_out=np.array(g) if red == "none" else g)
    np.testing.assert_allclose(oh, dH, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(ow, dW, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ library routine
def pin_torch_library(N=13, Hd=9, V=37, softcap=0.0, red="mean", seed=3):
    H, W, y = _case(N, Hd, V, seed=seed)
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    X = Ht @ Wt.T
    Z = softcap * torch.tanh(X / softcap) if softcap > 0 else X
    yt = torch.tensor(y)
    L = torch.nn.functional.cross_entropy(Z, yt, ignore_index=-100, reduction=red)
    g = torch.linspace(0.3, 1.9, N, dtype=torch.float64) if red == "none" else torch.tensor(1.3, dtype=torch.float64)
    (L * g).sum().backward()
    f = O.forward(H, W, y, softcap=softcap, reduction=red)
    np.testing.assert_allclose(f.loss, L.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f.lse, torch.logsumexp(Z, 1).detach().numpy(), rtol=1e-12)
    dH, dW = O.backward(H, W, y, f.lse, softcap=softcap, reduction=red, grad_out=g.numpy())
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-14)
    # sampled-row / sampled-vocab helpers agree with the full backward
    rows = np.array([0, 3, N - 1])
    vs = np.array([0, 5, V - 1, int(y[y >= 0][0])])
    np.testing.assert_allclose(O.dH_rows(H, W, y, f.lse[rows], rows, softcap=softcap, reduction=red,
                                         grad_out=g.numpy()), dH[rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(O.dW_rows(H, W, y, f.lse, vs, softcap=softcap, reduction=red,
                                         grad_out=g.numpy()), dW[vs], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(O.lse_rows(H, W, rows, softcap), f.lse[rows], rtol=1e-14)
    np.testing.assert_allclose(O.target_rows(H, W, y, rows, softcap=softcap), f.target[rows], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("softcap", [0.0, 3.0])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_torch_library(softcap, red):
    pin_torch_library(softcap=softcap, red=red)


# ------------------------------------------------------------------ finite differences
def pin_finite_differences(softcap=0.0, red="mean", N=4, Hd=3, V=11, seed=5):
    H, W, y = _case(N, Hd, V, seed=seed, ignore_frac=0.3)
    y[1] = -100
    g = np.linspace(0.4, 1.6, N) if red == "none" else 0.9

    def L(Hx, Wx):
        f = O.forward(Hx, Wx, y, softcap=softcap, reduction=red)
        return float(np.sum(np.asarray(f.loss) * g))

    f = O.forward(H, W, y, softcap=softcap, reduction=red)
    dH, dW = O.backward(H, W, y, f.lse, softcap=softcap, reduction=red, grad_out=g)
    eps = 1e-5
    for A, G in ((H, dH), (W, dW)):
        num = np.zeros_like(A)
        for idx in np.ndindex(A.shape):
            old = A[idx]
            A[idx] = old + eps
            lp = L(H, W)
            A[idx] = old - eps
            lm = L(H, W)
            A[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        err = np.abs(num - G).max() / max(1e-12, np.abs(G).max())
        assert err < 1e-7, err


@pytest.mark.parametrize("softcap", [0.0, 1.5])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_finite_differences(softcap, red):
    pin_finite_differences(softcap, red)


# ------------------------------------------------------------------ closed forms
def pin_closed_forms():
    N, Hd, V = 6, 5, 9
    H, _, y = _case(N, Hd, V, seed=11)
    W = np.zeros((V, Hd))
    f = O.forward(H, W, y)
    np.testing.assert_allclose(f.lse, math.log(V), rtol=1e-15)
    valid = y != -100
    np.testing.assert_allclose(f.loss, math.log(V), rtol=1e-14)
    dH, dW = O.backward(H, W, y, f.lse)
    assert np.abs(dH).max() == 0.0
    nv = valid.sum()
    expect = np.zeros((V, Hd))
    for i in np.nonzero(valid)[0]:
        for v in range(V):
            expect[v] += (1.0 / V - (v == y[i])) * H[i] / nv
    np.testing.assert_allclose(dW, expect, rtol=1e-12, atol=1e-15)
    # V = 1: a one-class softmax has loss 0 and no gradient
    H1, W1 = H, np.ones((1, Hd))
    y1 = np.where(valid, 0, -100)
    f1 = O.forward(H1, W1, y1)
    assert abs(float(f1.loss)) < 1e-15
    d1h, d1w = O.backward(H1, W1, y1, f1.lse)
    assert np.abs(d1h).max() < 1e-15 and np.abs(d1w).max() < 1e-15
    # huge logits: the stable form stays finite and exact
    Hb = np.array([[1.0]])
    Wb = np.array([[1e4], [1e4 - math.log(3.0)], [-1e4]])
    fb = O.forward(Hb, Wb, np.array([1]))
    assert abs(float(fb.loss) - math.log(4.0)) < 1e-9
    assert np.isfinite(fb.lse).all() and abs(fb.lse[0] - (1e4 + math.log(4 / 3))) < 1e-9
    # softcap -> infinity recovers the uncapped result
    H2, W2, y2 = _case(5, 4, 8, seed=12)
    a = O.forward(H2, W2, y2)
    b = O.forward(H2, W2, y2, softcap=1e7)
    np.testing.assert_allclose(a.lse, b.lse, rtol=1e-10)
    # a known softcap value: z = c tanh(x/c) at x = c gives c tanh(1)
    fc = O.forward(np.array([[2.0]]), np.array([[1.0], [0.0]]), np.array([1]), softcap=2.0)
    zc = 2.0 * math.tanh(1.0)
    assert abs(fc.lse[0] - math.log(math.exp(zc) + 1.0)) < 1e-14
    assert abs(float(fc.loss) - math.log(math.exp(zc) + 1.0)) < 1e-14


def test_closed_forms():
    pin_closed_forms()


# ------------------------------------------------------------------ split invariance
def pin_split_invariance(softcap=0.0, red="mean"):
    N, Hd, V = 23, 6, 2000
    H, W, y = _case(N, Hd, V, seed=21)
    y[5] = V - 1
    y[6] = 0
    full = O.forward(H, W, y, softcap=softcap, reduction=red)
    for rows, vocab in (([23], [2000]), ([1, 7, 15], [1, 7, 13, 1000, 979]),
                        ([10, 13], [1999, 1]), ([5, 5, 5, 8], [256] * 7 + [208])):
        sp = O.forward_split(H, W, y, rows, vocab, softcap=softcap, reduction=red)
        np.testing.assert_allclose(sp.lse, full.lse, rtol=1e-12)
        np.testing.assert_allclose(sp.loss, full.loss, rtol=1e-12)
        np.testing.assert_allclose(sp.target, full.target, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("softcap", [0.0, 4.0])
def test_split_invariance(softcap):
    pin_split_invariance(softcap)
    pin_split_invariance(softcap, red="sum")


def test_worked_example():
    pin_worked_example()


def test_two_tile_split():
    pin_two_tile_split()


# ------------------------------------------------------------------ label conventions
def pin_label_conventions():
    N, Hd, V = 8, 4, 10
    H, W, y = _case(N, Hd, V, seed=31, ignore_frac=0.0)
    y[2] = -100
    y[5] = V          # out of range -> bad, treated as ignored
    y[6] = -7         # negative and not ignore_index -> bad
    f = O.forward(H, W, y)
    assert f.n_valid == N - 3 and f.n_bad == 2
    assert f.loss_rows[2] == 0 and f.loss_rows[5] == 0 and f.loss_rows[6] == 0
    dH, dW = O.backward(H, W, y, f.lse)
    assert np.abs(dH[[2, 5, 6]]).max() == 0.0
    # an ignored row contributes nothing to dW: dropping it changes nothing
    keep = np.array([i for i in range(N) if i not in (2, 5, 6)])
    f2 = O.forward(H[keep], W, y[keep])
    _, dW2 = O.backward(H[keep], W, y[keep], f2.lse)
    np.testing.assert_allclose(dW, dW2, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(f.loss, f2.loss, rtol=1e-14)
    # all ignored: loss 0, zero gradient, n_valid 0 (mean and sum)
    ya = np.full(N, -100)
    for red in ("mean", "sum"):
        fa = O.forward(H, W, ya, reduction=red)
        assert float(fa.loss) == 0.0 and fa.n_valid == 0
        a, b = O.backward(H, W, ya, fa.lse, reduction=red)
        assert np.abs(a).max() == 0 and np.abs(b).max() == 0
    # LSE is reported for ignored rows too
    assert np.isfinite(f.lse).all() and abs(f.lse[2] - O.lse_rows(H, W, [2])[0]) < 1e-14
    # custom ignore_index
    yc = y.copy()
    yc[2] = 3
    fc = O.forward(H, W, yc, ignore_index=3)
    assert fc.n_valid == int(((yc != 3) & (yc >= 0) & (yc < V)).sum())


def test_label_conventions():
    pin_label_conventions()


def test_invariants():
    """sum_v dZ_iv = 0 for each valid row (no softcap), so the vocab-sum of dW vanishes."""
    H, W, y = _case(9, 5, 30, seed=41)
    f = O.forward(H, W, y)
    dH, dW = O.backward(H, W, y, f.lse)
    assert np.abs(dW.sum(axis=0)).max() < 1e-14
    P = np.exp(H @ W.T - f.lse[:, None])
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-13)


# ------------------------------------------------------------------ bf16 widening
# The parity tests hand the oracle the same bf16 bit patterns the GPU reads; widen_bf16
# turns them into float64.  bf16 is the upper half of an IEEE-754 binary32 value:
# 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits.
INF = float("inf")
BF16_FIXED = [  # (bits, value) fixed by that format
    (0x0000, 0.0), (0x8000, -0.0), (0x3F80, 1.0), (0xBF80, -1.0), (0xC040, -3.0),
    (0x3EAB, 0.333984375), (0x4049, 3.140625), (0x0001, 2.0 ** -133), (0x007F, 127 * 2.0 ** -133),
    (0x0080, 2.0 ** -126), (0x7F7F, 3.3895313892515355e38), (0xFF7F, -3.3895313892515355e38),
    (0x7F80, INF), (0xFF80, -INF),
]


def _bf16_from_fields(bits):
    """Decode one 16-bit pattern from its sign, exponent and fraction fields."""
    sign = -1.0 if bits >> 15 else 1.0
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0xFF:
        return sign * INF if f == 0 else float("nan")
    if e == 0:                                   # subnormal: 0.f x 2^-126
        return sign * math.ldexp(f, -126 - 7)
    return sign * math.ldexp(128 + f, e - 127 - 7)  # normal: 1.f x 2^(e - 127)


def pin_widen_bf16():
    bits = np.array([b for b, _ in BF16_FIXED], dtype=np.uint16)
    got = O.widen_bf16(bits)
    assert got.dtype == np.float64
    for (b, v), g in zip(BF16_FIXED, got):
        assert g == v and math.copysign(1.0, g) == math.copysign(1.0, v), (hex(b), g, v)
    with np.errstate(invalid="ignore"):        # signalling NaN patterns are among them
        assert np.isnan(O.widen_bf16(np.array([0x7FC0, 0xFFC1, 0x7F81], dtype=np.uint16))).all()
        # every one of the 65536 patterns against the field decoding
        allb = np.arange(1 << 16, dtype=np.int64).astype(np.uint16)
        w = O.widen_bf16(allb)
    ref = np.array([_bf16_from_fields(b) for b in range(1 << 16)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(w), nan)
    assert np.array_equal(w[~nan], ref[~nan])
    assert np.array_equal(np.signbit(w[~nan]), np.signbit(ref[~nan]))
    # the value, not the byte order of the container, decides: a big-endian array widens alike
    np.testing.assert_array_equal(O.widen_bf16(bits.astype(">u2")), got)
    # shape is kept
    with np.errstate(invalid="ignore"):
        assert O.widen_bf16(allb.reshape(256, 256)).shape == (256, 256)
    # binary32 values cut to their top 16 bits widen to exactly that truncated value
    rng = np.random.default_rng(77)
    x = (rng.standard_normal(4096) * np.exp(rng.uniform(-40.0, 40.0, 4096))).astype(np.float32)
    u = x.view(np.uint32)
    cut = (u & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(O.widen_bf16((u >> 16).astype(np.uint16)), cut)


def test_widen_bf16():
    pin_widen_bf16()


# ------------------------------------------------------------------ planted mistakes
ALL_PINS = [pin_worked_example, pin_two_tile_split, pin_torch_library,
            lambda: pin_torch_library(softcap=2.0), lambda: pin_torch_library(red="none"),
            lambda: pin_torch_library(red="sum"),
            pin_finite_differences, lambda: pin_finite_differences(softcap=1.5),
            pin_closed_forms, pin_split_invariance, pin_label_conventions, pin_widen_bf16,
            lambda: pin_filtered_backward()]


def _caught():
    n = 0
    for p in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                p()
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            n += 1
    return n


def _mutants():
    orig_lse, orig_cap_grad, orig_dl, orig_raw = O._lse, O._cap_grad, O._dlogits, O._raw_logits
    orig_scale, orig_merge, orig_status = O.row_scale, O.merge, O.label_status
    orig_dh_rows, orig_target_rows = O.dH_rows, O.target_rows

    def lse_no_shift(Z):                       # dropped max subtraction
        return np.log(np.exp(Z).sum(axis=1))

    def lse_max_only(Z):                       # dropped the log-sum term
        return Z.max(axis=1)

    def cap_grad_one(X, c):                    # dropped the softcap derivative
        return 1.0

    def dl_wrong_sign(X, Z, lse, labels, valid, scale, c, filt=0.0):  # +1 instead of -1 at the target
        D = orig_dl(X, Z, lse, labels, valid, scale, c, filt)
        rows = np.nonzero(valid)[0]
        D[rows, np.asarray(labels)[rows]] += 2.0 * scale[rows] * np.asarray(orig_cap_grad(X, c) * np.ones_like(X))[rows, np.asarray(labels)[rows]]
        return D

    def raw_reversed(Hf, Wf):                  # wrong vocabulary index
        return Hf @ Wf[::-1].T

    def scale_by_rows(valid, n_valid, red, g):  # mean over all rows, not valid rows
        return orig_scale(valid, len(valid), red, g)

    def merge_no_rescale(m1, s1, m2, s2):      # forgot to rescale the old sum
        m = np.maximum(m1, m2)
        return m, np.asarray(s1) + np.asarray(s2)

    def status_no_range(labels, V, ignore):    # out-of-range labels not caught
        y = np.asarray(labels)
        return y != ignore, np.zeros_like(y, dtype=bool)

    def widen_shift8(bits):                    # bf16 placed 8 bits too low
        return (np.asarray(bits).astype(np.uint32) << 8).view(np.float32).astype(np.float64)

    def widen_byteswap(bits):                  # the two bytes of each value swapped
        b = np.asarray(bits).astype(np.uint16).byteswap()
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def widen_as_fp16(bits):                   # read as IEEE half precision instead of bf16
        return np.asarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)

    def scale_sum_as_mean(valid, n_valid, red, g):  # the sum reduction divided by the valid count
        return orig_scale(valid, n_valid, "mean" if red == "sum" else red, g)

    def cap_inner_unscaled(X, c):              # c tanh(x) instead of c tanh(x / c)
        return c * np.tanh(X) if c > 0 else X

    def filter_drops_target(P, labels, valid, thr):  # the target entry filtered like the rest
        return np.where(P >= thr, P, 0.0) if thr > 0 else P

    def dh_rows_local_count(Hf, Wf, labels, lse, rows, *a, n_valid=None, **k):  # count of the sample only
        lab = np.asarray(labels)
        return orig_dh_rows(Hf, Wf, labels, lse, rows, *a, n_valid=int((lab[np.asarray(rows)] != -100).sum()), **k)

    def tile_sum_unshifted(Z):                 # sum of exp(z), not of exp(z - m)
        return Z.max(axis=1), np.exp(Z).sum(axis=1)

    def target_uncapped(Hf, Wf, labels, rows, ignore_index=-100, softcap=0.0):  # target before the cap
        return orig_target_rows(Hf, Wf, labels, rows, ignore_index, 0.0)

    return [("_lse", lse_no_shift), ("_lse", lse_max_only), ("_cap_grad", cap_grad_one),
            ("_dlogits", dl_wrong_sign), ("_raw_logits", raw_reversed), ("row_scale", scale_by_rows),
            ("merge", merge_no_rescale), ("label_status", status_no_range),
            ("widen_bf16", widen_shift8), ("widen_bf16", widen_byteswap), ("widen_bf16", widen_as_fp16),
            ("row_scale", scale_sum_as_mean), ("_cap", cap_inner_unscaled), ("_filter", filter_drops_target),
            ("dH_rows", dh_rows_local_count), ("tile_stats", tile_sum_unshifted),
            ("target_rows", target_uncapped)]


def test_pins_pass_on_the_oracle():
    assert _caught() == 0


@pytest.mark.parametrize("mutant", range(17))
def test_planted_mistake_is_caught(mutant, monkeypatch):
    name, fn = _mutants()[mutant]
    monkeypatch.setattr(O, name, fn)
    assert _caught() >= 1, name


# ------------------------------------------------------------------ gradient filtering
def pin_filtered_backward():
    """threshold 0 is the exact gradient; a threshold above every probability keeps only
    the target entries, whose closed form is dH_i = (p_iy - 1) s_i w_y and
    dW_v = sum over rows with y_i = v of (p_iy - 1) s_i h_i; an intermediate threshold
    drops exactly the entries below it (brute force)."""
    H, W, y = _case(7, 5, 23, seed=51)
    f = O.forward(H, W, y)
    exact = O.backward(H, W, y, f.lse)
    zero = O.backward(H, W, y, f.lse, filter_threshold=0.0)
    np.testing.assert_array_equal(exact[0], zero[0])
    np.testing.assert_array_equal(exact[1], zero[1])
    valid = y != -100
    nv = valid.sum()
    dH, dW = O.backward(H, W, y, f.lse, filter_threshold=2.0)
    eh = np.zeros_like(H)
    ew = np.zeros_like(W)
    for i in np.nonzero(valid)[0]:
        py = math.exp(float(H[i] @ W[y[i]]) - f.lse[i])
        eh[i] = (py - 1.0) / nv * W[y[i]]
        ew[y[i]] += (py - 1.0) / nv * H[i]
    np.testing.assert_allclose(dH, eh, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dW, ew, rtol=1e-12, atol=1e-15)
    thr = 0.05
    P = np.exp(H @ W.T - f.lse[:, None])
    D = np.zeros_like(P)
    for i in range(len(y)):
        if not valid[i]:
            continue
        for v in range(W.shape[0]):
            keep = P[i, v] >= thr or v == y[i]
            D[i, v] = ((P[i, v] if keep else 0.0) - (v == y[i])) / nv
    dH2, dW2 = O.backward(H, W, y, f.lse, filter_threshold=thr)
    np.testing.assert_allclose(dH2, D @ W, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dW2, D.T @ H, rtol=1e-12, atol=1e-15)
    rows = np.array([0, 3])
    np.testing.assert_allclose(O.dH_rows(H, W, y, f.lse[rows], rows, filter_threshold=thr), dH2[rows], rtol=1e-12,
                               atol=1e-15)
    vs = np.array([0, 4, 22])
    np.testing.assert_allclose(O.dW_rows(H, W, y, f.lse, vs, filter_threshold=thr), dW2[vs], rtol=1e-12, atol=1e-15)


def test_filtered_backward_pins():
    pin_filtered_backward()


# ------------------------------------------------------------------ vocabulary order
def _order_by_selection(keys):
    """Brute force: repeatedly take the largest remaining key, the smallest id on ties."""
    left = list(range(len(keys)))
    out = []
    while left:
        best = left[0]
        for v in left[1:]:
            if keys[v] > keys[best]:
                best = v
        out.append(best)
        left.remove(best)
    return out


def test_vocab_order_pins():
    """Hand-worked case: H = [[1, 0], [3, 2]], W rows (1,1), (0,2), (2,0), (1,1) give the
    logits [[1, 0, 2, 1], [5, 4, 6, 5]], mean logits [3, 2, 4, 3] and the order
    [2, 0, 3, 1] (ids 0 and 3 tie at 3 and keep id order)."""
    H = np.array([[1.0, 0.0], [3.0, 2.0]])
    W = np.array([[1.0, 1.0], [0.0, 2.0], [2.0, 0.0], [1.0, 1.0]])
    keys = O.vocab_keys(H, W)
    np.testing.assert_array_equal(keys, [3.0, 2.0, 4.0, 3.0])
    assert O.vocab_order(keys).tolist() == [2, 0, 3, 1]
    np.testing.assert_array_equal(O.vocab_keys(H, W, vocab=[3, 1]), [3.0, 2.0])
    # ties and stability
    assert O.vocab_order([1.0, 5.0, 5.0, -2.0, 5.0, 0.0]).tolist() == [1, 2, 4, 0, 5, 3]
    assert O.vocab_order([0.0, -0.0, 0.0]).tolist() == [0, 1, 2]
    # brute force on random keys with many ties
    rng = np.random.default_rng(61)
    for n in (1, 2, 17, 64):
        k = np.round(rng.standard_normal(n) * 2.0) / 2.0
        assert O.vocab_order(k).tolist() == _order_by_selection(list(k))
    # closed form: a constant first feature and nothing else makes the key that column
    Hc = np.zeros((9, 4))
    Hc[:, 0] = 1.0
    Wc = rng.standard_normal((11, 4))
    np.testing.assert_allclose(O.vocab_keys(Hc, Wc), Wc[:, 0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(O.vocab_keys(np.zeros((0, 4)), Wc), np.zeros(11))
    # the mean over rows, brute force on a small random case
    Hr, Wr = rng.standard_normal((5, 3)), rng.standard_normal((7, 3))
    brute = [sum(sum(Hr[i, k] * Wr[v, k] for k in range(3)) for i in range(5)) / 5 for v in range(7)]
    np.testing.assert_allclose(O.vocab_keys(Hr, Wr), brute, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("mutant", ["ascending", "ties_descending", "sum_not_mean", "mean_over_vocab"])
def test_vocab_order_mistake_is_caught(mutant, monkeypatch):
    orig_keys = O.vocab_keys
    if mutant == "ascending":
        monkeypatch.setattr(O, "vocab_order", lambda k: np.lexsort((np.arange(len(k)), np.asarray(k, float))))
    elif mutant == "ties_descending":
        monkeypatch.setattr(O, "vocab_order", lambda k: np.lexsort((-np.arange(len(k)), -np.asarray(k, float))))
    elif mutant == "sum_not_mean":
        monkeypatch.setattr(O, "vocab_keys", lambda H, W, vocab=None: orig_keys(H, W, vocab) * max(H.shape[0], 1))
    else:
        monkeypatch.setattr(O, "vocab_keys", lambda H, W, vocab=None: (H @ W.T).mean(axis=1))  # over vocab
    with pytest.raises((AssertionError, ValueError, IndexError)):
        test_vocab_order_pins()
