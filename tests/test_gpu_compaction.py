"""The backward runs on the rows that carry a gradient only (a valid label and a non-zero
upstream gradient): they are gathered to the front on the device, in their original order,
and dH is written back through a row map.  These tests cover what that changes:

* heavy padding (whole 256-row tiles of ignored rows, as in padded sequences), every
  reduction, a chunked backward, the softcap: parity with the fp64 oracle, and an exactly
  zero dH row for every row without a gradient;
* reduction "none" with upstream gradients that are exactly zero on some valid rows: those
  rows get a zero dH row and leave dW as if they were absent;
* invariance: inserting rows without a gradient anywhere in a batch leaves every other row's
  dH and the whole dW bit for bit unchanged (the compacted rows are the same, in the same
  order), for the exact, compensated and filtered backwards."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _padded_labels(y, rng, frac):
    """Ignore whole runs of rows (padded sequence ends) until about `frac` of them."""
    y = y.copy()
    N = len(y)
    while (y == -100).mean() < frac:
        a = int(rng.integers(0, N))
        y[a:a + int(rng.integers(64, 600))] = -100
    return y


@pytest.mark.parametrize("reduction,softcap", [("mean", 0.0), ("sum", 30.0), ("none", 0.0)])
def test_heavy_padding(reduction, softcap):
    w = S.scaled("llama3", N=1500, Hd=136, V=3001, seed=101, w_std=0.1, softcap=softcap)
    Hb, Wb, y = P.make_case(w)
    y = _padded_labels(y, np.random.default_rng(7), 0.7)
    out = P.run_gpu(Hb, Wb, y, -100, softcap, reduction, chunk_budget=1500 * 2 * 1024)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, -100, softcap, reduction)
    P.check_forward(out, ref, y, w.V, -100, reduction)
    valid, _ = O.label_status(y, w.V, -100)
    P.check_backward(out, dH, dW, no_grad_rows=~valid)
    assert (~valid).mean() >= 0.7


def test_zero_upstream_gradients():
    w = S.scaled("llama3", N=700, Hd=128, V=2500, seed=102, w_std=0.1)
    Hb, Wb, y = P.make_case(w)
    g = np.linspace(0.5, 1.5, w.N)
    g[::3] = 0.0                      # a third of the rows: valid labels, zero gradient
    out = P.run_gpu(Hb, Wb, y, reduction="none", grad=g)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, reduction="none", grad=g)
    valid, _ = O.label_status(y, w.V, -100)
    P.check_backward(out, dH, dW, no_grad_rows=(~valid) | (g == 0.0))


def _backward(Hb, Wb, y, **kw):
    import linear_cross_entropy_indexed_gb300 as F
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab, reduction="sum")
    dH, dW = F.flce_backward(H, W, lab, lse, counts, torch.ones(1, device="cuda"), reduction="sum",
                             chunk_budget=kw.pop("chunk_budget", 0), **kw)
    torch.cuda.synchronize()
    assert int(counts[2]) == 0
    return P.bf16_bits(dH), P.bf16_bits(dW)


@pytest.mark.parametrize("mode", ["exact", "compensated", "filtered"])
def test_rows_without_gradient_change_nothing(mode):
    kw = dict(exact={}, compensated=dict(compensated=True), filtered=dict(filter_threshold=2.0 ** -12))[mode]
    w = S.scaled("peaked" if mode == "filtered" else "llama3", N=600, Hd=128, V=3000, seed=103, w_std=0.1,
                 ignore_frac=0.0, peak=(6.0 if mode == "filtered" else 0.0))
    Hb, Wb, y = P.make_case(w)
    # the same rows with 700 rows without a gradient inserted between them
    rng = np.random.default_rng(8)
    extra_H = S.normal_bf16((700, w.Hd), 99, 1, 1.0)
    pos = np.sort(rng.choice(600 + 700, 700, replace=False))
    keep = np.setdiff1d(np.arange(1300), pos)
    H2 = np.empty((1300, w.Hd), dtype=np.uint16)
    H2[pos], H2[keep] = extra_H, Hb
    y2 = np.full(1300, -100, dtype=np.int64)
    y2[keep] = y
    y2[pos[::7]] = w.V + 5            # some of them bad labels rather than ignored
    # the same 1024-column vocabulary chunks for both batches (the chunking sets dH's
    # summation grouping)
    per_row = (4 if mode == "compensated" else 2) * 1024
    dh_a, dw_a = _backward(Hb, Wb, y, chunk_budget=600 * per_row, **kw)
    dh_b, dw_b = _backward(H2, Wb, y2, chunk_budget=1300 * per_row, **kw)
    assert np.array_equal(dw_a, dw_b)
    assert np.array_equal(dh_a, dh_b[keep])
    assert not np.any(dh_b[pos])
