"""Gradient filtering (CCE-style tile skipping) on the GPU.

With filter_threshold > 0 the backward drops softmax entries below the threshold
(other than a valid row's target) and skips every 64 x 64 block of dZ left all zero in
the dW and dH products.  Parity is checked against the oracle of the *filtered*
gradient (same rule in fp64) with the usual tolerances; the approximation error of the
filtered gradient against the exact one is measured and printed separately (it is a
property of the method, not of the kernels)."""
import numpy as np
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

THR = 2.0 ** -12


def _filtered_case(w, thr, chunk_budget=0, labels=None):
    Hb, Wb, y = P.make_case(w, labels)
    out = P.run_gpu(Hb, Wb, y, w.ignore_index, w.softcap, w.reduction, chunk_budget=chunk_budget,
                    filter_threshold=thr)
    ref, dH_f, dW_f = P.oracle_full(Hb, Wb, y, w.ignore_index, w.softcap, w.reduction, filter_threshold=thr)
    P.check_forward(out, ref, y, w.V, w.ignore_index, w.reduction)
    errs = P.check_backward(out, dH_f, dW_f)
    _, dH_x, dW_x = P.oracle_full(Hb, Wb, y, w.ignore_index, w.softcap, w.reduction)
    approx = dict(dH=P.fro_rel(dH_f, dH_x), dW=P.fro_rel(dW_f, dW_x))
    print("\n%s thr=%g parity %s, filtered-vs-exact %s" % (w.name, thr, errs, approx))
    return out, approx


@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_filtered_peaked_multi_chunk(softcap):
    # confident predictions; 3 vocabulary chunks with a ragged last chunk
    w = S.scaled("peaked", N=520, Hd=256, V=5000, seed=41, w_std=0.1, softcap=softcap)
    out, approx = _filtered_case(w, THR, chunk_budget=520 * 2 * 2048)
    assert approx["dH"] < 0.05 and approx["dW"] < 0.2


def test_filtered_flat_softmax_drops_almost_everything():
    # flat softmax (p ~ 1/V < threshold): only target entries survive, most blocks skip
    w = S.scaled("llama3", N=300, Hd=128, V=3000, seed=42)
    _filtered_case(w, THR, chunk_budget=300 * 2 * 1024)


def test_threshold_above_one_keeps_only_targets():
    w = S.scaled("peaked", N=257, Hd=64, V=2100, seed=43, w_std=0.1)
    _filtered_case(w, 2.0)


def test_filtered_all_ignored_is_zero():
    w = S.scaled("tiny", N=200, Hd=64, V=900, seed=44)
    Hb, Wb, _ = P.make_case(w)
    y = np.full(200, -100, dtype=np.int64)
    out = P.run_gpu(Hb, Wb, y, filter_threshold=THR)
    assert np.abs(out["dH"]).max() == 0.0 and np.abs(out["dW"]).max() == 0.0


def test_filter_zero_is_the_exact_path():
    w = S.scaled("peaked", N=300, Hd=128, V=2600, seed=45, w_std=0.1)
    Hb, Wb, y = P.make_case(w)
    a = P.run_gpu(Hb, Wb, y, filter_threshold=0.0)
    b = P.run_gpu(Hb, Wb, y)
    assert np.array_equal(a["dH"], b["dH"]) and np.array_equal(a["dW"], b["dW"])
