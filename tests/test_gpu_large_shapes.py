"""Shapes at the edges of the tiling and indexing: a hidden size of 8192 (128 K steps per
tile), a vocabulary of a million rows (977 forward partials per row, 245 sort runs and 8
merge passes), and 65536 token rows (256 pair tiles) with a small vocabulary.  Every
output is compared element by element with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _full_check(w, chunk_budget=0, **kw):
    Hb, Wb, y = P.make_case(w)
    out = P.run_gpu(Hb, Wb, y, w.ignore_index, w.softcap, w.reduction, chunk_budget=chunk_budget, **kw)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, w.ignore_index, w.softcap, w.reduction)
    P.check_forward(out, ref, y, w.V, w.ignore_index, w.reduction)
    errs = P.check_backward(out, dH, dW)
    print("\n%s N=%d Hd=%d V=%d: %s" % (w.name, w.N, w.Hd, w.V, errs))
    return Hb, Wb, y


def test_hidden_8192():
    w = S.scaled("llama3", N=384, Hd=8192, V=2100, seed=91, w_std=0.01)
    _full_check(w)


def test_vocabulary_of_a_million():
    w = S.scaled("llama3", N=96, Hd=64, V=1_000_003, seed=92, w_std=0.15)
    Hb, Wb, _ = _full_check(w)
    import linear_cross_entropy_indexed_gb300 as F
    keys, perm, inv = F.vocab_order(P.to_device(Hb), P.to_device(Wb))
    torch.cuda.synchronize()
    k = keys.cpu().numpy().astype(np.float64)
    assert np.array_equal(perm.cpu().numpy().astype(np.int64), O.vocab_order(k))
    vs = np.arange(0, w.V, 9973)
    np.testing.assert_allclose(k[vs], O.vocab_keys(O.widen_bf16(Hb), O.widen_bf16(Wb), vs), rtol=1e-4, atol=1e-6)


def test_sixty_four_thousand_rows():
    w = S.scaled("tiny", N=65536, Hd=64, V=520, seed=93, ignore_frac=0.07)
    _full_check(w, chunk_budget=65536 * 2 * 256)   # 3 vocabulary chunks of 256 columns
