"""Parity at the full workload sizes, in the launch configuration bench.py times
(default vocabulary chunk budget).

For each workload the fp64 oracle computes every row's LSE (row blocks, library
matmul), so lse, the target logits and the mean loss are compared for all rows.  dH
is compared on one random row of every 128-row block of tokens (the rows one CTA
owns in a 256-row output tile) plus the first and last row, and dW on one random
vocabulary row of every 128-row block plus the 48 most frequent labels and the last
48 ids (the ragged last tile), so every output tile of both products is sampled.
Their relative Frobenius errors are estimated on those samples, and every sampled row
is held to the per-row bound of tests/parity.py."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _one_per_block(n, rng, block=128):
    """One uniformly drawn index in each block of `block` consecutive indices of [0, n)."""
    starts = np.arange(0, n, block, dtype=np.int64)
    return starts + (rng.random(len(starts)) * np.minimum(block, n - starts)).astype(np.int64)


def _sample_rows(N, rng):
    return np.unique(np.concatenate([[0, N - 1], _one_per_block(N, rng)]))


def _sample_vocab(y, V, rng):
    yv = y[y >= 0]
    freq = np.bincount(yv, minlength=V)
    top = np.argsort(-freq, kind="stable")[:48]
    last = np.arange(V - 48, V)
    return np.unique(np.concatenate([top, _one_per_block(V, rng), last]))


@pytest.mark.parametrize("name", ["llama2", "llama3", "gemma2", "packed"])
def test_full_size_workload(name):
    import linear_cross_entropy_indexed_gb300 as F
    w = S.WORKLOADS[name]
    Hb, Wb, y = S.make_H(w), S.make_W(w), S.make_labels(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, tgt = F.flce_forward(H, W, lab, w.ignore_index, w.softcap, w.reduction, want_target=True)
    g = torch.ones(1, device="cuda")
    dH, dW = F.flce_backward(H, W, lab, lse, counts, g, w.ignore_index, w.softcap, w.reduction)
    torch.cuda.synchronize()
    got_lse = lse.double().cpu().numpy()
    got_t = tgt.double().cpu().numpy()
    c = counts.cpu().numpy()
    del H, W

    Hf, Wf = O.widen_bf16(Hb), O.widen_bf16(Wb)
    ref = O.forward(Hf, Wf, y, w.ignore_index, w.softcap, w.reduction, row_block=1024)
    valid, bad = O.label_status(y, w.V, w.ignore_index)
    assert int(c[0]) == ref.n_valid and int(c[1]) == ref.n_bad and int(c[2]) == 0
    lse_err = np.abs(got_lse - ref.lse)
    t_err = np.abs(got_t - ref.target)[valid].max()
    loss_rel = abs(float(loss) - float(ref.loss)) / float(ref.loss)
    assert lse_err.max() <= P.TOL_LSE_ABS
    assert t_err <= P.TOL_TARGET_ABS
    assert loss_rel <= P.TOL_LOSS_REL

    rng = np.random.default_rng(1000 + w.seed)
    rows = _sample_rows(w.N, rng)
    dh_ref = O.dH_rows(Hf, Wf, y, ref.lse[rows], rows, w.ignore_index, w.softcap, w.reduction, 1.0,
                       n_valid=ref.n_valid)
    dh_got = S.bf16_bits_to_f32(P.bf16_bits(dH[torch.from_numpy(rows).cuda()])).astype(np.float64)
    assert P.fro_rel(dh_got, dh_ref) <= P.TOL_GRAD_FRO
    rh = P.check_rows("dH", dh_got, dh_ref)
    vs = _sample_vocab(y, w.V, rng)
    dw_ref = O.dW_rows(Hf, Wf, y, ref.lse, vs, w.ignore_index, w.softcap, w.reduction, 1.0)
    dw_got = S.bf16_bits_to_f32(P.bf16_bits(dW[torch.from_numpy(vs).cuda()])).astype(np.float64)
    assert P.fro_rel(dw_got, dw_ref) <= P.TOL_GRAD_FRO
    rw = P.check_rows("dW", dw_got, dw_ref)
    print("\n%s: lse abs err max %.3g mean %.3g, signed mean %.3g; target abs err max %.3g; loss rel err %.3g; "
          "dH rel fro (%d sampled rows) %.3g, worst row %.3g; dW rel fro (%d sampled rows) %.3g, worst row %.3g" % (
              name, lse_err.max(), lse_err.mean(), float(np.mean(got_lse - ref.lse)), t_err, loss_rel,
              len(rows), P.fro_rel(dh_got, dh_ref), rh, len(vs), P.fro_rel(dw_got, dw_ref), rw))
    # ignored rows carry no gradient
    ign = np.nonzero(~valid)[0][:16]
    if len(ign):
        assert dH[torch.from_numpy(ign).cuda()].abs().max().item() == 0.0
