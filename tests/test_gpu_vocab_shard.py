"""Vocabulary-sharded (vocab-parallel) path on one GPU: the shards of W are processed one
after another (no cross-kernel waits), their per-shard LSE and target logits merged with
flce_merge_shards, and the backward run per shard from the global LSE; the summed dH
partials and the concatenated dW shards must match the fp64 oracle of the unsharded
problem (ai-infra-kb M011 §07: global max / exponential sum / target, dH summed over
shards)."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _sharded(Hb, Wb, y, cuts, softcap=0.0, reduction="mean", grad=None, chunk_budget=0, filter_threshold=0.0):
    import linear_cross_entropy_indexed_gb300 as F
    H = P.to_device(Hb)
    lab = torch.from_numpy(y).cuda()
    V = Wb.shape[0]
    bounds = [0] + list(cuts) + [V]
    shards = [(a, P.to_device(Wb[a:b])) for a, b in zip(bounds[:-1], bounds[1:])]
    parts = [F.flce_forward_shard(H, Ws, lab, off, V, softcap=softcap) for off, Ws in shards]
    c0 = parts[0][2].tolist()
    for _, _, c in parts:
        assert c.tolist() == c0  # every shard sees the same (global) validity
    loss, lse, counts = F.flce_merge_shards(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]),
                                            lab, V, reduction=reduction)
    N = len(y)
    g = torch.tensor(np.linspace(0.5, 1.5, N) if reduction == "none" else [1.0], dtype=torch.float32).cuda()
    dh = torch.zeros(N, Hb.shape[1], dtype=torch.float32, device="cuda")
    dws = []
    for off, Ws in shards:
        dh_part, dw = F.flce_backward_shard(H, Ws, lab, lse, counts, g, off, V, softcap=softcap, reduction=reduction,
                                            chunk_budget=chunk_budget, filter_threshold=filter_threshold)
        dh += dh_part
        dws.append(dw)
    torch.cuda.synchronize()
    out = dict(loss=loss.double().cpu().numpy(), lse=lse.double().cpu().numpy(), counts=counts.cpu().numpy(),
               dH=dh.double().cpu().numpy(),
               dW=S.bf16_bits_to_f32(P.bf16_bits(torch.cat(dws))).astype(np.float64))
    return out


@pytest.mark.parametrize("softcap,reduction", [(0.0, "mean"), (30.0, "none"), (0.0, "sum")])
def test_three_ragged_shards_match_the_unsharded_oracle(softcap, reduction):
    w = S.scaled("llama3", N=300, Hd=72, V=3001, seed=71, w_std=0.1, softcap=softcap)
    Hb, Wb, y = P.make_case(w)
    y[3] = 5000  # out of range for the whole vocabulary: bad everywhere
    out = _sharded(Hb, Wb, y, cuts=(1000, 2337), softcap=softcap, reduction=reduction)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, softcap=softcap, reduction=reduction)
    valid, bad = O.label_status(y, w.V, -100)
    assert int(out["counts"][0]) == ref.n_valid and int(out["counts"][1]) == ref.n_bad == 1
    assert np.abs(out["lse"] - ref.lse).max() <= P.TOL_LSE_ABS
    if reduction == "none":
        assert np.abs(out["loss"] - np.asarray(ref.loss)).max() <= P.TOL_LSE_ABS + P.TOL_TARGET_ABS
    else:
        assert abs(float(out["loss"]) - float(ref.loss)) <= P.TOL_LOSS_REL * abs(float(ref.loss))
    assert P.fro_rel(out["dH"], dH) <= P.TOL_GRAD_FRO
    assert P.fro_rel(out["dW"], dW) <= P.TOL_GRAD_FRO
    P.check_rows("dH", out["dH"], dH)
    P.check_rows("dW", out["dW"], dW)


def test_chunked_shards_and_single_shard():
    w = S.scaled("llama2", N=260, Hd=128, V=2600, seed=72, w_std=0.05)
    Hb, Wb, y = P.make_case(w)
    ref, dH, dW = P.oracle_full(Hb, Wb, y)
    for cuts, budget in (((700,), 260 * 2 * 512), ((), 0)):
        out = _sharded(Hb, Wb, y, cuts=cuts, chunk_budget=budget)
        assert abs(float(out["loss"]) - float(ref.loss)) <= P.TOL_LOSS_REL * float(ref.loss)
        assert P.fro_rel(out["dH"], dH) <= P.TOL_GRAD_FRO and P.fro_rel(out["dW"], dW) <= P.TOL_GRAD_FRO
        P.check_rows("dH", out["dH"], dH)
        P.check_rows("dW", out["dW"], dW)


def test_sharded_filtered_matches_filtered_oracle():
    w = S.scaled("peaked", N=256, Hd=128, V=2400, seed=73, w_std=0.1)
    Hb, Wb, y = P.make_case(w)
    thr = 2.0 ** -12
    out = _sharded(Hb, Wb, y, cuts=(1200,), filter_threshold=thr)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, filter_threshold=thr)
    assert P.fro_rel(out["dH"], dH) <= P.TOL_GRAD_FRO and P.fro_rel(out["dW"], dW) <= P.TOL_GRAD_FRO
    P.check_rows("dH", out["dH"], dH)
    P.check_rows("dW", out["dW"], dW)
