"""The compensated backward (FLCE_BWD_COMPENSATED) on the GPU.

Each dZ entry is carried as its bf16 value plus the bf16 rounding remainder, and dH and
dW accumulate both.  The gradients are compared with the fp64 oracle's exact gradients:
they must pass the usual tolerance and beat the plain bf16-dZ backward on the same
inputs.  With bf16 outputs the floor is the outputs' own rounding (the error of the
oracle's gradient rounded to bf16), which the compensated backward must reach; the
vocabulary-shard call returns dH in fp32, where the remainder removes almost all of the
error."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _floor(ref):
    """Relative Frobenius error of the exact gradient rounded to bf16 (nearest even)."""
    r = S.bf16_bits_to_f32(S.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    return P.fro_rel(r, ref)


def _check(e_plain, e_comp, floors):
    for k, f in zip(("dH_err", "dW_err"), floors):
        assert e_comp[k] <= 1.1 * f + 1e-6, (k, e_comp[k], f)
        assert e_comp[k] <= 1.02 * e_plain[k], k


def _both(w, chunk_budget=0, reduction=None, sort_vocab=False):
    red = w.reduction if reduction is None else reduction
    Hb, Wb, y = P.make_case(w)
    plain = P.run_gpu(Hb, Wb, y, w.ignore_index, w.softcap, red, chunk_budget=chunk_budget)
    comp = P.run_gpu(Hb, Wb, y, w.ignore_index, w.softcap, red, chunk_budget=chunk_budget, compensated=True,
                     sort_vocab=sort_vocab)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, w.ignore_index, w.softcap, red)
    P.check_forward(comp, ref, y, w.V, w.ignore_index, red)
    assert int(comp["counts_after"][2]) == 0
    e_plain = P.check_backward(plain, dH, dW)
    e_comp = P.check_backward(comp, dH, dW)
    floors = (_floor(dH), _floor(dW))
    print("\n%s plain %s compensated %s bf16 floor %s" % (w.name, e_plain, e_comp, floors))
    return e_plain, e_comp, floors


@pytest.mark.parametrize("name,softcap,reduction", [("llama3", 0.0, "mean"), ("gemma2", 30.0, "none"),
                                                    ("tiny", 0.0, "sum")])
def test_compensated_beats_plain(name, softcap, reduction):
    # ragged N, Hd and V; 4 vocabulary chunks (Vc = budget / 4N), the last ragged
    w = S.scaled(name, N=300, Hd=136, V=3500, seed=81, softcap=softcap, w_std=0.3 if softcap else 0.05)
    _check(*_both(w, chunk_budget=4 * 300 * 1024, reduction=reduction))


def test_compensated_with_sorted_vocabulary():
    w = S.scaled("unigram", N=256, Hd=128, V=5000, seed=82)
    _check(*_both(w, chunk_budget=(4 * 256 + 2 * 128) * 1024, sort_vocab=True))


def test_compensated_fp32_shard_partial():
    """The shard call's fp32 dH partial: the remainder takes the error from the bf16 dZ
    level (~1e-3) to the fp32 accumulation level."""
    import linear_cross_entropy_indexed_gb300 as F
    w = S.scaled("llama3", N=256, Hd=128, V=4000, seed=83, w_std=0.05)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    g = torch.ones(1, device="cuda")
    out = {}
    for comp in (False, True):
        dh, dw = F.flce_backward_shard(H, W, lab, lse, counts, g, 0, w.V, chunk_budget=4 * 256 * 1024,
                                       compensated=comp)
        torch.cuda.synchronize()
        out[comp] = dh.double().cpu().numpy()
    ref, dH, dW = P.oracle_full(Hb, Wb, y)
    e_plain, e_comp = P.fro_rel(out[False], dH), P.fro_rel(out[True], dH)
    print("\nfp32 dH partial: plain %.3g compensated %.3g" % (e_plain, e_comp))
    assert e_comp <= 1e-4 and e_comp < 0.1 * e_plain


def test_compensated_rejects_filtering():
    import linear_cross_entropy_indexed_gb300 as F
    w = S.scaled("tiny", N=64, Hd=64, V=500, seed=84)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    before = F.launch_count()
    with pytest.raises(F.FlceError, match="invalid argument"):
        F.flce_backward(H, W, lab, lse, counts, torch.ones(1, device="cuda"), filter_threshold=2.0 ** -12,
                        compensated=True)
    assert F.launch_count() == before


def test_full_size_llama3_compensated():
    """bench.py's llama3 workload with the compensated backward: sampled dH rows and dW rows
    against the oracle, next to the plain backward's errors on the same samples."""
    import linear_cross_entropy_indexed_gb300 as F
    w = S.WORKLOADS["llama3"]
    Hb, Wb, y = S.make_H(w), S.make_W(w), S.make_labels(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    g = torch.ones(1, device="cuda")
    rng = np.random.default_rng(85)
    rows = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, 46, replace=False)]))
    vs = np.unique(np.concatenate([rng.choice(w.V, 64, replace=False), np.arange(w.V - 16, w.V)]))
    got = {}
    for comp in (False, True):
        dH, dW = F.flce_backward(H, W, lab, lse, counts, g, compensated=comp)
        torch.cuda.synchronize()
        got[comp] = (S.bf16_bits_to_f32(P.bf16_bits(dH[torch.from_numpy(rows).cuda()])).astype(np.float64),
                     S.bf16_bits_to_f32(P.bf16_bits(dW[torch.from_numpy(vs).cuda()])).astype(np.float64))
        del dH, dW
    assert int(counts[2]) == 0
    Hf, Wf = O.widen_bf16(Hb), O.widen_bf16(Wb)
    ref = O.forward(Hf, Wf, y, row_block=1024)
    dh_ref = O.dH_rows(Hf, Wf, y, ref.lse[rows], rows, n_valid=ref.n_valid)
    dw_ref = O.dW_rows(Hf, Wf, y, ref.lse, vs)
    e = {c: (P.fro_rel(got[c][0], dh_ref), P.fro_rel(got[c][1], dw_ref)) for c in got}
    floors = (_floor(dh_ref), _floor(dw_ref))
    print("\nllama3 full size: plain dH %.3g dW %.3g; compensated dH %.3g dW %.3g; bf16 floor %.3g %.3g" % (
        e[False] + e[True] + floors))
    _check(dict(dH_err=e[False][0], dW_err=e[False][1]), dict(dH_err=e[True][0], dW_err=e[True][1]), floors)
    assert max(e[True]) <= P.TOL_GRAD_FRO
    for c in got:
        P.check_rows("dH", got[c][0], dh_ref)
        P.check_rows("dW", got[c][1], dw_ref)


def test_compensated_all_ignored_and_bad_labels():
    w = S.scaled("tiny", N=130, Hd=64, V=700, seed=86)
    Hb, Wb, y = P.make_case(w)
    y = np.full(130, -100, dtype=np.int64)
    out = P.run_gpu(Hb, Wb, y, compensated=True)
    assert np.abs(out["dH"]).max() == 0.0 and np.abs(out["dW"]).max() == 0.0
    y = S.make_labels(w)
    y[0] = 700
    out = P.run_gpu(Hb, Wb, y, compensated=True, reduction="sum")
    ref, dH, dW = P.oracle_full(Hb, Wb, y, reduction="sum")
    P.check_backward(out, dH, dW)
    assert int(out["counts"][1]) == 1 and np.abs(out["dH"][0]).max() == 0.0
