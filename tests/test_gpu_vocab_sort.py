"""Vocabulary sorting (FLCE_BWD_SORT_VOCAB) on the GPU.

flce_vocab_order's keys are compared with the oracle's mean raw logits, and its
permutation bit for bit with the oracle's order of the GPU's own fp32 keys (the float
keys decide the integer order, so both sides take that decision on the same values);
independently of the GPU keys, the oracle's keys taken in the permutation's order must
not rise by more than the key tolerance.
The sorted backward is compared element by element with the oracle's gradients, exact
and filtered; it computes the same sums in another order.  Cases span several sort
runs (4096 words each) and merge passes, ragged vocabulary chunks, the softcap and a
vocabulary shard; one case runs the full unigram workload."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

THR = 2.0 ** -12


def _order_gpu(Hb, Wb):
    import linear_cross_entropy_indexed_gb300 as F
    keys, perm, inv = F.vocab_order(P.to_device(Hb), P.to_device(Wb))
    torch.cuda.synchronize()
    return keys.cpu().numpy(), perm.cpu().numpy().astype(np.int64), inv.cpu().numpy().astype(np.int64)


def _check_order(Hb, Wb, vocab=None):
    keys, perm, inv = _order_gpu(Hb, Wb)
    V = Wb.shape[0]
    Hf, Wf = O.widen_bf16(Hb), O.widen_bf16(Wb)
    vs = np.arange(V) if vocab is None else vocab
    ref = O.vocab_keys(Hf, Wf, vs)
    # fp32 column mean then fp32 dot: error bounded by a few ulps of |hbar| |w_v|
    hbar = Hf.mean(axis=0) if Hf.shape[0] else np.zeros(Hf.shape[1])
    scale = np.linalg.norm(hbar) * np.linalg.norm(Wf[vs], axis=1) + np.abs(Wf[vs]).max(axis=1) * 1e-3
    err = np.abs(keys[vs].astype(np.float64) - ref)
    tol = 2e-5 * scale + 1e-7
    assert np.all(err <= tol), err.max()
    assert np.array_equal(perm, O.vocab_order(keys.astype(np.float64)))
    if vocab is None:
        # independently of the GPU keys: walked in perm order, the oracle's keys never rise
        # by more than the two entries' key tolerances
        rk, rt = ref[perm], tol[perm]
        rise = rk[1:] - rk[:-1] - (rt[1:] + rt[:-1])
        assert V < 2 or rise.max() <= 0.0, rise.max()
    assert np.array_equal(np.sort(perm), np.arange(V))
    assert np.array_equal(inv[perm], np.arange(V))
    return keys, perm


@pytest.mark.parametrize("name,N,Hd,V", [("tiny", 300, 72, 1000), ("unigram", 520, 264, 9001),
                                         ("unigram", 256, 128, 20000), ("llama3", 64, 64, 4096)])
def test_vocab_order_matches_oracle(name, N, Hd, V):
    w = S.scaled(name, N=N, Hd=Hd, V=V, seed=71)
    Hb, Wb, _ = P.make_case(w)
    _check_order(Hb, Wb)


def test_vocab_order_ties_and_no_rows():
    # duplicated weight rows give equal keys: ties keep ascending ids
    w = S.scaled("tiny", N=40, Hd=64, V=600, seed=72)
    Hb, Wb, _ = P.make_case(w)
    Wb[300:600] = Wb[0:300]
    keys, perm = _check_order(Hb, Wb)
    assert np.array_equal(keys[300:600], keys[0:300])
    # N = 0: every key is 0 and the order is the identity
    keys0, perm0, _ = _order_gpu(Hb[:0], Wb)
    assert np.all(keys0 == 0.0) and np.array_equal(perm0, np.arange(600))


def _sorted_case(w, thr, chunk_budget, reduction=None):
    red = w.reduction if reduction is None else reduction
    Hb, Wb, y = P.make_case(w)
    out = P.run_gpu(Hb, Wb, y, w.ignore_index, w.softcap, red, chunk_budget=chunk_budget, filter_threshold=thr,
                    sort_vocab=True)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, w.ignore_index, w.softcap, red, filter_threshold=thr,
                                grad=np.linspace(0.5, 1.5, w.N) if red == "none" else None)
    P.check_forward(out, ref, y, w.V, w.ignore_index, red)
    assert int(out["counts_after"][2]) == 0, "device error bits set"
    errs = P.check_backward(out, dH, dW)
    print("\n%s thr=%g sorted: %s" % (w.name, thr, errs))
    return Hb, Wb, y, out


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_sorted_exact_backward_multi_chunk(reduction):
    # 5 sorted chunks of 1024 positions, the last one ragged; filter off
    w = S.scaled("unigram", N=300, Hd=128, V=4500, seed=73)
    _sorted_case(w, 0.0, chunk_budget=(2 * 300 + 2 * 128) * 1024, reduction=reduction)


@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_sorted_filtered_backward(softcap):
    w = S.scaled("unigram", N=520, Hd=256, V=9001, seed=74, softcap=softcap)
    _sorted_case(w, THR, chunk_budget=(2 * 520 + 2 * 256) * 2048)


def test_sorted_equals_unsorted_up_to_order():
    """The sorted walk computes the same dW rows from the same dZ column values in the
    same token order, and dH over a permuted vocabulary order."""
    w = S.scaled("unigram", N=384, Hd=192, V=6000, seed=75)
    Hb, Wb, y = P.make_case(w)
    a = P.run_gpu(Hb, Wb, y, filter_threshold=THR, chunk_budget=(2 * 384 + 2 * 192) * 2048)
    b = P.run_gpu(Hb, Wb, y, filter_threshold=THR, chunk_budget=(2 * 384 + 2 * 192) * 2048, sort_vocab=True)
    assert P.fro_rel(b["dW"], a["dW"]) <= 1e-2 and P.fro_rel(b["dH"], a["dH"]) <= 1e-2
    print("\ndW identical: %s, dH rel diff %.3g" % (np.array_equal(a["dW"], b["dW"]), P.fro_rel(b["dH"], a["dH"])))


def test_sorted_backward_is_deterministic():
    w = S.scaled("unigram", N=260, Hd=128, V=5000, seed=76)
    Hb, Wb, y = P.make_case(w)
    a = P.run_gpu(Hb, Wb, y, filter_threshold=THR, chunk_budget=(2 * 260 + 2 * 128) * 1024, sort_vocab=True)
    b = P.run_gpu(Hb, Wb, y, filter_threshold=THR, chunk_budget=(2 * 260 + 2 * 128) * 1024, sort_vocab=True)
    assert np.array_equal(a["dH"], b["dH"]) and np.array_equal(a["dW"], b["dW"])


def test_sorted_vocab_shard():
    """A shard sorts its own rows; dH_partial and dW_shard against the oracle's
    filtered gradients restricted to the shard."""
    import linear_cross_entropy_indexed_gb300 as F
    w = S.scaled("unigram", N=256, Hd=128, V=5000, seed=77)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    off, vs = 1500, 2500
    g = torch.ones(1, device="cuda")
    dh_part, dw = F.flce_backward_shard(H, W[off:off + vs].contiguous(), lab, lse, counts, g, off, w.V,
                                        chunk_budget=(2 * 256 + 2 * 128) * 1024, filter_threshold=THR,
                                        sort_vocab=True)
    torch.cuda.synchronize()
    assert int(counts[2]) == 0
    Hf, Wf = O.widen_bf16(Hb), O.widen_bf16(Wb)
    ref = O.forward(Hf, Wf, y)
    valid, _ = O.label_status(y, w.V, -100)
    scale = O.row_scale(valid, ref.n_valid, "mean", 1.0)
    X = Hf @ Wf[off:off + vs].T
    Pm = np.exp(X - ref.lse[:, None])
    yl = np.where(valid & (y >= off) & (y < off + vs), y - off, -1)
    keep = (Pm >= THR)
    rows = np.nonzero(yl >= 0)[0]
    keep[rows, yl[rows]] = True
    D = np.where(keep, Pm, 0.0)
    D[rows, yl[rows]] -= 1.0
    D *= scale[:, None]
    dh_ref = D @ Wf[off:off + vs]
    dw_ref = D.T @ Hf
    assert P.fro_rel(dh_part.double().cpu().numpy(), dh_ref) <= P.TOL_GRAD_FRO
    P.check_rows("dH", dh_part.double().cpu().numpy(), dh_ref)
    got_w = S.bf16_bits_to_f32(P.bf16_bits(dw)).astype(np.float64)
    assert P.fro_rel(got_w, dw_ref) <= P.TOL_GRAD_FRO
    P.check_rows("dW", got_w, dw_ref)


def test_full_size_unigram_order_and_sorted_gradients():
    """The full unigram workload in bench.py's configuration with filtering and the
    sorted vocabulary: the whole permutation against the oracle's order of the GPU
    keys, 256 sampled keys against the oracle, the loss and every row's LSE, and dH / dW
    on sampled rows against the oracle's filtered gradients."""
    import linear_cross_entropy_indexed_gb300 as F
    w = S.WORKLOADS["unigram"]
    Wb = S.make_W(w)
    Hb, y = S.make_H(w, W=Wb), S.make_labels(w)
    rng = np.random.default_rng(78)
    vs = np.unique(np.concatenate([rng.choice(w.V, 200, replace=False), np.arange(56)]))
    _check_order(Hb, Wb, vocab=vs)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    dH, dW = F.flce_backward(H, W, lab, lse, counts, torch.ones(1, device="cuda"), filter_threshold=THR,
                             sort_vocab=True)
    torch.cuda.synchronize()
    assert int(counts[2]) == 0
    Hf, Wf = O.widen_bf16(Hb), O.widen_bf16(Wb)
    ref = O.forward(Hf, Wf, y, row_block=1024)
    assert np.abs(lse.double().cpu().numpy() - ref.lse).max() <= P.TOL_LSE_ABS
    assert abs(float(loss) - float(ref.loss)) / float(ref.loss) <= P.TOL_LOSS_REL
    rows = np.unique(np.concatenate([[0, w.N - 1], rng.choice(w.N, 62, replace=False)]))
    dh_ref = O.dH_rows(Hf, Wf, y, ref.lse[rows], rows, n_valid=ref.n_valid, filter_threshold=THR)
    dh_got = S.bf16_bits_to_f32(P.bf16_bits(dH[torch.from_numpy(rows).cuda()])).astype(np.float64)
    dw_ref = O.dW_rows(Hf, Wf, y, ref.lse, vs, filter_threshold=THR)
    dw_got = S.bf16_bits_to_f32(P.bf16_bits(dW[torch.from_numpy(vs).cuda()])).astype(np.float64)
    print("\nunigram full size, filtered + sorted: dH rel fro %.3g, dW rel fro %.3g" % (
        P.fro_rel(dh_got, dh_ref), P.fro_rel(dw_got, dw_ref)))
    assert P.fro_rel(dh_got, dh_ref) <= P.TOL_GRAD_FRO
    assert P.fro_rel(dw_got, dw_ref) <= P.TOL_GRAD_FRO
    P.check_rows("dH", dh_got, dh_ref)
    P.check_rows("dW", dw_got, dw_ref)


def test_sorted_with_bad_labels_and_custom_ignore_index():
    """Labels are mapped to positions only when valid: out-of-range and ignored rows keep no
    one-hot and no gradient under the sorted walk."""
    w = S.scaled("unigram", N=200, Hd=64, V=3000, seed=79)
    Hb, Wb, y = P.make_case(w)
    y = y.copy()
    y[y == -100] = 7          # 7 becomes the ignore index
    y[3] = 3000               # out of range
    y[4] = -5                 # negative, not the ignore index
    out = P.run_gpu(Hb, Wb, y, 7, 0.0, "sum", filter_threshold=THR, sort_vocab=True, chunk_budget=(2 * 200 + 2 * 64) * 1024)
    ref, dH, dW = P.oracle_full(Hb, Wb, y, 7, 0.0, "sum", filter_threshold=THR)
    P.check_forward(out, ref, y, w.V, 7, "sum")
    P.check_backward(out, dH, dW)
    assert int(out["counts"][1]) == 2
    assert np.abs(out["dH"][[3, 4]]).max() == 0.0


def test_sorted_all_ignored_is_zero():
    w = S.scaled("tiny", N=150, Hd=64, V=900, seed=80)
    Hb, Wb, _ = P.make_case(w)
    y = np.full(150, -100, dtype=np.int64)
    out = P.run_gpu(Hb, Wb, y, sort_vocab=True)
    assert np.abs(out["dH"]).max() == 0.0 and np.abs(out["dW"]).max() == 0.0
    assert int(out["counts_after"][2]) == 0
