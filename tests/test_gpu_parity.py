"""Element-by-element parity of the CUDA path (through the C ABI) with the fp64
oracle on seeded inputs small enough for the oracle to finish in seconds.  The cases
span several 128 x 256 tiles with ragged tails in N, Hd and V, every reduction, the
softcap, ignored / bad / all-ignored labels, a chunked backward and N = 0."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _run_and_check(w, y=None, reduction="mean", softcap=None, chunk_budget=0, grad=None, ignore_index=-100):
    Hb, Wb, yy = P.make_case(w, y)
    cap = w.softcap if softcap is None else softcap
    out = P.run_gpu(Hb, Wb, yy, ignore_index, cap, reduction, grad=grad, chunk_budget=chunk_budget)
    ref, dH, dW = P.oracle_full(Hb, Wb, yy, ignore_index, cap, reduction, grad=grad)
    f = P.check_forward(out, ref, yy, w.V, ignore_index, reduction)
    valid, _ = O.label_status(yy, w.V, ignore_index)
    b = P.check_backward(out, dH, dW, no_grad_rows=~valid)
    return out, ref, f, b


def test_tiny_config():
    """The small workload in full: N=256, Hd=64, V=2000 (V not a tile multiple)."""
    _run_and_check(S.WORKLOADS["tiny"])


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_ragged_shapes(reduction):
    # N, Hd and V all off the 128 / 64 / 256 tile grid
    w = S.scaled("tiny", N=300, Hd=72, V=1000, seed=11, ignore_frac=0.1)
    _run_and_check(w, reduction=reduction)


def test_several_tiles_uniform():
    w = S.scaled("llama2", N=520, Hd=264, V=3001, seed=12, w_std=0.05)
    _run_and_check(w)


def test_softcap_large_logits():
    # W std 0.5 at Hd 256 gives logits of std ~8, so the cap at 30 bends them
    w = S.scaled("gemma2", N=384, Hd=256, V=2600, seed=13, w_std=0.5)
    out, ref, f, b = _run_and_check(w)
    assert w.softcap == 30.0


def test_zipf_none_reduction_with_grad_vector():
    w = S.scaled("llama3", N=257, Hd=128, V=4099, seed=14)
    g = np.linspace(-1.0, 2.0, 257)
    _run_and_check(w, reduction="none", grad=g)


def test_chunked_backward_ragged_tail():
    # budget for 768 columns of dZ -> 7 vocabulary chunks, the last one partial
    w = S.scaled("llama2", N=384, Hd=128, V=5000, seed=15, w_std=0.05)
    _run_and_check(w, chunk_budget=384 * 2 * 768)


def test_chunked_backward_with_softcap():
    w = S.scaled("gemma2", N=200, Hd=96, V=3000, seed=16, w_std=0.3)
    _run_and_check(w, chunk_budget=200 * 2 * 512)


def test_packed_labels_small():
    w = S.scaled("packed", N=2 * 512, Hd=64, V=3000, seed=17, n_seq=2, seq_len=512, n_docs=4)
    y = S.make_labels(w)
    assert (y == -100).sum() == 8
    _run_and_check(w, y=y)


def test_bad_and_ignored_labels():
    w = S.scaled("tiny", N=130, Hd=64, V=700, seed=18)
    y = S.make_labels(w)
    y[0] = 700          # out of range
    y[5] = -3           # negative, not ignore_index
    y[6] = -100
    out, ref, f, b = _run_and_check(w, y=y)
    assert int(out["counts"][1]) == 2
    assert np.abs(out["dH"][[0, 5, 6]]).max() == 0.0


def test_custom_ignore_index():
    w = S.scaled("tiny", N=140, Hd=64, V=600, seed=19)
    y = S.make_labels(w)
    y[y == -100] = 5
    _run_and_check(w, y=y, ignore_index=5)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_all_ignored(reduction):
    w = S.scaled("tiny", N=150, Hd=64, V=500, seed=20)
    y = np.full(150, -100, dtype=np.int64)
    Hb, Wb, _ = P.make_case(w)
    out = P.run_gpu(Hb, Wb, y, reduction=reduction)
    assert float(out["loss"]) == 0.0
    assert int(out["counts"][0]) == 0
    assert np.abs(out["dH"]).max() == 0.0 and np.abs(out["dW"]).max() == 0.0
    ref = O.forward(O.widen_bf16(Hb), O.widen_bf16(Wb), y)
    assert np.abs(out["lse"] - ref.lse).max() <= P.TOL_LSE_ABS


def test_single_row_single_class():
    w = S.scaled("tiny", N=1, Hd=8, V=1, seed=21)
    y = np.array([0])
    out, ref, f, b = _run_and_check(w, y=y)
    assert abs(float(out["loss"])) < 1e-5


def test_zero_rows():
    import linear_cross_entropy_indexed_gb300 as F
    H = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = P.to_device(S.make_W(S.scaled("tiny", V=300)))
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    loss, lse, counts, _ = F.flce_forward(H, W, y)
    dH, dW = F.flce_backward(H, W, y, lse, counts, torch.ones(1, device="cuda"))
    torch.cuda.synchronize()
    assert float(loss) == 0.0 and counts.tolist() == [0, 0, 0]
    assert dW.abs().max().item() == 0.0


def test_worked_example_on_gpu():
    """The pages' worked example through the kernels: Hd=8, H row = e0, W[v] =
    bf16(ln(v+1)) e0, target 2; compared with the closed form on the bf16 values."""
    import math
    z = np.log(np.array([1.0, 2.0, 3.0, 4.0], dtype=np.float32))
    zb = S.f32_to_bf16_bits(z)
    Wb = np.zeros((4, 8), dtype=np.uint16)
    Wb[:, 0] = zb
    Hb = np.zeros((1, 8), dtype=np.uint16)
    Hb[0, 0] = S.f32_to_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    out = P.run_gpu(Hb, Wb, np.array([2]))
    zz = S.bf16_bits_to_f32(zb).astype(np.float64)
    expect = math.log(np.exp(zz).sum()) - zz[2]
    assert abs(float(out["loss"]) - expect) < 1e-5
    assert abs(expect - math.log(10 / 3)) < 5e-3   # bf16 rounding of ln(v+1)


def test_deterministic():
    w = S.scaled("llama2", N=300, Hd=128, V=3000, seed=22, w_std=0.05)
    Hb, Wb, y = P.make_case(w)
    a = P.run_gpu(Hb, Wb, y, chunk_budget=300 * 2 * 1024)
    b = P.run_gpu(Hb, Wb, y, chunk_budget=300 * 2 * 1024)
    for k in ("loss", "lse", "target", "dH", "dW"):
        assert np.array_equal(a[k], b[k]), k


def test_autograd_function():
    import linear_cross_entropy_indexed_gb300 as F
    w = S.scaled("tiny", N=2 * 96, Hd=64, V=900, seed=23)
    Hb, Wb, y = P.make_case(w)
    H = P.to_device(Hb).reshape(2, 96, 64).requires_grad_(True)
    W = P.to_device(Wb).requires_grad_(True)
    lab = torch.from_numpy(y).cuda().reshape(2, 96)
    loss = F.linear_cross_entropy(H, W, lab)
    (2.0 * loss).backward()
    ref, dH, dW = P.oracle_full(Hb, Wb, y, grad=2.0)
    assert abs(loss.item() - float(ref.loss)) / float(ref.loss) <= P.TOL_LOSS_REL
    gh = S.bf16_bits_to_f32(P.bf16_bits(H.grad.reshape(-1, 64))).astype(np.float64)
    gw = S.bf16_bits_to_f32(P.bf16_bits(W.grad)).astype(np.float64)
    assert P.fro_rel(gh, dH) <= P.TOL_GRAD_FRO and P.fro_rel(gw, dW) <= P.TOL_GRAD_FRO


def test_invariant_vocab_sum_of_dW():
    """Without softcap, sum_v dZ_iv = 0 per valid row, so sum_v dW_v ~ 0 (bf16)."""
    w = S.scaled("tiny", N=256, Hd=64, V=1500, seed=24)
    Hb, Wb, y = P.make_case(w)
    out = P.run_gpu(Hb, Wb, y, reduction="sum")
    col = out["dW"].sum(axis=0)
    assert np.abs(col).max() <= 1e-2 * np.abs(out["dW"]).sum(axis=0).max()
