"""Token-sharded data parallel with the CUDA kernels, the ranks emulated one after
another on one GPU.

Each "rank" holds all of W and a contiguous slice of the rows.  Per rank: flce_forward
with reduction="sum"; then, on the device, what the all-reduce of
linear_cross_entropy_indexed_gb300.dist.allreduce_counts_ leaves on every rank
(valid and bad counts summed over the ranks, error bits combined with a max) and the
global mean of global_mean_loss (the summed per-row losses divided once by the global
valid count, the "n_items" rule of the Unsloth notes §4); then flce_backward with
reduction="mean", which reads the global count from counts[0]; dW is summed over the
ranks as the data-parallel all-reduce would.  The loss, every rank's dH rows and the
summed dW must equal the unsharded fp64 oracle, also when one rank's rows are all
ignored (its gradient is zero, and it still gets the global loss)."""
import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _sharded_step(Hb, Wb, y, cuts, softcap=0.0, grad=1.25, chunk_budget=0):
    import linear_cross_entropy_indexed_gb300 as F
    W = P.to_device(Wb)
    bounds = [0] + list(cuts) + [len(y)]
    ranks = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        H = P.to_device(Hb[a:b])
        lab = torch.from_numpy(np.ascontiguousarray(y[a:b])).cuda()
        loss_sum, lse, counts, _ = F.flce_forward(H, W, lab, -100, softcap, "sum")
        ranks.append(dict(a=a, b=b, H=H, lab=lab, loss_sum=loss_sum, lse=lse, counts=counts))
    # the exchange, on the device: no host synchronisation between the two passes
    head = torch.stack([r["counts"][0:2] for r in ranks]).sum(0)
    bits = torch.stack([r["counts"][2] for r in ranks]).max()
    total = torch.stack([r["loss_sum"].double() for r in ranks]).sum()
    n = head[0].double()
    loss = torch.where(n > 0, total / torch.clamp(n, min=1), torch.zeros_like(total))
    for r in ranks:
        r["counts"][0:2].copy_(head)
        r["counts"][2].copy_(bits)
    g = torch.tensor([grad], dtype=torch.float32, device="cuda")
    dW = torch.zeros(Wb.shape, dtype=torch.float64, device="cuda")
    dH = []
    for r in ranks:
        dh, dw = F.flce_backward(r["H"], W, r["lab"], r["lse"], r["counts"], g, -100, softcap, "mean",
                                 chunk_budget)
        dW += dw.double()      # the data-parallel sum of the ranks' dW
        dH.append(S.bf16_bits_to_f32(P.bf16_bits(dh)).astype(np.float64))
        r["dw"] = dw
    torch.cuda.synchronize()
    return dict(loss=float(loss), counts=[r["counts"].cpu().numpy() for r in ranks], dH=np.concatenate(dH),
                dW=dW.cpu().numpy(), dW_ranks=[r["dw"] for r in ranks], bounds=bounds)


def _check(out, Hb, Wb, y, softcap=0.0, grad=1.25):
    ref, dH, dW = P.oracle_full(Hb, Wb, y, softcap=softcap, grad=np.array([grad]))
    for c in out["counts"]:
        assert int(c[0]) == ref.n_valid and int(c[1]) == ref.n_bad and int(c[2]) == 0
    assert abs(out["loss"] - float(ref.loss)) <= P.TOL_LOSS_REL * abs(float(ref.loss))
    got = dict(dH=out["dH"], dW=out["dW"], counts_after=out["counts"][0])
    valid, _ = O.label_status(y, Wb.shape[0], -100)
    return ref, P.check_backward(got, dH, dW, no_grad_rows=~valid)


@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_two_ragged_row_shards_match_unsharded(softcap):
    w = S.scaled("llama3", N=600, Hd=136, V=3001, seed=91, w_std=0.1, softcap=softcap)
    Hb, Wb, y = P.make_case(w)
    out = _sharded_step(Hb, Wb, y, cuts=(257,), softcap=softcap)
    _check(out, Hb, Wb, y, softcap)


def test_three_shards_multi_chunk_backward():
    w = S.scaled("llama2", N=700, Hd=128, V=4000, seed=92, w_std=0.05)
    Hb, Wb, y = P.make_case(w)
    out = _sharded_step(Hb, Wb, y, cuts=(100, 450), chunk_budget=450 * 2 * 1024)
    _check(out, Hb, Wb, y)


def test_a_rank_with_every_row_ignored():
    w = S.scaled("llama3", N=520, Hd=128, V=2500, seed=93, w_std=0.1)
    Hb, Wb, y = P.make_case(w)
    y = y.copy()
    y[300:] = -100                       # the second rank's rows are all ignored
    out = _sharded_step(Hb, Wb, y, cuts=(300,))
    ref, _ = _check(out, Hb, Wb, y)
    assert ref.n_valid > 0
    assert torch.count_nonzero(out["dW_ranks"][1]).item() == 0
    assert np.all(out["dH"][300:] == 0.0)
