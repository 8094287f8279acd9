"""Shared helpers of the GPU parity tests: seeded inputs, the CUDA path through the
C ABI (via the binding), and comparisons with the fp64 oracle.

Tolerances (fp32 accumulation of bf16 products, bf16 gradient outputs):
  loss      relative error <= 1e-3; where the exact loss is 0 with valid rows (V = 1),
            absolute error <= (2e-3 + 1e-3) per reduced row; all rows ignored: exactly 0
  lse       absolute error <= 2e-3 per row
  target    absolute error <= 1e-3 per valid row (the indexed-dot output)
  dH, dW    relative Frobenius error <= 1e-2, and per row (a token row of dH, a
            vocabulary row of dW) relative error <= 1e-2, a row's error measured against
            max(its reference norm, 1e-3 x the largest reference row norm) so that rows
            whose exact gradient is nearly zero are held to an absolute bound instead.
            Derivation: each dZ entry is rounded to bf16 once (relative 2^-9) and each
            output element once more (2^-9); a row whose terms all round the same way
            is off by at most about 2 x 2^-9 = 3.9e-3 relative, fp32 accumulation adds
            ~1e-6.  The per-row bound catches what the global norm hides: one wrong
            256 x 256 output tile is 1/512 of an 8192 x 4096 dH but most of a row.
  counts    bit-exact
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synthetic as S

TOL_LOSS_REL = 1e-3
TOL_LSE_ABS = 2e-3
TOL_TARGET_ABS = 1e-3
TOL_GRAD_FRO = 1e-2
TOL_GRAD_ROW = 1e-2
ROW_FLOOR = 1e-3


def to_device(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def fro_rel(a: np.ndarray, ref: np.ndarray) -> float:
    num = np.linalg.norm((a - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    return float(num / den) if den > 0 else float(num)


def row_rel_max(a: np.ndarray, ref: np.ndarray, floor_frac: float = ROW_FLOOR) -> float:
    """Largest per-row error ||a_r - ref_r|| / max(||ref_r||, floor_frac * max_r ||ref_r||)
    (absolute when every reference row is zero)."""
    if a.size == 0:
        return 0.0
    num = np.linalg.norm(a - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    top = den.max()
    if top == 0:
        return float(num.max())
    return float((num / np.maximum(den, floor_frac * top)).max())


def check_rows(name: str, got: np.ndarray, ref: np.ndarray, tol: float = TOL_GRAD_ROW) -> float:
    e = row_rel_max(got, ref)
    if e > tol:
        num = np.linalg.norm(got - ref, axis=1)
        den = np.maximum(np.linalg.norm(ref, axis=1), ROW_FLOOR * np.linalg.norm(ref, axis=1).max())
        worst = np.argsort(-(num / den))[:5]
        raise AssertionError("%s per-row rel err %g > %g (worst rows %s: %s)" % (
            name, e, tol, worst.tolist(), (num / den)[worst].tolist()))
    return e


def make_case(w: S.Workload, labels: np.ndarray | None = None):
    Wb = S.make_W(w)
    Hb = S.make_H(w, W=Wb)
    y = S.make_labels(w) if labels is None else labels
    return Hb, Wb, y


def run_gpu(Hb, Wb, y, ignore_index=-100, softcap=0.0, reduction="mean", grad=None, chunk_budget=0,
            backward=True, filter_threshold=0.0, sort_vocab=False, compensated=False):
    import linear_cross_entropy_indexed_gb300 as F
    H = to_device(Hb)
    W = to_device(Wb)
    lab = torch.from_numpy(np.asarray(y, dtype=np.int64)).cuda()
    loss, lse, counts, tgt = F.flce_forward(H, W, lab, ignore_index, softcap, reduction, want_target=True)
    out = dict(loss=loss.double().cpu().numpy(), lse=lse.double().cpu().numpy(), counts=counts.cpu().numpy(),
               target=tgt.double().cpu().numpy())
    if backward:
        N = H.shape[0]
        if grad is None:
            grad = np.linspace(0.5, 1.5, N) if reduction == "none" else np.array([1.0])
        g = torch.tensor(np.asarray(grad, dtype=np.float32)).cuda()
        dH, dW = F.flce_backward(H, W, lab, lse, counts, g, ignore_index, softcap, reduction, chunk_budget,
                                 filter_threshold=filter_threshold, sort_vocab=sort_vocab, compensated=compensated)
        out["dH"] = S.bf16_bits_to_f32(bf16_bits(dH)).astype(np.float64)
        out["dW"] = S.bf16_bits_to_f32(bf16_bits(dW)).astype(np.float64)
        out["counts_after"] = counts.cpu().numpy()
    torch.cuda.synchronize()
    return out


def check_forward(out, ref: O.Forward, y, V, ignore_index=-100, reduction="mean"):
    valid, bad = O.label_status(y, V, ignore_index)
    assert int(out["counts"][0]) == ref.n_valid, (out["counts"], ref.n_valid)
    assert int(out["counts"][1]) == ref.n_bad
    assert int(out["counts"][2]) == 0, "device error bits set"
    lse_err = np.abs(out["lse"] - ref.lse).max() if len(ref.lse) else 0.0
    assert lse_err <= TOL_LSE_ABS, "lse abs err %g" % lse_err
    t_err = np.abs(out["target"] - ref.target)[valid].max() if valid.any() else 0.0
    assert t_err <= TOL_TARGET_ABS, "target abs err %g" % t_err
    assert np.all(out["target"][~valid] == 0)
    if reduction == "none":
        ref_l = np.asarray(ref.loss)
        err = np.abs(out["loss"] - ref_l).max() if len(ref_l) else 0.0
        assert err <= TOL_LSE_ABS + TOL_TARGET_ABS, "per-row loss err %g" % err
        assert np.all(out["loss"][~valid] == 0)
    else:
        ref_l = float(ref.loss)
        got = float(out["loss"])
        if ref.n_valid == 0:
            assert got == 0.0  # all rows ignored: zero by convention, exactly
        elif ref_l == 0.0:
            # every valid row's loss is exactly zero (V = 1: lse = z = target), so a relative
            # error is undefined; bound it by the per-row lse and target tolerances summed
            # over the rows the reduction adds up
            rows = ref.n_valid if reduction == "sum" else 1
            assert abs(got) <= rows * (TOL_LSE_ABS + TOL_TARGET_ABS), got
        else:
            assert abs(got - ref_l) / abs(ref_l) <= TOL_LOSS_REL, (got, ref_l)
    return dict(lse_err=float(lse_err), target_err=float(t_err))


def check_backward(out, dH_ref, dW_ref, no_grad_rows=None):
    """Frobenius and per-row bounds on dH and dW; `no_grad_rows` (a boolean mask of
    ignored or bad-label rows) must come out exactly zero in dH."""
    eh = fro_rel(out["dH"], dH_ref)
    ew = fro_rel(out["dW"], dW_ref)
    assert np.isfinite(out["dH"]).all() and np.isfinite(out["dW"]).all()
    assert eh <= TOL_GRAD_FRO, "dH rel fro err %g" % eh
    assert ew <= TOL_GRAD_FRO, "dW rel fro err %g" % ew
    rh = check_rows("dH", out["dH"], dH_ref)
    rw = check_rows("dW", out["dW"], dW_ref)
    if no_grad_rows is not None and np.any(no_grad_rows):
        assert np.all(out["dH"][np.asarray(no_grad_rows)] == 0.0), "an ignored row has a non-zero dH"
    assert int(out["counts_after"][2]) == 0, "device error bits set"
    return dict(dH_err=eh, dW_err=ew, dH_row_err=rh, dW_row_err=rw)


def oracle_full(Hb, Wb, y, ignore_index=-100, softcap=0.0, reduction="mean", grad=None, filter_threshold=0.0):
    Hf = O.widen_bf16(Hb)
    Wf = O.widen_bf16(Wb)
    ref = O.forward(Hf, Wf, y, ignore_index, softcap, reduction)
    N = Hf.shape[0]
    if grad is None:
        grad = np.linspace(0.5, 1.5, N) if reduction == "none" else 1.0
    g = np.asarray(grad, dtype=np.float32).astype(np.float64)
    if reduction != "none":
        g = float(np.asarray(g).reshape(-1)[0])
    dH, dW = O.backward(Hf, Wf, y, ref.lse, ignore_index, softcap, reduction, g, filter_threshold=filter_threshold)
    return ref, dH, dW
