"""User-facing API on the GPU: the module form, argument checks of the binding, a
whole forward + backward step captured in a CUDA graph and replayed, and the lazy,
synchronisation-free report of bad labels in the autograd path."""
import numpy as np
import pytest
import torch

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_module_matches_function_and_oracle():
    import linear_cross_entropy_indexed_gb300 as F
    w = S.scaled("gemma2", N=200, Hd=96, V=1500, seed=81, w_std=0.3)
    Hb, Wb, y = P.make_case(w)
    H = P.to_device(Hb).requires_grad_(True)
    W = P.to_device(Wb).requires_grad_(True)
    lab = torch.from_numpy(y).cuda()
    m = F.FusedLinearCrossEntropyLoss(softcap=w.softcap)
    loss = m(W, H, lab)
    loss.backward()
    ref, dH, dW = P.oracle_full(Hb, Wb, y, softcap=w.softcap)
    assert abs(loss.item() - float(ref.loss)) <= P.TOL_LOSS_REL * float(ref.loss)
    gh = S.bf16_bits_to_f32(P.bf16_bits(H.grad)).astype(np.float64)
    gw = S.bf16_bits_to_f32(P.bf16_bits(W.grad)).astype(np.float64)
    assert P.fro_rel(gh, dH) <= P.TOL_GRAD_FRO and P.fro_rel(gw, dW) <= P.TOL_GRAD_FRO
    assert "softcap=30" in repr(m)


def test_binding_rejects_bad_inputs():
    import linear_cross_entropy_indexed_gb300 as F
    H = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(10, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(F.FlceError):
        F.flce_forward(H.float(), W, y)
    with pytest.raises(F.FlceError):
        F.flce_forward(H, W[:, :32], y)
    with pytest.raises(F.FlceError):
        F.flce_forward(H, W, y.int())
    with pytest.raises(F.FlceError):
        F.flce_forward(H[:, :60], W[:, :60], y)  # hidden size not a multiple of 8
    with pytest.raises(ValueError):
        F.flce_forward(H, W, y, reduction="avg")
    y[0] = 10
    loss, lse, counts, _ = F.flce_forward(H, W, y)
    with pytest.raises(F.FlceError):
        F.check_counts(counts)  # one label outside [0, V)


@pytest.mark.parametrize("mode", ["exact", "filtered_sorted", "compensated"])
def test_step_captured_in_a_cuda_graph(mode):
    """Forward + backward through the C ABI captured once and replayed: the library
    neither allocates nor synchronises, so the graph replays the same kernels (also with
    the vocabulary order's sort and gather kernels, and with the compensated split)."""
    import linear_cross_entropy_indexed_gb300 as F
    opts = dict(exact={}, filtered_sorted=dict(filter_threshold=2.0 ** -12, sort_vocab=True),
                compensated=dict(compensated=True))[mode]
    w = S.scaled("unigram" if mode == "filtered_sorted" else "llama2", N=384, Hd=128, V=3000, seed=82, w_std=0.05)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    N, Hd, V = 384, 128, 3000
    budget = 384 * 2 * 1024
    ws = torch.empty(max(F.forward_workspace_size(N, Hd, V),
                         F.backward_workspace_size(N, Hd, V, budget, opts.get("sort_vocab", False),
                                                   opts.get("compensated", False))),
                     dtype=torch.uint8, device="cuda")
    dH = torch.empty_like(H)
    dW = torch.empty_like(W)
    g = torch.ones(1, device="cuda")
    # eager reference and warm-up (device setup happens on the first call)
    loss_e, lse_e, counts_e, _ = F.flce_forward(H, W, lab, workspace=ws)
    F.flce_backward(H, W, lab, lse_e, counts_e, g, chunk_budget=budget, workspace=ws, dH=dH, dW=dW, **opts)
    torch.cuda.synchronize()
    dH_e, dW_e, loss_eager = dH.clone(), dW.clone(), loss_e.item()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            loss_g, lse_g, counts_g, _ = F.flce_forward(H, W, lab, workspace=ws)
            F.flce_backward(H, W, lab, lse_g, counts_g, g, chunk_budget=budget, workspace=ws, dH=dH, dW=dW, **opts)
    torch.cuda.current_stream().wait_stream(stream)
    dH.zero_()
    dW.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert loss_g.item() == loss_eager
    assert torch.equal(dH, dH_e) and torch.equal(dW, dW_e)


def test_skipping_a_gradient():
    """dW or dH can be skipped (NULL at the ABI): the other one is bit-identical to a full
    backward and the skipped gradient's kernels are not launched (per vocabulary chunk the
    dW product, or the dH product and, when dH is split, its combining pass, and the zeroing
    of the dH rows that carry no gradient); autograd asks for dH only when the weight is
    frozen."""
    import linear_cross_entropy_indexed_gb300 as F
    w = S.scaled("llama3", N=300, Hd=128, V=3000, seed=61, w_std=0.05)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    g = torch.ones(1, device="cuda")
    budget = 300 * 2 * 1024           # 3 vocabulary chunks

    def run(**kw):
        sink = F.EventSink(capacity=64)
        with sink:
            out = F.flce_backward(H, W, lab, lse, counts, g, chunk_budget=budget, **kw)
        torch.cuda.synchronize()
        return out, [name for name, _ in sink.durations_ms()]

    (dH, dW), full = run()
    (dH_only, none_w), h_only = run(compute_dW=False)
    (none_h, dW_only), w_only = run(compute_dH=False)
    assert none_w is None and none_h is None
    assert torch.equal(dH_only, dH) and torch.equal(dW_only, dW)
    assert full.count("dw") == 3 and full.count("dh") == 3
    assert h_only == [k for k in full if k != "dw"]
    assert w_only == [k for k in full if k not in ("dh", "dh_combine", "dh_zero")]
    with pytest.raises(F.FlceError, match="nothing to compute"):
        F.flce_backward(H, W, lab, lse, counts, g, compute_dH=False, compute_dW=False)
    # autograd with a frozen weight: H.grad matches, no dW launched
    # (autograd runs the backward on its own thread, whose launch counter is separate)
    Hg = H.clone().requires_grad_(True)
    F.linear_cross_entropy(Hg, W, lab, chunk_budget=budget).backward()
    torch.cuda.synchronize()
    assert torch.equal(Hg.grad, dH) and W.grad is None


def test_bad_label_is_reported_by_the_next_call():
    """The autograd path does not synchronise to look at the counts: a label outside
    [0, V) is treated as ignored by the kernels, and the next linear_cross_entropy() call
    (here after the step has finished) raises FlceError; a clean step triggers no host
    synchronisation and reports nothing."""
    import linear_cross_entropy_indexed_gb300 as F
    F.check_pending(wait=True)  # nothing left over from earlier tests
    w = S.scaled("tiny", N=200, Hd=64, V=900, seed=83)
    Hb, Wb, y = P.make_case(w)
    H = P.to_device(Hb).requires_grad_(True)
    W = P.to_device(Wb).requires_grad_(True)
    good = torch.from_numpy(y).cuda()
    bad = good.clone()
    bad[5] = 900
    torch.cuda.set_sync_debug_mode("error")  # any synchronising torch call raises
    try:
        F.linear_cross_entropy(H, W, good).backward()
        loss = F.linear_cross_entropy(H, W, bad)   # nothing raised yet: nothing waited
        loss.backward()
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()
    with pytest.raises(F.FlceError, match="1 labels outside"):
        F.linear_cross_entropy(H, W, good)
    # reported once: the following steps are clean
    F.linear_cross_entropy(H, W, good).backward()
    torch.cuda.synchronize()
    assert F.check_pending(wait=True) == 0
    # an explicit check after a bad step, without a further call
    F.linear_cross_entropy(H, W, bad).backward()
    with pytest.raises(F.FlceError, match="labels outside"):
        F.check_pending(wait=True)
    assert F.check_pending(wait=True) == 0
