"""The no-allocation forward entry point (flce_forward_noalloc) against flce_forward.

flce_forward_noalloc serves callers that cannot allocate device memory where they
compute the loss (for example a plug-in inside a runtime that owns all device memory
through its own pool): it takes no workspace and uses a static scratch array inside the
library.  This test calls it through the C ABI twice in a row on the same inputs and
checks every output against the workspace-taking flce_forward within the parity
tolerances, and checks that a problem too large for the static scratch is refused
before anything runs.  It lives in a file of its own that pytest collects last and is
self-contained, so it passes alone in a fresh process and after the other tests."""
import ctypes

import pytest
import torch

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _lib():
    import linear_cross_entropy_indexed_gb300 as F
    from linear_cross_entropy_indexed_gb300 import _build
    _build.build()
    lib = F.library()
    vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.flce_forward_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, f32, i32, vp, vp, vp, vp, vp]
    lib.flce_forward_noalloc.restype = i32
    lib.flce_static_scratch_bytes.restype = ctypes.c_size_t
    return F, lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("name,N,Hd,V,reduction", [("tiny", 300, 72, 1000, "mean"),
                                                   ("gemma2", 520, 128, 3001, "none"),
                                                   # the documented limit: 8192 tokens, a 256K vocabulary
                                                   ("gemma2", 8192, 64, 256128, "mean")])
def test_noalloc_forward_matches_workspace_forward(name, N, Hd, V, reduction):
    F, lib = _lib()
    w = S.scaled(name, N=N, Hd=Hd, V=V, seed=31, w_std=0.1)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    ref_loss, ref_lse, ref_counts, ref_t = F.flce_forward(H, W, lab, w.ignore_index, w.softcap, reduction,
                                                          want_target=True)
    red = F.REDUCTIONS[reduction]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        loss = torch.full((N if red == 2 else 1,), float("nan"), device="cuda")
        lse = torch.full((N,), float("nan"), device="cuda")
        tgt = torch.full((N,), float("nan"), device="cuda")
        counts = torch.full((3,), -1, dtype=torch.int64, device="cuda")
        st = lib.flce_forward_noalloc(_p(H), _p(W), _p(lab), N, Hd, V, w.ignore_index, w.softcap, red, _p(loss),
                                      _p(lse), _p(tgt), _p(counts), stream)
        assert st == 0, lib.flce_strerror(st)
        torch.cuda.synchronize()
        assert counts.tolist() == ref_counts.tolist(), call
        assert torch.allclose(lse, ref_lse, rtol=0, atol=P.TOL_LSE_ABS), call
        assert torch.allclose(tgt, ref_t, rtol=0, atol=P.TOL_TARGET_ABS), call
        ref_l = ref_loss.reshape(-1)
        assert torch.allclose(loss, ref_l, rtol=P.TOL_LOSS_REL, atol=P.TOL_LSE_ABS), call


def test_noalloc_refuses_sizes_beyond_the_static_scratch():
    F, lib = _lib()
    limit = int(lib.flce_static_scratch_bytes())
    N, Hd, V = 8192, 8, 1_000_000
    assert F.forward_workspace_size(N, Hd, V) > limit
    H = torch.zeros(N, Hd, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(V, Hd, dtype=torch.bfloat16, device="cuda")
    lab = torch.zeros(N, dtype=torch.int64, device="cuda")
    loss = torch.zeros(1, device="cuda")
    lse = torch.zeros(N, device="cuda")
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    before = F.launch_count()
    st = lib.flce_forward_noalloc(_p(H), _p(W), _p(lab), N, Hd, V, -100, 0.0, 0, _p(loss), _p(lse), None,
                                  _p(counts), None)
    assert st == 3  # FLCE_ERR_WORKSPACE
    assert F.launch_count() == before
