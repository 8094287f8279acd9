"""Failure detection on the GPU without a fault: a bounded device wait is made to run
out (an mbarrier that nothing arrives on) and must return with the error bit set,
after which the context still runs the fused loss correctly."""
import ctypes

import pytest
import torch

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

FLCE_DEVERR_WAIT_TIMEOUT = 1


def test_bounded_wait_times_out_and_reports():
    import linear_cross_entropy_indexed_gb300 as F
    lib = F.library()
    status = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.flce_selftest_wait_timeout(ctypes.c_void_p(status.data_ptr()), stream) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == FLCE_DEVERR_WAIT_TIMEOUT
    # the context is intact: a normal forward + backward still matches the oracle
    w = S.scaled("tiny", N=130, Hd=64, V=700, seed=61)
    Hb, Wb, y = P.make_case(w)
    out = P.run_gpu(Hb, Wb, y)
    ref, dH, dW = P.oracle_full(Hb, Wb, y)
    P.check_forward(out, ref, y, w.V)
    P.check_backward(out, dH, dW)


def test_selftest_rejects_bad_arguments():
    import linear_cross_entropy_indexed_gb300 as F
    lib = F.library()
    assert lib.flce_selftest_wait_timeout(None, None) == 1
