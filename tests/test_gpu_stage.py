"""flce_stage_h2d: pinned host buffer -> device memory by SM loads.

The copy must reproduce every byte (16-byte words plus a ragged tail of 1..15 bytes),
run in stream order on the current stream, and refuse, before enqueuing anything, a host
buffer that is not pinned, a misaligned pointer and mismatched sizes."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _pinned_bytes(n, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(0, 256, size=n, dtype=np.uint8)).pin_memory()


@pytest.mark.parametrize("n", [1, 15, 16, 17, 4096 + 7, 1 << 20, (10 << 20) + 3])
def test_bytes_reproduced(n):
    import linear_cross_entropy_indexed_gb300 as F
    src = _pinned_bytes(n, n)
    dst = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    F.stage_h2d(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)


def test_typed_tensors_and_stream_order():
    # bf16 and int64 inputs as the end-to-end loop stages them, on a side stream, then
    # consumed on the main stream after an event
    import linear_cross_entropy_indexed_gb300 as F
    H = torch.randn(300, 136, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    y = torch.randint(-100, 5000, (300,), dtype=torch.int64).pin_memory()
    dH = torch.empty(300, 136, dtype=torch.bfloat16, device="cuda")
    dy = torch.empty(300, dtype=torch.int64, device="cuda")
    side = torch.cuda.Stream()
    done = torch.cuda.Event()
    with torch.cuda.stream(side):
        F.stage_h2d(dH, H)
        F.stage_h2d(dy, y)
        done.record(side)
    torch.cuda.current_stream().wait_event(done)
    total = dH.float().sum() + dy.sum().float()
    assert torch.equal(dH.cpu(), H) and torch.equal(dy.cpu(), y)
    assert abs(float(total) - (float(H.float().sum()) + float(y.sum()))) < 1e-2 * max(1.0, abs(float(total)))


def test_refusals():
    import linear_cross_entropy_indexed_gb300 as F
    lib = F.library()
    n = 4096
    src = _pinned_bytes(n, 1)
    dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    unpinned = torch.zeros(n, dtype=torch.uint8)
    with pytest.raises(F.FlceError):
        F.stage_h2d(dst, unpinned)
    with pytest.raises(F.FlceError):
        F.stage_h2d(dst[: n - 16], src)
    with pytest.raises(F.FlceError):
        F.stage_h2d(src, dst)  # wrong direction
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the C entry point checks before it enqueues: unpinned host memory (ARG, although on
    # a Grace host the GPU could read it), a host or pinned destination (ARG), misaligned
    # pointers (ALIGN), null pointers (ARG); zero bytes is a no-op
    assert lib.flce_stage_h2d(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(unpinned.data_ptr()), n, stream) == 1
    assert lib.flce_stage_h2d(ctypes.c_void_p(unpinned.data_ptr()), ctypes.c_void_p(src.data_ptr()), n, stream) == 1
    other = _pinned_bytes(n, 2)
    assert lib.flce_stage_h2d(ctypes.c_void_p(other.data_ptr()), ctypes.c_void_p(src.data_ptr()), n, stream) == 1
    assert lib.flce_stage_h2d(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(dst.data_ptr()), n, stream) == 1
    assert lib.flce_stage_h2d(ctypes.c_void_p(dst.data_ptr() + 1), ctypes.c_void_p(src.data_ptr()), 64, stream) == 2
    assert lib.flce_stage_h2d(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr() + 8), 64, stream) == 2
    assert lib.flce_stage_h2d(None, ctypes.c_void_p(src.data_ptr()), 64, stream) == 1
    assert lib.flce_stage_h2d(None, None, 0, stream) == 0
    before = F.launch_count()
    assert lib.flce_stage_h2d(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), 0, stream) == 0
    assert F.launch_count() == before
    torch.cuda.synchronize()
    assert not dst.any()  # nothing was copied by the refused calls
