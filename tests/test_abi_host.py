"""C-ABI checks that need no GPU: the library builds and loads, exports every symbol
declared in include/flce.h, sizes the workspace, and rejects bad arguments with a
status before it touches the device."""
import ctypes
import os
import re

import pytest

from linear_cross_entropy_indexed_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")

OK, ARG, ALIGN, WS, OVERFLOW, CUDA, UNSUP = range(7)


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    import linear_cross_entropy_indexed_gb300 as F
    return F.library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FLCE_API\s+[\w\s\*]+?\b(flce_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("flce_forward", "flce_backward", "flce_forward_workspace_size", "flce_backward_workspace_size",
              "flce_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n
    nm = os.popen("nm -D --defined-only %s" % _build.LIB).read()
    exported = set(re.findall(r"\bT (flce_\w+)", nm))
    assert set(declared_symbols()) <= exported


def test_strerror(lib):
    for s in range(7):
        assert lib.flce_strerror(s)
    assert b"unknown" in lib.flce_strerror(99)


def test_workspace_sizes(lib):
    f = lib.flce_forward_workspace_size
    b = lib.flce_backward_workspace_size
    assert f(256, 64, 2000) > 0
    assert f(0, 64, 2000) > 0 or f(0, 64, 2000) == 0
    assert f(-1, 64, 2000) == 0 and f(8, 63, 100) == 0 and f(8, 64, 0) == 0
    # forward scratch is O(N * V / 1024): one (max, sum) pair per row per group of 4 to 8
    # vocabulary tiles of 256 columns
    n, hd, v = 8192, 4096, 128256
    tiles = -(-v // 256)
    assert f(n, hd, v) >= 2 * (-(-tiles // 8)) * n * 4
    assert f(n, hd, v) < 2 * (-(-tiles // 4)) * n * 4 + (1 << 20)
    # backward: one bf16 [N, Vc] chunk plus an fp32 [N, Hd] accumulator when chunked, one
    # byte per 64 x 64 block of the chunk for the filtered mode, and the row compaction
    # (the rows that carry a gradient gathered to the front): a bf16 copy of H and RowInfo
    # for N rounded up to a 256-row tile, a row map, per-1024-row counts and the count
    def compact(n_, hd_):
        cap = -(-n_ // 256) * 256
        return cap * hd_ * 2 + cap * 16 + n_ * 4 + max(-(-n_ // 1024), 1) * 4 + 4
    budget = 64 << 20
    vc = (budget // (2 * n)) // 256 * 256
    size = b(n, hd, v, budget, 0)
    flags = (n // 64) * (vc // 64)
    assert size >= n * vc * 2 + n * hd * 4 + n * 16 + flags + compact(n, hd)
    assert size < n * vc * 2 + n * hd * 4 + n * 16 + flags + compact(n, hd) + (1 << 12)
    # chunks of equal width: a 1 GiB budget allows 65536 columns, so V = 128256 takes two
    # chunks, each ceil(128256 / 2) = 64128 columns rounded up to 256 = 64256
    size_1g = b(n, hd, v, 1 << 30, 0)
    base_1g = n * 64256 * 2 + n * hd * 4 + n * 16 + (n // 64) * (64256 // 64) + compact(n, hd)
    assert base_1g <= size_1g < base_1g + (1 << 14)  # + the K-step masks of the filtered mode
    # a single chunk needs no fp32 accumulator when dH is not split: 8192 x 4096 has 512 dH
    # tiles of 256 x 256, which fill 76 SM pairs to within 4%, so it is not split
    one = b(n, hd, 2000, 0, 0)
    flags1 = (n // 64) * (2048 // 64) + compact(n, hd)
    assert n * 2048 * 2 + n * 16 + flags1 <= one < n * 2048 * 2 + n * 16 + flags1 + (1 << 12)
    # few dH tiles: each tile's vocabulary range is split (256 x 64 is one tile: 4 parts),
    # which needs the fp32 accumulator and three fp32 [N, Hd] part sums even for one chunk
    small = b(256, 64, 2000, 0, 0)
    base_s = 256 * 2048 * 2 + 256 * 16 + 4 * 256 * 64 * 4 + compact(256, 64)
    assert base_s <= small < base_s + (256 // 64) * (2048 // 64) + (1 << 12)
    # 4096 x 4096: 256 tiles, split in 2 (4 waves of 76 pairs -> 3.5): one part buffer
    v2 = (budget // (2 * 4096)) // 256 * 256
    two = b(4096, 4096, v, budget, 0)
    base_2 = 4096 * v2 * 2 + 4096 * 16 + 2 * 4096 * 4096 * 4 + (4096 // 64) * (v2 // 64) + compact(4096, 4096)
    assert base_2 <= two < base_2 + (1 << 13)
    # the compensated mode is never split
    assert b(256, 64, 2000, 0, 2) < 2 * 256 * 2048 * 2 + 256 * 16 + compact(256, 64) + (1 << 13)
    # the sorted vocabulary: the budget also covers the sorted bf16 weight rows of the
    # chunk, Vc = budget / (2N + 2Hd), plus the order (key, two sort words, perm, inv:
    # 28 bytes per vocabulary row) and the column sums of H
    vs = (budget // (2 * n + 2 * hd)) // 256 * 256
    flags_s = (n // 64) * (vs // 64)
    size_s = b(n, hd, v, budget, 1)
    base = n * vs * 2 + vs * hd * 2 + n * hd * 4 + n * 16 + flags_s + 28 * v + 128 * hd * 4 + hd * 4 + compact(n, hd)
    assert base <= size_s < base + (1 << 13)
    assert b(n, hd, v, budget, 4) == 0 and b(n, hd, v, budget, 0x80000000) == 0
    # compensated: two bf16 dZ chunks, Vc = budget / 4N
    vcc = (budget // (4 * n)) // 256 * 256
    size_c = b(n, hd, v, budget, 2)
    base_c = 2 * n * vcc * 2 + n * hd * 4 + n * 16 + (n // 64) * (vcc // 64) + compact(n, hd)
    assert base_c <= size_c < base_c + (1 << 13)
    o = lib.flce_vocab_order_workspace_size
    assert 28 * v + 128 * hd * 4 + hd * 4 <= o(n, hd, v) < 28 * v + 128 * hd * 4 + hd * 4 + (1 << 12)
    assert o(0, 64, 10) > 0 and o(8, 60, 10) == 0 and o(8, 64, 0) == 0


def _fwd(lib, H=0x1000, W=0x2000, labels=0x3000, N=16, Hd=64, V=100, red=0, loss=0x4000, lse=0x5000,
         counts=0x6000, ws=0x10000, ws_bytes=1 << 20, softcap=0.0):
    return lib.flce_forward(H, W, labels, N, Hd, V, -100, softcap, red, loss, lse, None, counts, ws, ws_bytes, None)


def _bwd(lib, N=16, Hd=64, V=100, red=0, filt=0.0, ws_bytes=1 << 24, dW=0x7000, W=0x2000, options=0, dH=0x9000):
    return lib.flce_backward(0x1000, W, 0x3000, 0x5000, 0x6000, N, Hd, V, -100, 0.0, red, 0x8000, filt, options,
                             dH, dW, 0x10000, ws_bytes, 0, None)


def test_argument_errors_before_any_device_work(lib):
    assert _fwd(lib, H=None) == ARG
    assert _fwd(lib, W=None) == ARG
    assert _fwd(lib, red=3) == ARG
    assert _fwd(lib, N=-1) == ARG
    assert _fwd(lib, V=0) == ARG
    assert _fwd(lib, softcap=float("nan")) == ARG
    assert _fwd(lib, Hd=60) == ALIGN
    assert _fwd(lib, H=0x1008) == ALIGN
    assert _fwd(lib, W=0x2004) == ALIGN
    assert _fwd(lib, ws_bytes=16) == WS
    assert _fwd(lib, ws=0x10010) == WS
    assert _fwd(lib, N=1 << 40) == OVERFLOW
    assert _bwd(lib, filt=-0.5) == ARG
    assert _bwd(lib, filt=float("nan")) == ARG
    assert _bwd(lib, dW=None, dH=None) == ARG   # nothing to compute
    assert _bwd(lib, ws_bytes=16) == WS
    assert _bwd(lib, W=0x2002) == ALIGN
    assert _bwd(lib, options=4) == ARG
    assert _bwd(lib, options=2, filt=0.25) == ARG  # the compensated mode is exact-only
    assert _bwd(lib, options=1, ws_bytes=lib.flce_backward_workspace_size(16, 64, 100, 0, 0)) == WS
    vo = lambda H=0x1000, W=0x2000, perm=0x3000, ws_bytes=1 << 20, Hd=64: lib.flce_vocab_order(
        H, W, 16, Hd, 100, None, perm, None, 0x10000, ws_bytes, None)
    assert vo(perm=None) == ARG and vo(W=None) == ARG and vo(H=None) == ARG
    assert vo(W=0x2008) == ALIGN and vo(perm=0x3002) == ALIGN and vo(Hd=60) == ALIGN
    assert vo(ws_bytes=16) == WS


def test_shard_argument_errors(lib):
    f = lambda vs, off, vt: lib.flce_forward_shard(0x1000, 0x2000, 0x3000, 16, 64, vs, off, vt, -100, 0.0, 0x5000,
                                                   0x5400, 0x6000, 0x10000, 1 << 20, None)
    assert f(100, -1, 300) == ARG
    assert f(100, 250, 300) == ARG
    assert f(0, 0, 300) == ARG
    assert f(100, 0, 1 << 40) == OVERFLOW
    b = lambda off, vt: lib.flce_backward_shard(0x1000, 0x2000, 0x3000, 0x5000, 0x6000, 16, 64, 100, off, vt, -100,
                                                0.0, 0, 0x8000, 0.0, 0, 0x9000, 0x7000, 0x10000, 1 << 24, 0, None)
    assert b(-5, 300) == ARG and b(201, 300) == ARG
    m = lambda n, red: lib.flce_merge_shards(0x1000, 0x2000, n, 0x3000, 16, 300, -100, red, 0x4000, 0x5000, 0x6000,
                                             0x10000, 1 << 20, None)
    assert m(0, 0) == ARG and m(2, 5) == ARG
    assert lib.flce_merge_shards_workspace_size(1000) > 0


def test_valid_arguments_without_a_device_fail_cleanly(lib):
    # Arguments pass the checks; without a GPU the first CUDA call fails and the
    # library reports FLCE_ERR_CUDA (nothing is dereferenced on the host).
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert _fwd(lib) == CUDA
    assert lib.flce_last_cuda_error() != 0


def test_event_sink_toggles(lib):
    lib.flce_set_event_sink(None, None, None, 0)
    assert lib.flce_event_sink_used() == 0
    assert lib.flce_launch_count() >= 0


def test_static_scratch_covers_the_documented_limit(lib):
    """flce_forward_noalloc's static scratch holds the forward workspace of 8192 tokens
    with a 256K vocabulary (the Gemma-2-shaped head) at every hidden size the workloads
    use; the planner's vocabulary-tile group (at least 4 tiles per partial) is what keeps
    it inside, so a planner change that breaks the documented limit fails here."""
    import ctypes
    lib.flce_static_scratch_bytes.restype = ctypes.c_size_t
    limit = lib.flce_static_scratch_bytes()
    assert limit == 16 << 20
    for hd in (64, 2304, 3584, 4096, 8192):
        need = lib.flce_forward_workspace_size(8192, hd, 256128)
        assert 0 < need <= limit, (hd, need, limit)
    assert lib.flce_forward_workspace_size(8192, 64, 1_000_000) > limit

