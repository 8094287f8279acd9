"""Fused LM-head linear + softmax cross-entropy for GB300 (sm_103a).

A thin Python binding over the C ABI in ``include/flce.h`` (``libflce.so`` built in
tree by ``_build.py``).  This file only marshals arguments: PyTorch provides device
memory and the current stream; every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing or the device is
not an sm_103 GPU, the calls raise.

User entry point::

    loss = linear_cross_entropy(hidden, lm_head_weight, labels,
                                ignore_index=-100, softcap=0.0, reduction="mean")
    loss.backward()        # dH and dW through the fused backward

``hidden`` is [..., Hd] bf16, ``lm_head_weight`` is [V, Hd] bf16 (the layout of a
PyTorch ``nn.Linear(Hd, V).weight``), ``labels`` is [...] int64 and already shifted
for next-token prediction.  The N x V logits are never materialised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "linear_cross_entropy", "FusedLinearCrossEntropyLoss", "flce_forward", "flce_backward", "flce_forward_shard", "flce_merge_shards",
    "flce_backward_shard", "forward_workspace_size",
    "backward_workspace_size", "vocab_order", "FlceError", "check_counts", "check_pending", "library",
    "launch_count", "EventSink", "KERNEL_NAMES", "stage_h2d",
]

REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}
KERNEL_NAMES = {0: "label_dot", 1: "linear_lse", 2: "lse_merge", 3: "reduce", 4: "bwd_prep",
                5: "dz", 6: "dw", 7: "dh", 8: "zero", 9: "block_mask", 10: "selftest", 11: "shard_merge",
                12: "vocab_keys", 13: "vocab_sort", 14: "gather", 15: "dh_combine", 16: "compact",
                17: "dh_zero", 18: "stage"}
BWD_SORT_VOCAB = 1
BWD_COMPENSATED = 2


def _options(sort_vocab: bool, compensated: bool) -> int:
    return (BWD_SORT_VOCAB if sort_vocab else 0) | (BWD_COMPENSATED if compensated else 0)

_lock = threading.Lock()
_lib = None


class FlceError(RuntimeError):
    pass


def library() -> ctypes.CDLL:
    """The loaded ``libflce.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise FlceError("libflce.so is not built (run __graft_entry__.build() or "
                                "python -m linear_cross_entropy_indexed_gb300._build)")
            lib = ctypes.CDLL(_build.LIB)
            i64, sz, vp, f32, i32 = (ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p,
                                     ctypes.c_float, ctypes.c_int)
            lib.flce_forward_workspace_size.argtypes = [i64, i64, i64]
            lib.flce_forward_workspace_size.restype = sz
            u32 = ctypes.c_uint
            lib.flce_backward_workspace_size.argtypes = [i64, i64, i64, sz, u32]
            lib.flce_backward_workspace_size.restype = sz
            lib.flce_forward.argtypes = [vp, vp, vp, i64, i64, i64, i64, f32, i32, vp, vp, vp, vp, vp, sz, vp]
            lib.flce_forward.restype = i32
            lib.flce_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, i32, vp, f32, u32, vp, vp,
                                          vp, sz, sz, vp]
            lib.flce_vocab_order_workspace_size.argtypes = [i64, i64, i64]
            lib.flce_vocab_order_workspace_size.restype = sz
            lib.flce_vocab_order.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, vp, sz, vp]
            lib.flce_vocab_order.restype = i32
            lib.flce_backward.restype = i32
            lib.flce_strerror.argtypes = [i32]
            lib.flce_strerror.restype = ctypes.c_char_p
            lib.flce_last_cuda_error.restype = i32
            lib.flce_launch_count.restype = ctypes.c_uint64
            lib.flce_set_event_sink.argtypes = [vp, vp, vp, i32]
            lib.flce_set_event_sink.restype = i32
            lib.flce_event_sink_used.restype = i32
            lib.flce_forward_shard.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp, vp, vp, sz, vp]
            lib.flce_forward_shard.restype = i32
            lib.flce_merge_shards_workspace_size.argtypes = [i64]
            lib.flce_merge_shards_workspace_size.restype = sz
            lib.flce_merge_shards.argtypes = [vp, vp, i64, vp, i64, i64, i64, i32, vp, vp, vp, vp, sz, vp]
            lib.flce_merge_shards.restype = i32
            lib.flce_backward_shard.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, i32, vp, f32,
                                                u32, vp, vp, vp, sz, sz, vp]
            lib.flce_backward_shard.restype = i32
            lib.flce_selftest_wait_timeout.argtypes = [vp, vp]
            lib.flce_selftest_wait_timeout.restype = i32
            lib.flce_stage_h2d.argtypes = [vp, vp, sz, vp]
            lib.flce_stage_h2d.restype = i32
            _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != 0:
        lib = library()
        raise FlceError("flce: %s (status %d, cuda error %d)" % (
            lib.flce_strerror(status).decode(), status, lib.flce_last_cuda_error()))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _reduction(r) -> int:
    if isinstance(r, int):
        return r
    try:
        return REDUCTIONS[r]
    except KeyError:
        raise ValueError("reduction must be one of %s" % list(REDUCTIONS)) from None


def forward_workspace_size(N: int, Hd: int, V: int) -> int:
    return int(library().flce_forward_workspace_size(N, Hd, V))


def backward_workspace_size(N: int, Hd: int, V: int, chunk_budget: int = 0, sort_vocab: bool = False,
                            compensated: bool = False) -> int:
    return int(library().flce_backward_workspace_size(N, Hd, V, chunk_budget, _options(sort_vocab, compensated)))


def vocab_order(H, W, workspace=None):
    """Sort keys (mean raw logit of every vocabulary row over the rows of H) and the
    order the sorted backward walks: (keys fp32 [V], perm int32 [V], inv int32 [V]),
    perm[p] = the row at position p, keys descending, ties by ascending row."""
    if not (H.is_cuda and W.is_cuda and H.is_contiguous() and W.is_contiguous()):
        raise FlceError("H and W must be contiguous CUDA tensors")
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise FlceError("H and W must be bfloat16")
    N, Hd = H.shape
    V = W.shape[0]
    dev = W.device
    with torch.cuda.device(dev):
        keys = torch.empty(V, dtype=torch.float32, device=dev)
        perm = torch.empty(V, dtype=torch.int32, device=dev)
        inv = torch.empty(V, dtype=torch.int32, device=dev)
        need = int(library().flce_vocab_order_workspace_size(N, Hd, V))
        ws = workspace if workspace is not None else torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(library().flce_vocab_order(_p(H), _p(W), N, Hd, V, _p(keys), _p(perm), _p(inv), _p(ws), ws.numel(),
                                          _stream(dev)))
    return keys, perm, inv


def _check_inputs(H, W, labels):
    for name, t in (("H", H), ("W", W), ("labels", labels)):
        if not t.is_cuda:
            raise FlceError("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise FlceError("%s must be contiguous" % name)
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise FlceError("H and W must be bfloat16")
    if labels.dtype != torch.int64:
        raise FlceError("labels must be int64")
    if H.dim() != 2 or W.dim() != 2 or labels.dim() != 1:
        raise FlceError("expected H [N, Hd], W [V, Hd], labels [N]")
    if H.shape[1] != W.shape[1] or labels.shape[0] != H.shape[0]:
        raise FlceError("shape mismatch: H %s, W %s, labels %s" % (tuple(H.shape), tuple(W.shape),
                                                                     tuple(labels.shape)))
    if not (H.device == W.device == labels.device):
        raise FlceError("H, W and labels must be on one device")


def flce_forward(H, W, labels, ignore_index: int = -100, softcap: float = 0.0, reduction="mean",
                 want_target: bool = False, workspace=None):
    """One forward call.  Returns (loss, lse, counts, target_or_None); loss is a
    0-d tensor for mean/sum and [N] for none; counts = [n_valid, n_bad, error_bits]."""
    _check_inputs(H, W, labels)
    red = _reduction(reduction)
    N, Hd = H.shape
    V = W.shape[0]
    dev = H.device
    with torch.cuda.device(dev):
        loss = torch.empty(N if red == 2 else 1, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        counts = torch.empty(3, dtype=torch.int64, device=dev)
        tgt = torch.empty(N, dtype=torch.float32, device=dev) if want_target else None
        need = forward_workspace_size(N, Hd, V)
        ws = workspace if workspace is not None else torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(library().flce_forward(_p(H), _p(W), _p(labels), N, Hd, V, int(ignore_index), float(softcap), red,
                                      _p(loss), _p(lse), _p(tgt), _p(counts), _p(ws), ws.numel(), _stream(dev)))
    return (loss if red == 2 else loss[0]), lse, counts, tgt


def flce_backward(H, W, labels, lse, counts, grad_out, ignore_index: int = -100, softcap: float = 0.0,
                  reduction="mean", chunk_budget: int = 0, workspace=None, dH=None, dW=None,
                  filter_threshold: float = 0.0, sort_vocab: bool = False, compensated: bool = False,
                  compute_dH: bool = True, compute_dW: bool = True):
    """One backward call from the saved LSE and counts.  Returns (dH, dW) in bf16; a
    gradient with compute_dH / compute_dW False is not computed and returned as None.
    filter_threshold > 0 turns on gradient filtering (softmax entries below it, other
    than the target, are dropped and all-zero blocks are skipped): an approximation.
    sort_vocab walks the vocabulary in mean-logit order (see vocab_order), which gathers
    the surviving entries into fewer blocks; the result is the same sums reordered.
    compensated carries the bf16 rounding remainder of every dZ entry into dH and dW
    (twice the dW / dH work; exact gradient only, not with filter_threshold > 0)."""
    _check_inputs(H, W, labels)
    red = _reduction(reduction)
    N, Hd = H.shape
    V = W.shape[0]
    dev = H.device
    g = grad_out.to(device=dev, dtype=torch.float32).reshape(-1).contiguous()
    if g.numel() != (N if red == 2 else 1):
        raise FlceError("grad_out has %d elements" % g.numel())
    with torch.cuda.device(dev):
        if not (compute_dH or compute_dW):
            raise FlceError("nothing to compute: compute_dH and compute_dW are both False")
        dH = None if not compute_dH else (dH if dH is not None else torch.empty_like(H))
        dW = None if not compute_dW else (dW if dW is not None else torch.empty_like(W))
        need = backward_workspace_size(N, Hd, V, chunk_budget, sort_vocab, compensated)
        ws = workspace if workspace is not None else torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(library().flce_backward(_p(H), _p(W), _p(labels), _p(lse), _p(counts), N, Hd, V, int(ignore_index),
                                       float(softcap), red, _p(g), float(filter_threshold),
                                       _options(sort_vocab, compensated), _p(dH), _p(dW), _p(ws), ws.numel(),
                                       int(chunk_budget), _stream(dev)))
    return dH, dW


# ----------------------------------------------------------------- vocabulary sharding
def flce_forward_shard(H, W_shard, labels, v_offset: int, V_total: int, ignore_index: int = -100,
                       softcap: float = 0.0, workspace=None):
    """Forward over one vocabulary shard (W rows [v_offset, v_offset + V_shard) of V_total).
    Returns (lse_shard, target_shard, counts); merge the shards with flce_merge_shards."""
    _check_inputs(H, W_shard, labels)
    N, Hd = H.shape
    Vs = W_shard.shape[0]
    dev = H.device
    with torch.cuda.device(dev):
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        tgt = torch.empty(N, dtype=torch.float32, device=dev)
        counts = torch.empty(3, dtype=torch.int64, device=dev)
        need = forward_workspace_size(N, Hd, Vs)
        ws = workspace if workspace is not None else torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(library().flce_forward_shard(_p(H), _p(W_shard), _p(labels), N, Hd, Vs, int(v_offset), int(V_total),
                                            int(ignore_index), float(softcap), _p(lse), _p(tgt), _p(counts), _p(ws),
                                            ws.numel(), _stream(dev)))
    return lse, tgt, counts


def flce_merge_shards(lse_parts, target_parts, labels, V_total: int, ignore_index: int = -100, reduction="mean"):
    """Fixed-order merge of [n_shards, N] per-shard LSEs and target logits (shard order)
    into (loss, global lse, counts)."""
    red = _reduction(reduction)
    lse_parts = lse_parts.float().contiguous()
    target_parts = target_parts.float().contiguous()
    R, N = lse_parts.shape
    dev = lse_parts.device
    with torch.cuda.device(dev):
        loss = torch.empty(N if red == 2 else 1, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        counts = torch.empty(3, dtype=torch.int64, device=dev)
        need = int(library().flce_merge_shards_workspace_size(N))
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(library().flce_merge_shards(_p(lse_parts), _p(target_parts), R, _p(labels), N, int(V_total),
                                           int(ignore_index), red, _p(loss), _p(lse), _p(counts), _p(ws), ws.numel(),
                                           _stream(dev)))
    return (loss if red == 2 else loss[0]), lse, counts


def flce_backward_shard(H, W_shard, labels, lse, counts, grad_out, v_offset: int, V_total: int,
                        ignore_index: int = -100, softcap: float = 0.0, reduction="mean", chunk_budget: int = 0,
                        filter_threshold: float = 0.0, sort_vocab: bool = False, compensated: bool = False):
    """Backward over one vocabulary shard from the global lse and counts.  Returns
    (dH_partial fp32 [N, Hd], to be summed over the shards; dW_shard bf16)."""
    _check_inputs(H, W_shard, labels)
    red = _reduction(reduction)
    N, Hd = H.shape
    Vs = W_shard.shape[0]
    dev = H.device
    g = grad_out.to(device=dev, dtype=torch.float32).reshape(-1).contiguous()
    with torch.cuda.device(dev):
        dh = torch.empty(N, Hd, dtype=torch.float32, device=dev)
        dw = torch.empty_like(W_shard)
        need = backward_workspace_size(N, Hd, Vs, chunk_budget, sort_vocab, compensated)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check(library().flce_backward_shard(_p(H), _p(W_shard), _p(labels), _p(lse), _p(counts), N, Hd, Vs,
                                             int(v_offset), int(V_total), int(ignore_index), float(softcap), red,
                                             _p(g), float(filter_threshold), _options(sort_vocab, compensated),
                                             _p(dh), _p(dw), _p(ws), ws.numel(), int(chunk_budget), _stream(dev)))
    return dh, dw


def _raise_on_counts(c, where: str = "", labels: bool = True) -> None:
    if c[2] != 0:
        raise FlceError("%sdevice error bits %#x (1: a bounded wait expired, 2: a vocabulary order index "
                        "out of range)" % (where, c[2]))
    if labels and c[1] != 0:
        raise FlceError("%s%d labels outside [0, V) that are not ignore_index" % (where, c[1]))


def check_counts(counts) -> tuple[int, int]:
    """Host check of a counts tensor (synchronises): raises on bad labels or on a
    device-side wait timeout; returns (n_valid, n_bad)."""
    c = counts.tolist()
    _raise_on_counts(c)
    return c[0], c[1]


# Lazy checks of the autograd path.  After each forward and each backward of
# linear_cross_entropy() the three counts are copied, on the launch stream, into pinned
# host memory and an event is recorded; nothing waits.  The next call (or check_pending())
# looks at every copy whose event has completed and raises FlceError if a forward saw
# labels outside [0, V) (rows the kernels treated as ignored) or a forward or backward
# set a device error bit.  The backward's copy reports error bits only, so a bad label
# is reported once, by its forward.
_pending = []
_pending_lock = threading.Lock()


def _watch_counts(counts, what: str, labels: bool) -> None:
    if torch.cuda.is_current_stream_capturing():
        return  # a captured graph has no host side to report to; use check_counts on its counts
    host = torch.empty(3, dtype=torch.int64, pin_memory=True)
    host.copy_(counts, non_blocking=True)
    ev = torch.cuda.Event()
    ev.record()
    with _pending_lock:
        _pending.append((ev, host, what, labels))


def check_pending(wait: bool = False) -> int:
    """Raise FlceError if an earlier linear_cross_entropy() forward saw labels outside
    [0, V) that are not ignore_index, or a forward or backward set a device error bit.
    Only copies whose event has completed are looked at, unless wait=True (which waits
    for all of them).  Each step is reported once.  Returns how many are still pending."""
    with _pending_lock:
        done, left = [], []
        for item in _pending:
            if wait:
                item[0].synchronize()
            (done if item[0].query() else left).append(item)
        _pending[:] = left
        n_left = len(left)
    for _, host, what, labels in done:
        _raise_on_counts(host.tolist(), "an earlier %s: " % what, labels)
    return n_left


class _FusedLinearCrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, labels, ignore_index, softcap, reduction, chunk_budget, filter_threshold, sort_vocab,
                compensated):
        loss, lse, counts, _ = flce_forward(H, W, labels, ignore_index, softcap, reduction)
        _watch_counts(counts, "linear_cross_entropy forward", labels=True)
        ctx.save_for_backward(H, W, labels, lse, counts)
        ctx.cfg = (ignore_index, softcap, reduction, chunk_budget, filter_threshold, sort_vocab, compensated)
        return loss

    @staticmethod
    def backward(ctx, grad):
        H, W, labels, lse, counts = ctx.saved_tensors
        ignore_index, softcap, reduction, chunk_budget, filter_threshold, sort_vocab, compensated = ctx.cfg
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (need_h or need_w):
            return (None,) * 10
        dH, dW = flce_backward(H, W, labels, lse, counts, grad, ignore_index, softcap, reduction, chunk_budget,
                               filter_threshold=filter_threshold, sort_vocab=sort_vocab, compensated=compensated,
                               compute_dH=need_h, compute_dW=need_w)
        _watch_counts(counts, "linear_cross_entropy backward", labels=False)
        return (dH, dW, None, None, None, None, None, None, None, None)


def linear_cross_entropy(hidden, weight, labels, ignore_index: int = -100, softcap: float = 0.0,
                         reduction: str = "mean", chunk_budget: int = 0, filter_threshold: float = 0.0,
                         sort_vocab: bool = False, compensated: bool = False):
    """Cross-entropy of ``hidden @ weight.T`` against ``labels`` without materialising
    the logits.  ``hidden`` [..., Hd] bf16, ``weight`` [V, Hd] bf16, ``labels`` [...]
    int64.  reduction: "mean" (over rows whose label is valid), "sum" or "none".
    filter_threshold > 0 (e.g. 2**-12) makes the backward approximate, sort_vocab lets it
    skip more blocks, compensated makes the exact backward more precise: see
    flce_backward.

    Labels outside [0, V) that are not ignore_index are treated as ignored by the
    kernels; they, and device error bits, are reported without a host synchronisation:
    the next call (or check_pending()) raises FlceError once the step that saw them has
    finished on the GPU."""
    check_pending()
    Hd = hidden.shape[-1]
    H2 = hidden.reshape(-1, Hd)
    y = labels.reshape(-1)
    out = _FusedLinearCrossEntropy.apply(H2.contiguous(), weight.contiguous(), y.contiguous(), int(ignore_index),
                                         float(softcap), reduction, int(chunk_budget), float(filter_threshold),
                                         bool(sort_vocab), bool(compensated))
    if reduction == "none":
        out = out.reshape(labels.shape)
    return out


class FusedLinearCrossEntropyLoss(torch.nn.Module):
    """Module form of :func:`linear_cross_entropy`.

    ``forward(weight, hidden, labels)`` takes the LM-head weight first, the argument
    order of Liger's fused linear cross-entropy loss (Liger-CCE blog, §四); use
    :func:`linear_cross_entropy` for the hidden-first order of CCE's
    ``linear_cross_entropy(hidden, weight, labels)``.  Labels must already be shifted
    for next-token prediction.
    """

    def __init__(self, ignore_index: int = -100, softcap: float = 0.0, reduction: str = "mean",
                 chunk_budget: int = 0, filter_threshold: float = 0.0, sort_vocab: bool = False,
                 compensated: bool = False):
        super().__init__()
        _reduction(reduction)
        self.ignore_index = int(ignore_index)
        self.softcap = float(softcap)
        self.reduction = reduction
        self.chunk_budget = int(chunk_budget)
        self.filter_threshold = float(filter_threshold)
        self.sort_vocab = bool(sort_vocab)
        self.compensated = bool(compensated)

    def forward(self, weight, hidden, labels):
        return linear_cross_entropy(hidden, weight, labels, self.ignore_index, self.softcap, self.reduction,
                                    self.chunk_budget, self.filter_threshold, self.sort_vocab, self.compensated)

    def extra_repr(self):
        return "ignore_index=%d, softcap=%g, reduction=%s, filter_threshold=%g, sort_vocab=%s, compensated=%s" % (
            self.ignore_index, self.softcap, self.reduction, self.filter_threshold, self.sort_vocab, self.compensated)


def stage_h2d(dst, src):
    """Copy the pinned host tensor `src` into the device tensor `dst` (same byte size,
    both contiguous) on the current stream of dst's device, by SM loads through the host
    buffer's device mapping (flce_stage_h2d) rather than the copy engine: meant for a side
    stream that brings the next step's inputs in while this step's kernels run, which a
    copy-engine transfer from host memory slows several times more.  Returns dst."""
    if not dst.is_cuda or src.is_cuda:
        raise FlceError("stage_h2d copies a host tensor into a CUDA tensor")
    if not src.is_pinned():
        raise FlceError("stage_h2d needs a pinned host tensor (pin_memory())")
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise FlceError("stage_h2d needs contiguous tensors")
    nbytes = dst.numel() * dst.element_size()
    if nbytes != src.numel() * src.element_size():
        raise FlceError("stage_h2d: %d bytes into %d" % (src.numel() * src.element_size(), nbytes))
    with torch.cuda.device(dst.device):
        _check(library().flce_stage_h2d(_p(dst), ctypes.c_void_p(src.data_ptr()), nbytes, _stream(dst.device)))
    return dst


def launch_count() -> int:
    """Kernels launched through the library by this thread so far."""
    return int(library().flce_launch_count())


class EventSink:
    """Bracket every library kernel launch with a pair of CUDA events (for timing
    per kernel class on the launch stream).  Use as a context manager."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.start = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        self.end = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.start + self.end:
            e.record()  # materialise the underlying cudaEvent_t
        self._s = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.start])
        self._e = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.end])
        self._ids = (ctypes.c_int * capacity)()
        self.used = 0

    def __enter__(self):
        library().flce_set_event_sink(self._s, self._e, self._ids, self.capacity)
        return self

    def __exit__(self, *exc):
        self.used = int(library().flce_event_sink_used())
        library().flce_set_event_sink(None, None, None, 0)
        return False

    def durations_ms(self):
        """[(kernel_name, ms)] for every recorded launch (call after a synchronize)."""
        return [(KERNEL_NAMES.get(self._ids[k], str(self._ids[k])), self.start[k].elapsed_time(self.end[k]))
                for k in range(self.used)]
