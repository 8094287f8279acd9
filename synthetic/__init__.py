"""Seeded synthetic inputs for the fused linear + cross-entropy workloads.

This module is shared by the CUDA path's tests/benchmark and by the fp64 oracle's
tests.  It holds no arithmetic of the method itself: it only draws hidden states H,
head weights W (both bf16, stored as uint16 bit patterns) and integer labels.

Recipes (one per workload; sizes follow the shapes the pages discuss):

* ``tiny``    N=256,   Hd=64,   V=2000,   H~N(0,1), W~N(0,1/Hd), labels uniform,
              10% ignored (Bernoulli), mean, no softcap, seed 0.
* ``llama2``  N=8192,  Hd=4096, V=32000,  H~N(0,1), W~N(0,0.02^2), labels uniform,
              5% ignored, mean, seed 1.
* ``llama3``  N=8192,  Hd=4096, V=128256, labels Zipf(s=1.1) over ranks mapped to ids
              by a seeded permutation, 5% ignored, mean, seed 2.
* ``gemma2``  N=8192,  Hd=2304, V=256128, as llama3 plus tanh softcap 30.0, seed 3.
* ``packed``  N=32768 (8 x 4096), Hd=3584, V=152064: each 4096-long row packs 4
              documents (3 distinct uniform cut points, every document >= 2 long),
              token ids Zipf(1.1); label[p] = token[p+1] inside a document and
              ignore_index at each document's last position; mean, seed 4.
* ``peaked``  the llama3 shape with confident predictions: h_i = e_i + b w_{y_i} / |w_{y_i}|^2
              (e_i ~ N(0,1), b = 14) for rows with a valid label, so the target logit
              stands about 14 above the rest (p_y ~ 0.8, other entries mostly < 2^-12);
              seed 5.  Used to measure gradient filtering.
* ``unigram`` the llama3 shape with a unigram prior, standing in for a trained model whose
              logits favour frequent words: feature 0 of every hidden state is 1 and
              feature 0 of w_v is -2 ln(rank(v) + 1), rank(v) being v's rank in the
              label draw (frequent labels have high prior logits); the other features are
              the peaked recipe with b = 8 (applied to features 1..Hd-1 only).  About
              2.3e-4 of the softmax entries exceed 2^-12 (~30 per row), mostly the
              frequent words, scattered over the ids by the rank permutation; seed 6.
              Used to measure vocabulary sorting.

Random numbers come from the counter-based generator in ``synth.c`` (splitmix64 +
Box-Muller), so a row range of H or W can be regenerated alone.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_H = 1
STREAM_W = 2
STREAM_LABEL = 3
STREAM_IGNORE = 4
STREAM_PERM = 5
STREAM_DOCS = 6

IGNORE_INDEX = -100


def build(force: bool = False) -> str:
    """Compile the generator with the host C compiler (portable C, no ISA flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                              ctypes.c_int]
            lib.synth_uniform_f64.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_uint64, ctypes.c_uint64]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(shape, seed: int, stream: int, std: float, offset: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of std * N(0,1), elements [offset, offset+prod(shape))."""
    out = np.empty(shape, dtype=np.uint16)
    n = out.size
    _get().synth_normal_bf16(out.ctypes.data, int(offset), int(n), int(seed), int(stream),
                             float(std), _threads())
    return out


def uniform(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _get().synth_uniform_f64(out.ctypes.data, int(offset), int(n), int(seed), int(stream))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (bf16 is the top half of fp32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even), returning uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def zipf_ranks(u: np.ndarray, V: int, s: float) -> np.ndarray:
    """Inverse-CDF draw of ranks 0..V-1 with P(rank k) proportional to (k+1)^-s."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    r = np.searchsorted(cdf, u, side="right")
    return np.minimum(r, V - 1).astype(np.int64)


def permutation(V: int, seed: int) -> np.ndarray:
    """Seeded permutation of 0..V-1 (argsort of V counter uniforms)."""
    return np.argsort(uniform(V, seed, STREAM_PERM), kind="stable").astype(np.int64)


@dataclass
class Workload:
    name: str
    N: int
    Hd: int
    V: int
    seed: int
    w_std: float
    labels: str            # "uniform" | "zipf" | "packed"
    ignore_frac: float
    softcap: float = 0.0
    reduction: str = "mean"
    ignore_index: int = IGNORE_INDEX
    zipf_s: float = 1.1
    n_seq: int = 0
    seq_len: int = 0
    n_docs: int = 0
    peak: float = 0.0       # b of the peaked recipe (0: H is plain N(0,1))
    unigram: float = 0.0    # slope of the unigram prior in feature 0 (0: none)
    extra: dict = field(default_factory=dict)

    @property
    def flops_fwd(self) -> float:
        return 2.0 * self.N * self.Hd * self.V

    @property
    def flops_bwd(self) -> float:
        return 6.0 * self.N * self.Hd * self.V


WORKLOADS = {
    "tiny": Workload("tiny", 256, 64, 2000, 0, 1.0 / 8.0, "uniform", 0.10),
    "llama2": Workload("llama2", 8192, 4096, 32000, 1, 0.02, "uniform", 0.05),
    "llama3": Workload("llama3", 8192, 4096, 128256, 2, 0.02, "zipf", 0.05),
    "gemma2": Workload("gemma2", 8192, 2304, 256128, 3, 0.02, "zipf", 0.05, softcap=30.0),
    "packed": Workload("packed", 32768, 3584, 152064, 4, 0.02, "packed", 0.0,
                       n_seq=8, seq_len=4096, n_docs=4),
    "peaked": Workload("peaked", 8192, 4096, 128256, 5, 0.02, "zipf", 0.05, peak=14.0),
    "unigram": Workload("unigram", 8192, 4096, 128256, 6, 0.02, "zipf", 0.05, peak=8.0, unigram=2.0),
}


def scaled(name: str, N: int | None = None, Hd: int | None = None, V: int | None = None,
           seed: int | None = None, **kw) -> Workload:
    """A named recipe with some sizes replaced (for small parity cases)."""
    w = WORKLOADS[name]
    d = dict(w.__dict__)
    d.update({k: v for k, v in dict(N=N, Hd=Hd, V=V, seed=seed).items() if v is not None})
    d.update(kw)
    d["name"] = d.get("name", w.name)
    return Workload(**d)


def make_labels(w: Workload) -> np.ndarray:
    N, V = w.N, w.V
    if w.labels == "packed":
        return packed_labels(w)
    u = uniform(N, w.seed, STREAM_LABEL)
    if w.labels == "uniform":
        y = np.minimum((u * V).astype(np.int64), V - 1)
    elif w.labels == "zipf":
        y = permutation(V, w.seed)[zipf_ranks(u, V, w.zipf_s)]
    else:
        raise ValueError(w.labels)
    if w.ignore_frac > 0:
        drop = uniform(N, w.seed, STREAM_IGNORE) < w.ignore_frac
        y = np.where(drop, w.ignore_index, y)
    return y.astype(np.int64)


def doc_cuts(w: Workload, seq: int) -> list[int]:
    """Sorted document start offsets (first is 0) for packed row `seq`."""
    L, k = w.seq_len, w.n_docs
    j = 0
    while True:
        u = uniform(k - 1, w.seed, STREAM_DOCS, offset=(seq * 1024 + j) * (k - 1))
        cuts = sorted(set(int(x) for x in (2 + u * (L - 3)).astype(np.int64)))
        bounds = [0] + cuts + [L]
        if len(cuts) == k - 1 and all(b - a >= 2 for a, b in zip(bounds[:-1], bounds[1:])):
            return [0] + cuts
        j += 1


def packed_labels(w: Workload) -> np.ndarray:
    L = w.seq_len
    u = uniform(w.n_seq * L, w.seed, STREAM_LABEL)
    tokens = permutation(w.V, w.seed)[zipf_ranks(u, w.V, w.zipf_s)]
    y = np.empty(w.n_seq * L, dtype=np.int64)
    for s in range(w.n_seq):
        starts = doc_cuts(w, s)
        ends = starts[1:] + [L]
        base = s * L
        for a, b in zip(starts, ends):
            y[base + a:base + b - 1] = tokens[base + a + 1:base + b]
            y[base + b - 1] = w.ignore_index
    return y


def make_H(w: Workload, rows: slice | None = None, W: np.ndarray | None = None) -> np.ndarray:
    """H rows [r0, r1) as bf16 bits.  For the peaked recipe the target direction is
    added (W, the full bf16 weight, may be passed to avoid regenerating it); with the
    unigram prior feature 0 is set to 1 and carries no part of that direction."""
    r0, r1 = (0, w.N) if rows is None else (rows.start, rows.stop)
    e = normal_bf16((r1 - r0, w.Hd), w.seed, STREAM_H, 1.0, offset=r0 * w.Hd)
    if w.peak <= 0 and w.unigram <= 0:
        return e
    h = bf16_bits_to_f32(e).astype(np.float64)
    if w.peak > 0:
        y = make_labels(w)[r0:r1]
        ok = (y >= 0) & (y < w.V)
        Wb = make_W(w) if W is None else W
        wy = bf16_bits_to_f32(Wb[np.where(ok, y, 0)]).astype(np.float64)
        if w.unigram > 0:
            wy[:, 0] = 0.0
        h[ok] += w.peak * wy[ok] / (wy[ok] ** 2).sum(axis=1, keepdims=True)
    if w.unigram > 0:
        h[:, 0] = 1.0
    return f32_to_bf16_bits(h.astype(np.float32))


def unigram_prior(w: Workload) -> np.ndarray:
    """-s ln(rank(v) + 1) for every id v, rank(v) its rank in the Zipf label draw."""
    rank = np.empty(w.V, dtype=np.int64)
    rank[permutation(w.V, w.seed)] = np.arange(w.V)
    return -w.unigram * np.log(rank + 1.0)


def make_W(w: Workload, rows: slice | None = None) -> np.ndarray:
    r0, r1 = (0, w.V) if rows is None else (rows.start, rows.stop)
    Wb = normal_bf16((r1 - r0, w.Hd), w.seed, STREAM_W, w.w_std, offset=r0 * w.Hd)
    if w.unigram > 0:
        Wb[:, 0] = f32_to_bf16_bits(unigram_prior(w)[r0:r1].astype(np.float32))
    return Wb


def make_inputs(w: Workload | str) -> dict:
    if isinstance(w, str):
        w = WORKLOADS[w]
    Wb = make_W(w)
    return dict(H=make_H(w, W=Wb), W=Wb, labels=make_labels(w), workload=w)
