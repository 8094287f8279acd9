"""Seeded sweep of small shapes: the CUDA path (through the C ABI) against the fp64
oracle, element by element, on many combinations that the hand-picked cases of the
other parity files do not reach.

Each case draws N, Hd and V from seeded lists that mix the tile boundaries (1, 127,
128, 129, 255, 256, 257, ... rows or columns; every hidden size the ABI accepts from
8 upward in steps of 8) with uniform random sizes, then crosses them with every
reduction, the softcap, a custom ignore_index, out-of-range labels, a vocabulary split
into several backward chunks, and the backward options (exact, compensated, sorted
vocabulary, gradient filtering with and without sorting).  Tolerances are those of
the other parity tests (tests/parity.py), the per-row gradient bounds included, and
ignored or bad-label rows must get an exactly zero dH row; the filtered modes are
compared with the oracle's filtered gradient."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

HIDDEN = [8, 16, 24, 40, 56, 64, 72, 120, 128, 136, 200, 256, 264, 328]
EDGE_N = [1, 2, 127, 128, 129, 255, 256, 257, 511, 512, 513]
EDGE_V = [1, 2, 3, 255, 256, 257, 511, 512, 513, 1023, 1025]
MODES = ["exact", "compensated", "sorted", "filtered", "exact", "filtered_sorted"]
THRESHOLD = 2.0 ** -12


def _cases(n=36, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        N = int(rng.choice(EDGE_N)) if k % 3 == 0 else int(rng.integers(1, 700))
        V = int(rng.choice(EDGE_V)) if k % 3 == 1 else int(rng.integers(1, 6000))
        Hd = int(rng.choice(HIDDEN))
        mode = MODES[k % len(MODES)]
        out.append(dict(
            N=N, Hd=Hd, V=V, mode=mode,
            reduction=("mean", "sum", "none")[k % 3],
            softcap=30.0 if k % 4 == 3 else 0.0,
            chunks=3 if k % 4 in (0, 1) else 1,     # backward vocabulary chunks wanted
            ignore_index=7 if k % 5 == 4 else -100,
            bad_labels=k % 7 == 5,
            seed=100 + k,
        ))
    return out


CASES = _cases()


def _id(c):
    return "N%d-Hd%d-V%d-%s-%s%s%s%s%s" % (
        c["N"], c["Hd"], c["V"], c["reduction"], c["mode"], "-cap" if c["softcap"] else "",
        "-chunked" if c["chunks"] > 1 else "", "-ign%d" % c["ignore_index"] if c["ignore_index"] != -100 else "",
        "-bad" if c["bad_labels"] else "")


def _chunk_budget(c):
    """The backward budget that splits V into about c['chunks'] vocabulary chunks
    (chunk widths are multiples of 256; 0 keeps the default, one chunk here)."""
    if c["chunks"] <= 1:
        return 0
    per_col = c["N"] * (4 if c["mode"] == "compensated" else 2)
    if c["mode"] in ("sorted", "filtered_sorted"):
        per_col += 2 * c["Hd"]
    vc = 256 * max(1, -(-c["V"] // (256 * c["chunks"])))
    return vc * per_col


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_shape_sweep(c):
    filtered = c["mode"] in ("filtered", "filtered_sorted")
    # logits of std ~2-3 so that the softcap bends the larger ones; confident rows for
    # the filtered modes so that the threshold drops entries
    w = S.scaled("peaked" if filtered else "llama3", N=c["N"], Hd=c["Hd"], V=c["V"], seed=c["seed"],
                 w_std=(0.5 if c["softcap"] else 2.0 / np.sqrt(c["Hd"])), peak=(6.0 if filtered else 0.0),
                 ignore_frac=0.1)
    Hb, Wb, y = P.make_case(w)
    if c["ignore_index"] != -100:
        y = np.where(y == -100, c["ignore_index"], y)
    if c["bad_labels"] and c["N"] >= 3:
        y = y.copy()
        y[0], y[c["N"] // 2] = c["V"], -5  # out of range and not the ignore index: counted, treated as ignored
    thr = THRESHOLD if filtered else 0.0
    out = P.run_gpu(Hb, Wb, y, c["ignore_index"], c["softcap"], c["reduction"], chunk_budget=_chunk_budget(c),
                    filter_threshold=thr, sort_vocab=c["mode"] in ("sorted", "filtered_sorted"),
                    compensated=c["mode"] == "compensated")
    ref, dH, dW = P.oracle_full(Hb, Wb, y, c["ignore_index"], c["softcap"], c["reduction"], filter_threshold=thr)
    P.check_forward(out, ref, y, c["V"], c["ignore_index"], c["reduction"])
    valid, _ = O.label_status(y, c["V"], c["ignore_index"])
    P.check_backward(out, dH, dW, no_grad_rows=~valid)
