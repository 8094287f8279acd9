"""fp64 CPU oracle for the fused LM-head linear + softmax cross-entropy.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may import or call anything in this package.  The
product path (the C-ABI library and its Python binding) never does; it shares no
code, header, table or helper with this file.

What it computes is the plain definition, row by row, in double precision:

* logits        Z = H W^T, W stored [V, Hd] like an LM-head weight
                (ai-infra-kb M011 "模型最后一层为什么也能占很多内存", §01)
* softcap       z = c * tanh(x / c) on the raw logit x before the loss, with
                derivative factor 1 - tanh^2(x / c) in the backward; off when c <= 0
                (Unsloth fused-CE notes, §4 forward "Gemma2 softcap" and backward)
* per-row loss  loss_i = LSE(z_i) - z_{i,y_i}, LSE computed in the stable form
                m + log(sum(exp(z - m)))  (ai-infra-kb M011, §03; Liger-Kernel paper
                summary, "CrossEntropy Loss Kernel (Section 3.2, Eq. 15-16)", safe log)
* labels        y == ignore_index contributes no loss and no gradient; out-of-range
                labels are counted as "bad" and treated as ignored (a reading: the
                pages are silent on them)
* reduction     mean = sum of per-row losses / number of valid rows, divided once,
                never a mean of chunk means (ai-infra-kb M011, §04 and §07; Unsloth
                notes, §4 "n_items"); sum; none (the per-row vector).  All rows ignored
                under mean gives loss 0 and zero gradients (a reading of M011 §07,
                which asks for an explicit convention).
* gradient      dL/dx = (softmax(z) - onehot(y)) * scale_i * cap'(x), with softmax
                recomputed as exp(z - LSE) from the saved LSE; dH = dZ W, dW = dZ^T H
                (ai-infra-kb M011, §06; Liger-CCE blog "一、这堵墙" observation 1)
* filtering     optionally, softmax entries below a threshold (other than a valid row's
                target) are dropped before forming dZ: CCE's gradient filtering
                (Liger-CCE blog, §三), an approximation of the exact gradient
* vocab order   the sort key of each vocabulary entry (its raw logit averaged over the
                batch's rows) and the order that puts high keys first (Liger-CCE blog,
                §三: the forward tallies each word's mean logit and the backward places
                the frequent words in neighbouring blocks so that skipping is block-aligned)

``forward_split`` is a blockwise restatement (row chunks x vocab chunks merged with
the running (m, s) rule of ai-infra-kb M011 §05) used only by the oracle's own
self-tests to pin split invariance; the plain functions never call it.

Every function here is pinned by ``tests/test_oracle_pins.py`` (worked example,
two-tile split, finite differences, closed forms, the library routine
``torch.nn.functional.cross_entropy`` in fp64, brute force on tiny inputs).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

REDUCTIONS = ("mean", "sum", "none")


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of fp32)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- steps
def _raw_logits(Hf: np.ndarray, Wf: np.ndarray) -> np.ndarray:
    """x_{iv} = h_i . w_v for the rows given (a library matmul in fp64)."""
    return Hf @ Wf.T


def _cap(X: np.ndarray, softcap: float) -> np.ndarray:
    """Tanh logit softcap z = c tanh(x / c); identity when c <= 0."""
    if softcap > 0:
        return softcap * np.tanh(X / softcap)
    return X


def _cap_grad(X: np.ndarray, softcap: float) -> np.ndarray | float:
    """dz/dx = 1 - tanh^2(x / c); 1 when the softcap is off."""
    if softcap > 0:
        t = np.tanh(X / softcap)
        return 1.0 - t * t
    return 1.0


def _lse(Z: np.ndarray) -> np.ndarray:
    """Row log-sum-exp in the stable form m + log(sum exp(z - m))."""
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


def label_status(labels: np.ndarray, V: int, ignore_index: int):
    """(valid, bad) boolean masks: valid = not ignored and 0 <= y < V."""
    y = np.asarray(labels, dtype=np.int64)
    not_ignored = y != ignore_index
    in_range = (y >= 0) & (y < V)
    return not_ignored & in_range, not_ignored & ~in_range


def row_scale(valid: np.ndarray, n_valid: int, reduction: str, grad_out) -> np.ndarray:
    """Per-row factor that multiplies (softmax - onehot): g/n_valid, g, or g_i; 0 if ignored."""
    if reduction == "mean":
        s = np.full(valid.shape, (float(grad_out) / n_valid) if n_valid > 0 else 0.0)
    elif reduction == "sum":
        s = np.full(valid.shape, float(grad_out))
    elif reduction == "none":
        s = np.asarray(grad_out, dtype=np.float64).reshape(valid.shape).copy()
    else:
        raise ValueError(reduction)
    return np.where(valid, s, 0.0)


def _filter(P, labels, valid, filter_threshold):
    """Gradient filtering: softmax entries below the threshold are dropped, except the
    target entry of a valid row (Liger-CCE blog, §三: entries under 2^-12 vanish in the
    bf16 gradient and are skipped).  threshold <= 0: nothing is dropped."""
    if filter_threshold <= 0:
        return P
    keep = P >= filter_threshold
    rows = np.nonzero(valid)[0]
    keep[rows, np.asarray(labels)[rows]] = True
    return np.where(keep, P, 0.0)


def _dlogits(X, Z, lse, labels, valid, scale, softcap, filter_threshold=0.0):
    """dL/dx for a block of rows: (exp(z - lse) - onehot(y)) * scale * cap'(x)."""
    P = _filter(np.exp(Z - lse[:, None]), labels, valid, filter_threshold)
    rows = np.nonzero(valid)[0]
    P[rows, np.asarray(labels)[rows]] -= 1.0
    return P * scale[:, None] * _cap_grad(X, softcap)


# ----------------------------------------------------------------------------- forward
@dataclass
class Forward:
    loss: np.ndarray        # scalar (mean/sum) or [N] (none)
    lse: np.ndarray         # [N] float64, every row (ignored rows too)
    loss_rows: np.ndarray   # [N] per-row loss, 0 for ignored/bad rows
    target: np.ndarray      # [N] z_{i,y_i} (capped) for valid rows, 0 otherwise
    n_valid: int
    n_bad: int


def forward(Hf, Wf, labels, ignore_index: int = -100, softcap: float = 0.0,
            reduction: str = "mean", row_block: int = 512) -> Forward:
    """Loss, per-row LSE and counts.  Rows are independent, so they are visited in
    blocks of `row_block` purely to bound memory; nothing is merged across blocks."""
    Hf = np.asarray(Hf, dtype=np.float64)
    Wf = np.asarray(Wf, dtype=np.float64)
    labels = np.asarray(labels, dtype=np.int64)
    N, V = Hf.shape[0], Wf.shape[0]
    valid, bad = label_status(labels, V, ignore_index)
    lse = np.zeros(N)
    target = np.zeros(N)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Z = _cap(_raw_logits(Hf[r0:r1], Wf), softcap)
        lse[r0:r1] = _lse(Z)
        v = valid[r0:r1]
        idx = np.nonzero(v)[0]
        target[r0 + idx] = Z[idx, labels[r0:r1][idx]]
    loss_rows = np.where(valid, lse - target, 0.0)
    n_valid = int(valid.sum())
    if reduction == "mean":
        loss = np.float64(loss_rows.sum() / n_valid) if n_valid > 0 else np.float64(0.0)
    elif reduction == "sum":
        loss = np.float64(loss_rows.sum())
    elif reduction == "none":
        loss = loss_rows.copy()
    else:
        raise ValueError(reduction)
    return Forward(loss, lse, loss_rows, target, n_valid, int(bad.sum()))


def lse_rows(Hf, Wf, rows, softcap: float = 0.0) -> np.ndarray:
    """LSE of selected rows only (for sampled checks at large sizes)."""
    rows = np.asarray(rows, dtype=np.int64)
    return _lse(_cap(_raw_logits(np.asarray(Hf, np.float64)[rows], np.asarray(Wf, np.float64)), softcap))


def target_rows(Hf, Wf, labels, rows, ignore_index: int = -100, softcap: float = 0.0):
    """z_{i,y_i} of selected rows (0 where the row is not valid)."""
    Hf = np.asarray(Hf, np.float64)
    Wf = np.asarray(Wf, np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    y = np.asarray(labels, np.int64)[rows]
    valid, _ = label_status(y, Wf.shape[0], ignore_index)
    out = np.zeros(len(rows))
    for k in np.nonzero(valid)[0]:
        x = float(Hf[rows[k]] @ Wf[y[k]])
        out[k] = float(_cap(np.array([x]), softcap)[0])
    return out


# ----------------------------------------------------------------------------- backward
def backward(Hf, Wf, labels, lse, ignore_index: int = -100, softcap: float = 0.0,
             reduction: str = "mean", grad_out=1.0, row_block: int = 512, filter_threshold: float = 0.0):
    """(dH, dW) from the saved per-row LSE.  dH sums over the vocabulary, dW over
    the tokens; row blocks only bound memory.  filter_threshold > 0 gives the
    gradient of the filtered softmax (see _filter), an approximation of the exact one."""
    Hf = np.asarray(Hf, dtype=np.float64)
    Wf = np.asarray(Wf, dtype=np.float64)
    labels = np.asarray(labels, dtype=np.int64)
    N, V = Hf.shape[0], Wf.shape[0]
    valid, _ = label_status(labels, V, ignore_index)
    scale = row_scale(valid, int(valid.sum()), reduction, grad_out)
    dH = np.zeros_like(Hf)
    dW = np.zeros_like(Wf)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        X = _raw_logits(Hf[r0:r1], Wf)
        Z = _cap(X, softcap)
        dX = _dlogits(X, Z, np.asarray(lse)[r0:r1], labels[r0:r1], valid[r0:r1], scale[r0:r1], softcap,
                      filter_threshold)
        dH[r0:r1] = dX @ Wf
        dW += dX.T @ Hf[r0:r1]
    return dH, dW


def dH_rows(Hf, Wf, labels, lse, rows, ignore_index=-100, softcap=0.0, reduction="mean",
            grad_out=1.0, n_valid=None, filter_threshold=0.0):
    """dH for selected rows.  `lse` holds the oracle's LSE of those rows; `n_valid`
    is the global valid count (needed by the mean reduction)."""
    Hf = np.asarray(Hf, np.float64)
    Wf = np.asarray(Wf, np.float64)
    labels = np.asarray(labels, np.int64)
    rows = np.asarray(rows, np.int64)
    V = Wf.shape[0]
    valid_all, _ = label_status(labels, V, ignore_index)
    nv = int(valid_all.sum()) if n_valid is None else int(n_valid)
    g = grad_out if reduction != "none" else np.asarray(grad_out)[rows]
    valid = valid_all[rows]
    scale = row_scale(valid, nv, reduction, g)
    X = _raw_logits(Hf[rows], Wf)
    Z = _cap(X, softcap)
    dX = _dlogits(X, Z, np.asarray(lse, np.float64), labels[rows], valid, scale, softcap, filter_threshold)
    return dX @ Wf


def dW_rows(Hf, Wf, labels, lse_all, vocab, ignore_index=-100, softcap=0.0, reduction="mean",
            grad_out=1.0, filter_threshold=0.0):
    """dW for selected vocabulary rows v: sum over every token of dZ_iv h_i.
    Needs the oracle's LSE of all N rows."""
    Hf = np.asarray(Hf, np.float64)
    Wf = np.asarray(Wf, np.float64)
    labels = np.asarray(labels, np.int64)
    vocab = np.asarray(vocab, np.int64)
    V = Wf.shape[0]
    valid, _ = label_status(labels, V, ignore_index)
    scale = row_scale(valid, int(valid.sum()), reduction, grad_out)
    X = _raw_logits(Hf, Wf[vocab])                 # [N, |vocab|]
    Z = _cap(X, softcap)
    P = np.exp(Z - np.asarray(lse_all, np.float64)[:, None])
    onehot = (labels[:, None] == vocab[None, :]) & valid[:, None]
    if filter_threshold > 0:
        P = np.where((P >= filter_threshold) | onehot, P, 0.0)
    dX = (P - onehot) * scale[:, None] * _cap_grad(X, softcap)
    return dX.T @ Hf


# ----------------------------------------------------------------------------- blockwise
# ------------------------------------------------------------------ vocabulary order
def vocab_keys(Hf, Wf, vocab=None) -> np.ndarray:
    """Sort key of each vocabulary entry v: (1/N) sum_i x_iv, the raw logit h_i . w_v
    (before any softcap) averaged over all N rows, ignored rows included; 0 when N = 0
    (Liger-CCE blog, §三, the forward's per-word mean logit; which logit and which rows
    is a reading, the pages name neither).  ``vocab`` restricts the output to those ids."""
    Ws = Wf if vocab is None else Wf[np.asarray(vocab)]
    if Hf.shape[0] == 0:
        return np.zeros(Ws.shape[0])
    return _raw_logits(Hf, Ws).mean(axis=0)


def vocab_order(keys) -> np.ndarray:
    """The sorted vocabulary as a permutation: perm[p] is the id placed at position p.
    Keys descending (the frequent, high-logit words first); equal keys keep ascending
    id order, so the permutation is unique (Liger-CCE blog, §三)."""
    k = np.asarray(keys, dtype=np.float64)
    return np.lexsort((np.arange(k.size), -k)).astype(np.int64)


def merge(m1, s1, m2, s2):
    """Merge two (running max, scaled sum) pairs: m' = max(m1, m2),
    s' = s1 e^{m1-m'} + s2 e^{m2-m'}.  A side that has seen nothing (m = -inf, s = 0)
    contributes nothing, which is the "first block initialises directly" rule
    (ai-infra-kb M011, §05)."""
    m1 = np.asarray(m1, np.float64)
    m2 = np.asarray(m2, np.float64)
    m = np.maximum(m1, m2)
    with np.errstate(invalid="ignore"):
        a = np.where(np.isneginf(m1), 0.0, np.asarray(s1) * np.exp(m1 - m))
        b = np.where(np.isneginf(m2), 0.0, np.asarray(s2) * np.exp(m2 - m))
    return m, a + b


def tile_stats(Z: np.ndarray):
    """(m, s) of one vocabulary tile: its row max and sum of exp(z - m)."""
    m = Z.max(axis=1)
    return m, np.exp(Z - m[:, None]).sum(axis=1)


def forward_split(Hf, Wf, labels, row_chunks, vocab_chunks, ignore_index=-100, softcap=0.0,
                  reduction="mean"):
    """Blockwise forward: rows in chunks of the given sizes, vocabulary in tiles of the
    given sizes, (m, s) merged tile by tile, target picked in the tile holding it,
    per-row losses summed and divided once by the global valid count.  Self-test only."""
    Hf = np.asarray(Hf, np.float64)
    Wf = np.asarray(Wf, np.float64)
    labels = np.asarray(labels, np.int64)
    N, V = Hf.shape[0], Wf.shape[0]
    assert sum(row_chunks) == N and sum(vocab_chunks) == V
    valid, _ = label_status(labels, V, ignore_index)
    lse = np.zeros(N)
    target = np.zeros(N)
    r0 = 0
    for rc in row_chunks:
        rows = slice(r0, r0 + rc)
        m = np.full(rc, -np.inf)
        s = np.zeros(rc)
        v0 = 0
        for vc in vocab_chunks:
            Z = _cap(Hf[rows] @ Wf[v0:v0 + vc].T, softcap)
            mb, sb = tile_stats(Z)
            m, s = merge(m, s, mb, sb)
            y = labels[rows]
            hit = valid[rows] & (y >= v0) & (y < v0 + vc)
            idx = np.nonzero(hit)[0]
            target[r0 + idx] = Z[idx, y[idx] - v0]
            v0 += vc
        lse[rows] = m + np.log(s)
        r0 += rc
    loss_rows = np.where(valid, lse - target, 0.0)
    n_valid = int(valid.sum())
    total = 0.0
    r0 = 0
    for rc in row_chunks:                  # chunk sums, then one division
        total += loss_rows[r0:r0 + rc].sum()
        r0 += rc
    if reduction == "mean":
        loss = total / n_valid if n_valid > 0 else 0.0
    elif reduction == "sum":
        loss = total
    else:
        loss = loss_rows
    return Forward(np.float64(loss) if reduction != "none" else loss, lse, loss_rows, target,
                   n_valid, int((~valid & (labels != ignore_index)).sum()))
