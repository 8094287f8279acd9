"""The dH K split against the fp64 oracle.

When a dH launch has few 256 x 256 output tiles, the backward splits every tile's
vocabulary range into 2 to 4 parts run as separate units and adds the parts' fp32 sums in
part order (k_dh_combine).  These cases pick shapes for each split count (checked through
the kernel sequence the event sink records: one combining pass per chunk) and compare dH
and dW with the oracle, single- and multi-chunk, and for the vocabulary-sharded backward,
whose fp32 dH partial receives the combined sums."""
import numpy as np
import pytest
import torch

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _run(w, chunk_budget=0):
    import linear_cross_entropy_indexed_gb300 as F
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    g = torch.ones(1, device="cuda")
    sink = F.EventSink(capacity=256)
    with sink:
        dH, dW = F.flce_backward(H, W, lab, lse, counts, g, chunk_budget=chunk_budget)
    torch.cuda.synchronize()
    names = [n for n, _ in sink.durations_ms()]
    ref, dH_ref, dW_ref = P.oracle_full(Hb, Wb, y)
    got = dict(dH=S.bf16_bits_to_f32(P.bf16_bits(dH)).astype(np.float64),
               dW=S.bf16_bits_to_f32(P.bf16_bits(dW)).astype(np.float64), counts_after=counts.cpu().numpy())
    P.check_backward(got, dH_ref, dW_ref)
    return names


def test_two_parts_at_256_tiles():
    # 4096 x 4096: 16 x 16 = 256 dH tiles, 4 waves of 76 pairs whole, 3.5 split in 2
    w = S.scaled("llama3", N=4096, Hd=4096, V=1000, seed=71)
    names = _run(w)
    assert names.count("dh") == 1 and names.count("dh_combine") == 1


def test_three_parts_at_50_tiles():
    # 1280 x 2560: 5 x 10 = 50 tiles; 3 parts take 150 units in 2 waves of a third each
    w = S.scaled("llama3", N=1280, Hd=2560, V=3000, seed=72)
    names = _run(w)
    assert names.count("dh_combine") == 1


def test_split_across_vocabulary_chunks():
    # 256 tiles split in 2, and 4 vocabulary chunks: each chunk's parts join the fp32
    # running sum, the last chunk's go to the bf16 dH
    N, Hd, V = 4096, 4096, 2000
    w = S.scaled("llama3", N=N, Hd=Hd, V=V, seed=73)
    names = _run(w, chunk_budget=N * 2 * 512)
    assert names.count("dh") == 4 and names.count("dh_combine") == 4


def test_split_sharded_fp32_partial():
    import linear_cross_entropy_indexed_gb300 as F
    N, Hd, V = 1280, 2560, 3000
    w = S.scaled("llama3", N=N, Hd=Hd, V=V, seed=74)
    Hb, Wb, y = P.make_case(w)
    H, W = P.to_device(Hb), P.to_device(Wb)
    lab = torch.from_numpy(y).cuda()
    loss, lse, counts, _ = F.flce_forward(H, W, lab)
    g = torch.ones(1, device="cuda")
    cut = 1700
    parts = [F.flce_backward_shard(H, W[a:b].contiguous(), lab, lse, counts, g, a, V)
             for a, b in ((0, cut), (cut, V))]
    torch.cuda.synchronize()
    dh = sum(p[0].double().cpu().numpy() for p in parts)
    dw = np.concatenate([S.bf16_bits_to_f32(P.bf16_bits(p[1])).astype(np.float64) for p in parts])
    ref, dH_ref, dW_ref = P.oracle_full(Hb, Wb, y)
    assert P.fro_rel(dh, dH_ref) <= P.TOL_GRAD_FRO and P.fro_rel(dw, dW_ref) <= P.TOL_GRAD_FRO
    P.check_rows("dH", dh, dH_ref)
    P.check_rows("dW", dw, dW_ref)
    # the fp32 partials are summed before any bf16 rounding: close to the oracle
    assert P.fro_rel(dh, dH_ref) <= 5e-3
