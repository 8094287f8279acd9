"""World-size-2 gloo tests (CPU) of the multi-rank host logic.

Token-sharded data parallel: each rank runs the fp64 oracle on its rows as its local
step, the ranks exchange (loss sum, valid count) with the helpers of
``linear_cross_entropy_indexed_gb300.dist`` and all-reduce dW; the result must equal
the unsharded oracle.  The same holds for ``dist.data_parallel_step`` (the step
bench.py times with NCCL on N > 1 GPUs) with the oracle passed in as its forward and
backward.  Vocab-parallel: each rank holds a vocabulary shard, computes
per-row (max, sum, target) over it, and the ranks merge them in rank order with the
running (m, s) rule (ai-infra-kb M011 §05 and §07); the merged LSE and loss must equal
the unsharded oracle."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _data(N=37, Hd=6, V=53, seed=3, all_ignored_rank1=False):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, Hd))
    W = rng.standard_normal((V, Hd)) * 0.7
    y = rng.integers(0, V, N)
    y[rng.random(N) < 0.2] = -100
    if all_ignored_rank1:
        y[N // 2 + 1:] = -100
    return H, W, y


def _dp_worker(rank, world, port, q, all_ignored_rank1):
    import oracle as O
    from linear_cross_entropy_indexed_gb300.dist import allreduce_counts_, global_mean_loss, shard_rows
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        H, W, y = _data(all_ignored_rank1=all_ignored_rank1)
        sl = shard_rows(len(y), world, rank)
        f = O.forward(H[sl], W, y[sl], reduction="sum")
        counts = torch.tensor([f.n_valid, f.n_bad, 0], dtype=torch.int64)
        allreduce_counts_(counts)
        loss = global_mean_loss(torch.tensor(float(f.loss)), counts)
        g = 1.3
        n_glob = int(counts[0])
        # the backward's mean scale uses the global count: g / n_valid_global per valid row
        dH, dW = O.backward(H[sl], W, y[sl], f.lse, reduction="sum", grad_out=(g / n_glob if n_glob else 0.0))
        dWt = torch.from_numpy(dW)
        dist.all_reduce(dWt)
        q.put((rank, float(loss), int(counts[0]), sl.start, sl.stop, dH, dWt.numpy()))
    finally:
        dist.destroy_process_group()


def _oracle_forward(H, W, labels, ignore_index, softcap, reduction, workspace=None):
    """The fp64 oracle in the shape of flce_forward's return value (CPU tensors)."""
    import oracle as O
    f = O.forward(H.numpy(), W.numpy(), labels.numpy(), ignore_index, softcap, reduction)
    counts = torch.tensor([f.n_valid, f.n_bad, 0], dtype=torch.int64)
    return torch.tensor(float(f.loss), dtype=torch.float64), torch.from_numpy(f.lse), counts, None


def _oracle_backward(H, W, labels, lse, counts, grad_out, ignore_index, softcap, reduction, workspace=None):
    """The fp64 oracle in the shape of flce_backward: like the library, the mean scale is
    grad / counts[0] with whatever count counts holds (the global one after the exchange)."""
    import oracle as O
    assert reduction == "mean"
    n = int(counts[0])
    g = float(grad_out.reshape(-1)[0]) / n if n else 0.0
    dH, dW = O.backward(H.numpy(), W.numpy(), labels.numpy(), lse.numpy(), ignore_index, softcap, "sum", g)
    return torch.from_numpy(dH), torch.from_numpy(dW)


def _dp_step_worker(rank, world, port, q, all_ignored_rank1):
    from linear_cross_entropy_indexed_gb300.dist import data_parallel_step, shard_rows
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        H, W, y = _data(all_ignored_rank1=all_ignored_rank1)
        sl = shard_rows(len(y), world, rank)
        names = []

        class Timer:
            def __init__(self, name):
                names.append(name)

            def __enter__(self):
                return self

            def __exit__(self, *a):
                return False

        loss, dH, dW, counts = data_parallel_step(torch.from_numpy(H[sl]), torch.from_numpy(W), torch.from_numpy(y[sl]),
                                          grad_out=torch.tensor([1.3], dtype=torch.float64), softcap=0.0,
                                          forward=_oracle_forward, backward=_oracle_backward, timer=Timer)
        assert counts.tolist() == [int((y != -100).sum()), 0, 0]
        q.put((rank, float(loss), sl.start, sl.stop, dH.numpy(), dW.numpy(), names))
    finally:
        dist.destroy_process_group()


def _vp_worker(rank, world, port, q):
    import oracle as O
    from linear_cross_entropy_indexed_gb300.dist import shard_rows
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        H, W, y = _data()
        vs = shard_rows(W.shape[0], world, rank)
        Z = H @ W[vs].T
        m, s = O.tile_stats(Z)
        hit = (y >= vs.start) & (y < vs.stop)
        t = np.where(hit, Z[np.arange(len(y)), np.clip(y - vs.start, 0, Z.shape[1] - 1)], 0.0)
        stats = torch.from_numpy(np.stack([m, s, t]))
        gathered = [torch.zeros_like(stats) for _ in range(world)]
        dist.all_gather(gathered, stats)
        M = np.full(len(y), -np.inf)
        S = np.zeros(len(y))
        T = np.zeros(len(y))
        for r in range(world):                     # fixed rank order
            M, S = O.merge(M, S, gathered[r][0].numpy(), gathered[r][1].numpy())
            T += gathered[r][2].numpy()
        q.put((rank, M + np.log(S), T))
    finally:
        dist.destroy_process_group()


def _run(target, *args, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda r: r[0])


def test_shard_rows_cover_exactly():
    from linear_cross_entropy_indexed_gb300.dist import shard_rows
    for N in (0, 1, 7, 8192, 32769):
        for world in (1, 2, 3, 8):
            parts = [shard_rows(N, world, r) for r in range(world)]
            assert parts[0].start == 0 and parts[-1].stop == N
            assert all(a.stop == b.start for a, b in zip(parts, parts[1:]))
            sizes = [p.stop - p.start for p in parts]
            assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("all_ignored_rank1", [False, True])
def test_token_sharded_global_mean_matches_unsharded(all_ignored_rank1):
    import oracle as O
    res = _run(_dp_worker, all_ignored_rank1)
    H, W, y = _data(all_ignored_rank1=all_ignored_rank1)
    ref = O.forward(H, W, y)
    dH_ref, dW_ref = O.backward(H, W, y, ref.lse, grad_out=1.3)
    for rank, loss, n, a, b, dH, dW in res:
        assert n == ref.n_valid
        assert abs(loss - float(ref.loss)) <= 1e-6 * abs(float(ref.loss))
        np.testing.assert_allclose(dH, dH_ref[a:b], rtol=1e-10, atol=1e-14)
        np.testing.assert_allclose(dW, dW_ref, rtol=1e-10, atol=1e-14)


def test_vocab_parallel_merge_matches_unsharded():
    import oracle as O
    res = _run(_vp_worker)
    H, W, y = _data()
    ref = O.forward(H, W, y)
    valid = y != -100
    for rank, lse, t in res:
        np.testing.assert_allclose(lse, ref.lse, rtol=1e-12)
        np.testing.assert_allclose(t[valid], ref.target[valid], rtol=1e-12, atol=1e-14)
        loss = np.where(valid, lse - t, 0.0).sum() / valid.sum()
        assert abs(loss - float(ref.loss)) < 1e-12
        # a shard's own LSE alone (no exchange) is a different, wrong denominator
        Zr = H @ W[:W.shape[0] // 2].T
        own = Zr.max(1) + np.log(np.exp(Zr - Zr.max(1)[:, None]).sum(1))
        assert np.abs(own - ref.lse).max() > 0.1


@pytest.mark.parametrize("all_ignored_rank1", [False, True])
def test_data_parallel_step_matches_unsharded(all_ignored_rank1):
    """dist.data_parallel_step, the step bench.py times on N > 1 GPUs, with the fp64
    oracle standing in for the CUDA forward / backward: loss, every rank's dH rows and
    the all-reduced dW equal the unsharded oracle, also when one rank has no valid row."""
    import oracle as O
    res = _run(_dp_step_worker, all_ignored_rank1)
    H, W, y = _data(all_ignored_rank1=all_ignored_rank1)
    ref = O.forward(H, W, y)
    dH_ref, dW_ref = O.backward(H, W, y, ref.lse, grad_out=1.3)
    for rank, loss, a, b, dH, dW, names in res:
        assert abs(loss - float(ref.loss)) <= 1e-6 * abs(float(ref.loss))
        np.testing.assert_allclose(dH, dH_ref[a:b], rtol=1e-10, atol=1e-14)
        np.testing.assert_allclose(dW, dW_ref, rtol=1e-10, atol=1e-14)
        assert names == ["counts", "dW"]

