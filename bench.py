"""Benchmark of the fused linear + cross-entropy forward + backward on GB300.

One step = one forward and one backward pass of the whole path (label scan and
indexed dot, tensor-core linear-LSE, merge and reduction, dZ recompute, dW and dH)
over one synthetic batch.  Default workload: the Llama-3-shaped head, N=8192 tokens,
Hd=4096, V=128256, bf16, Zipf(1.1) labels with 5% ignored, mean reduction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama3] [--impl ours|reference]

Under torchrun (N > 1) the step is token-sharded data parallel (weak scaling): every
rank holds the same W and its own batch of N rows, and each step runs
``dist.data_parallel_step`` — the local forward, an all-reduce of the valid counts and
loss sums (the global mean divides once by the global valid count), the local backward
scaled by that count, and an all-reduce of dW — with NCCL (``--dist-backend``).  Rank 0
prints one JSON line with the collectives' share of the step.  ``--impl reference``
times the fp64 CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused linear-CE fwd+bwd tokens/s at 1 GB300; % of bf16 tensor peak; peak extra MB"
L2_BYTES = 129 * 10**6

# DRAM traffic per launch of the dominant kernel class from one ncu capture, keyed by
# the kernel class, the workload, the backward chunk budget (a per-chunk launch's traffic
# depends on its width) and the hash of the kernel sources it was taken on (null once the
# sources change, or for a budget never captured).
MEASURED_TRAFFIC = {
    # ncu capture of the four tensor-core kernels at the llama2 size (DRAM read + written
    # per launch), scaled by tiles per launch to llama3 with 1 GiB chunks: x 4.008 for the
    # linear-LSE launch (501 / 125 vocabulary tiles), x 2.004 for the per-chunk dZ / dW / dH
    # launches; both sizes have 32 token tiles, so the banded schedules stream W twice per
    # launch in both
    ("linear_lse", "llama3", 1 << 30, "226080fb59c1dd05"): 3.31e9,   # 0.822 + 0.004 GB at llama2
    ("dz", "llama3", 1 << 30, "226080fb59c1dd05"): 2.38e9,           # 0.683 + 0.505 GB
    ("dw", "llama3", 1 << 30, "226080fb59c1dd05"): 5.12e9,           # 2.300 + 0.257 GB
    ("dh", "llama3", 1 << 30, "226080fb59c1dd05"): 5.03e9,           # 2.446 + 0.063 GB
    # direct ncu capture at llama3 with the 512 MiB default (4 chunks of 126 / 125
    # vocabulary tiles), mean of two launches per kernel, DRAM read + written
    ("linear_lse", "llama3", 512 << 20, "226080fb59c1dd05"): 4.43e9,  # 4.421 + 0.010 GB
    ("dz", "llama3", 512 << 20, "226080fb59c1dd05"): 1.19e9,          # 0.685 + 0.506 GB
    ("dw", "llama3", 512 << 20, "226080fb59c1dd05"): 2.60e9,          # 2.342 + 0.256 GB
    ("dh", "llama3", 512 << 20, "226080fb59c1dd05"): 2.68e9,          # 2.586 + 0.091 GB
    # the same capture after the backward's row compaction (dZ and dH walk 31 of 32 token
    # tiles and dW 122 of 128 K steps at the llama3 workload's 7756 rows with a gradient)
    ("linear_lse", "llama3", 512 << 20, "be3b667aaba63e36"): 6.46e9,  # 6.454 + 0.010 GB
    ("dz", "llama3", 512 << 20, "be3b667aaba63e36"): 1.20e9,          # 0.716 + 0.488 GB
    ("dw", "llama3", 512 << 20, "be3b667aaba63e36"): 2.26e9,          # 2.010 + 0.255 GB
    ("dh", "llama3", 512 << 20, "be3b667aaba63e36"): 2.66e9,          # 2.570 + 0.092 GB
}
DEFAULT_CHUNK_BUDGET = 512 << 20  # the library's default (flce_api.cu)


# the sources that define the tensor-core kernels (engine, PTX wrappers, tile constants
# and epilogue parameters, their two translation units)
TC_KERNEL_SOURCES = ("gemm_bwd.cu", "gemm_fwd.cu", "internal.cuh", "ptx.cuh", "tc_gemm.cuh")


def kernel_source_hash(root: str = ROOT) -> str:
    h = hashlib.sha256()
    for name in TC_KERNEL_SOURCES:
        with open(os.path.join(root, "linear_cross_entropy_indexed_gb300", "csrc", name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    sm_max=d.get("sm_max_mhz"), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max=2070.0, source="fallback")


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", "flce_clocks_%d_%d.csv" % (os.getpid(), device_index))

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()
        return False

    def summary(self, sm_max_default=None, window=None):
        """Median SM clock over the samples taken inside `window` (host wall-clock start
        and end of the timed region; all samples if none falls inside), the highest max
        clock, and every throttle reason seen in any sample."""
        out = {"sm_mhz": None, "sm_max_mhz": sm_max_default, "reasons": [], "samples": 0}
        if self.proc is None or not os.path.exists(self.path):
            out["reasons"] = ["clock sampling unavailable"]
            return out
        rows, reasons = [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = None
            try:
                rows.append((t, float(parts[2]), float(parts[3])))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if rows:
            inside = [r for r in rows if window and r[0] is not None and window[0] <= r[0] <= window[1]]
            use = inside or rows
            out.update(sm_mhz=statistics.median(r[1] for r in use), sm_max_mhz=max(r[2] for r in rows),
                       samples=len(use), samples_all=len(rows),
                       window="timed region" if inside else "all samples (none inside the timed region)")
        out["reasons"] = sorted(reasons)
        return out


# ---------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workload_desc(w) -> str:
    s = "%s: N=%d tokens, Hd=%d, V=%d, labels %s" % (w.name, w.N, w.Hd, w.V, w.labels)
    if w.softcap > 0:
        s += ", softcap %.1f" % w.softcap
    if w.peak > 0:
        s += ", target logit raised by %g" % w.peak
    if w.unigram > 0:
        s += ", unigram prior slope %g" % w.unigram
    return s


def oracle_sample_step(Hf, Wf, y, w):
    import oracle as O
    ref = O.forward(Hf, Wf, y, w.ignore_index, w.softcap, w.reduction)
    O.backward(Hf, Wf, y, ref.lse, w.ignore_index, w.softcap, w.reduction, 1.0)
    return ref


def blas_threads() -> int:
    """Threads numpy's BLAS actually uses: asked of the loaded OpenBLAS library itself,
    else the usual environment variables, else the core count."""
    import ctypes
    try:
        with open("/proc/self/maps") as fh:
            libs = sorted({l.split()[-1] for l in fh if "openblas" in l.lower() and "/" in l})
        for path in libs:
            lib = ctypes.CDLL(path)
            for name in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                         "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
                if hasattr(lib, name):
                    getattr(lib, name).restype = ctypes.c_int
                    n = int(getattr(lib, name)())
                    if n > 0:
                        return n
    except OSError:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), with the online core count."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                name = v.strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if name is None:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    k, _, v = line.partition(":")
                    if k.strip() in ("model name", "Model", "CPU part") and v.strip():
                        name = v.strip()
                        break
        except OSError:
            pass
    return "%s, %d cores online" % (name or "unknown CPU", os.cpu_count() or 0)


def cpu_baseline(w, sample_tokens: int, repeats: int = 1):
    """Time the fp64 oracle (as it stands) on the first `sample_tokens` rows of the
    workload: a full forward + backward of that smaller batch with the whole W."""
    import oracle as O
    import synthetic as S
    sample_tokens = min(sample_tokens, w.N)  # the tiny workload is timed in full
    Hb = S.make_H(w, rows=slice(0, sample_tokens))
    y = S.make_labels(w)[:sample_tokens]
    Hf = O.widen_bf16(Hb)
    Wf = O.widen_bf16(S.make_W(w))
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        oracle_sample_step(Hf, Wf, y, w)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return dict(value=sample_tokens / t, unit="tokens/s", cores=blas_threads(), cpu_model=cpu_model(), kind="oracle",
                sample="first %d of %d tokens of %s, full W [%d x %d]; fp64 forward + backward, %d run(s), "
                       "median %.2f s" % (sample_tokens, w.N, w.name, w.V, w.Hd, repeats, t),
                seconds=t)


# ---------------------------------------------------------------------------- reference arm
def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as O
    import synthetic as S
    n = min(args.ref_sample, w.N)
    Hf = O.widen_bf16(S.make_H(w, rows=slice(0, n)))
    y = S.make_labels(w)[:n]
    Wf = O.widen_bf16(S.make_W(w))
    for _ in range(args.warmup):
        oracle_sample_step(Hf, Wf, y, w)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(Hf, Wf, y, w)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w), "sample_tokens_per_step": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": "first %d tokens of %s per step, full W" % (n, w.name)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- our arm
def run_ours(args, w):
    import torch
    import synthetic as S
    import linear_cross_entropy_indexed_gb300 as F

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local % torch.cuda.device_count())
        dist.init_process_group(args.dist_backend)
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()

    # inputs resident in HBM: the same W on every rank (replicated weights), each rank its
    # own batch of H and labels (seed offset by rank)
    wr = S.scaled(w.name, seed=w.seed + 1000 * rank) if rank else w
    Wb = S.make_W(w)
    Hb, yb = S.make_H(wr, W=Wb), S.make_labels(wr)
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    H, W = to_dev(Hb), to_dev(Wb)
    y = torch.from_numpy(yb).to(dev)
    N, Hd, V = w.N, w.Hd, w.V
    red = w.reduction
    budget = args.chunk_budget
    ws_bytes = max(F.forward_workspace_size(N, Hd, V),
                   F.backward_workspace_size(N, Hd, V, budget, args.sort_vocab, args.compensated))
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    dH = torch.empty_like(H)
    dW = torch.empty_like(W)
    g = torch.ones(1, dtype=torch.float32, device=dev)

    # collectives of the data-parallel step, timed with events on the launch stream while
    # `coll_on` holds (the timed region)
    coll, coll_on = [], [False]

    class CollTimer:
        def __init__(self, name):
            self.name = name

        def __enter__(self):
            if coll_on[0]:
                self.e0 = torch.cuda.Event(enable_timing=True)
                self.e0.record()
            return self

        def __exit__(self, *a):
            if coll_on[0]:
                e1 = torch.cuda.Event(enable_timing=True)
                e1.record()
                coll.append((self.name, self.e0, e1))
            return False

    def step():
        if ws > 1:
            from linear_cross_entropy_indexed_gb300.dist import data_parallel_step
            loss, _, _, counts = data_parallel_step(
                H, W, y, g, w.ignore_index, w.softcap, timer=CollTimer, workspace=workspace, chunk_budget=budget,
                dH=dH, dW=dW, filter_threshold=args.filter_threshold, sort_vocab=args.sort_vocab,
                compensated=args.compensated)
            return loss, counts
        loss, lse, counts, _ = F.flce_forward(H, W, y, w.ignore_index, w.softcap, red, workspace=workspace)
        F.flce_backward(H, W, y, lse, counts, g, w.ignore_index, w.softcap, red, budget, workspace=workspace,
                        dH=dH, dW=dW, filter_threshold=args.filter_threshold, sort_vocab=args.sort_vocab,
                        compensated=args.compensated)
        return loss, counts

    for _ in range(args.warmup):
        n0 = F.launch_count()
        loss, counts = step()
        launches_per_step = F.launch_count() - n0
    torch.cuda.synchronize()
    F.check_counts(counts)

    # timed region: inputs (W 1 GB) larger than L2, so no flush is needed between steps
    stream = torch.cuda.current_stream(dev)
    n_launch0 = F.launch_count()
    per_step = None
    sink = F.EventSink(capacity=args.steps * launches_per_step + 16)
    with ClockSampler(dev.index) as clk:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        t_begin = time.time()
        coll_on[0] = True
        with sink:
            e0.record(stream)
            for _ in range(args.steps):
                loss, counts = step()
            e1.record(stream)
        coll_on[0] = False
        torch.cuda.synchronize()
        t_end = time.time()
        if ws > 1:
            torch.distributed.barrier()
    launches = F.launch_count() - n_launch0
    if sink.used < launches:
        raise RuntimeError("event sink overflow: %d of %d launches recorded" % (sink.used, launches))
    ms = e0.elapsed_time(e1) / args.steps
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    F.check_counts(counts)
    clocks = clk.summary(peaks["sm_max"], window=(t_begin, t_end))
    # The backward runs on the rows that carry a gradient only (the rest are exact zeros):
    # its useful work is 6 * Nv * Hd * V, Nv this rank's rows with a valid label.
    nv_rank = int(((yb != w.ignore_index) & (yb >= 0) & (yb < V)).sum())

    # the data-parallel collectives' time per step (events on the launch stream around each)
    coll_summary = None
    if ws > 1:
        per = {}
        for name, a, b in coll:
            per[name] = per.get(name, 0.0) + a.elapsed_time(b)
        tot = sum(per.values()) / args.steps
        coll_summary = {"ms_per_step": {k: v / args.steps for k, v in sorted(per.items())},
                        "share_of_step": tot / ms, "backend": args.dist_backend,
                        "what": "all-reduce of counts and per-rank loss sums (global mean), all-reduce of dW"}

    # per kernel class time inside the timed region (events on the launch stream)
    per_class = {}
    for name, d in sink.durations_ms():
        c = per_class.setdefault(name, [0, 0.0])
        c[0] += 1
        c[1] += d
    # per step: from the first launch's start event to the last launch's end event (every
    # step launches the same kernels), reported as median and [0.2, 0.8] quantiles
    L = launches // args.steps
    step_ms = sorted(sink.start[k * L].elapsed_time(sink.end[(k + 1) * L - 1]) for k in range(args.steps))
    q = lambda f: step_ms[min(len(step_ms) - 1, int(round(f * (len(step_ms) - 1))))]
    fwd_classes = ("label_dot", "linear_lse", "lse_merge", "reduce")
    fwd_ms = sum(v[1] for k, v in per_class.items() if k in fwd_classes) / args.steps
    bwd_ms = sum(v[1] for k, v in per_class.items() if k not in fwd_classes) / args.steps
    # per step, summed over that class's launches; the compensated backward multiplies both
    # the bf16 value and the rounding remainder of dZ, twice the dW and dH products
    prod = 4.0 if args.compensated else 2.0
    flops_per_class = {"linear_lse": 2.0 * N * Hd * V, "dz": 2.0 * nv_rank * Hd * V, "dw": prod * nv_rank * Hd * V,
                       "dh": prod * nv_rank * Hd * V}
    # the dominant tensor-core kernel class (at every real workload also the dominant class
    # overall; at tiny sizes a latency-bound small kernel can take longer)
    tc = [k for k in per_class if k in flops_per_class]
    dom = max(tc, key=lambda k: per_class[k][1]) if tc else None
    roof = None
    if dom is not None:
        launches_dom, tot_ms = per_class[dom]
        per_launch_ms = tot_ms / launches_dom
        per_launch_flops = flops_per_class[dom] * args.steps / launches_dom
        achieved = per_launch_flops / (per_launch_ms * 1e-3) / 1e12
        h = kernel_source_hash()
        traffic = MEASURED_TRAFFIC.get((dom, w.name, budget or DEFAULT_CHUNK_BUDGET, h))
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["bf16_sus"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_sus"], "traffic": traffic,
                "peak_kind": "bf16_tflops_sustained (%s)" % peaks["source"],
                "frac_of_burst": achieved / peaks["bf16"], "launches": launches_dom,
                "ms_per_launch": per_launch_ms}

    # end to end through the public API with host buffers: every step copies its inputs
    # (H, W, labels) from pinned host memory, runs the autograd forward + backward and reads
    # the loss back to the host.  The copy of step i+1 runs on a second stream while step i
    # computes (double-buffered device inputs), as a training loop would prefetch its next
    # batch, through the library's staging call (SM loads from the pinned buffers: a
    # copy-engine transfer from host memory slows the running kernels several times more);
    # the loss goes to pinned host memory asynchronously and the host reads step i's value
    # once step i+1 is enqueued, so the GPU never waits for the host between steps.
    e2e = None
    if not args.no_e2e:
        Hh = torch.from_numpy(np.ascontiguousarray(Hb).view(np.int16)).view(torch.bfloat16).pin_memory()
        Wh = torch.from_numpy(np.ascontiguousarray(Wb).view(np.int16)).view(torch.bfloat16).pin_memory()
        yh = torch.from_numpy(yb).pin_memory()
        bufs = [(torch.empty_like(H), torch.empty_like(W), torch.empty_like(y)) for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        loss_host = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
        loss_ready = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def enqueue_copy(i):
            b = bufs[i % 2]
            with torch.cuda.stream(copy_stream):
                if used[i % 2]:
                    copy_stream.wait_event(freed[i % 2])  # the buffer's previous step is done
                F.stage_h2d(b[0], Hh)  # SM loads from the pinned buffers (the library's staging call)
                F.stage_h2d(b[1], Wh)
                F.stage_h2d(b[2], yh)
                copied[i % 2].record(copy_stream)

        def compute(i):
            b = bufs[i % 2]
            cur = torch.cuda.current_stream(dev)
            cur.wait_event(copied[i % 2])
            if ws > 1:  # the public data-parallel step: exchange of counts and loss, dW all-reduce
                from linear_cross_entropy_indexed_gb300.dist import data_parallel_step
                loss, _, _, _ = data_parallel_step(
                    b[0], b[1], b[2], g, w.ignore_index, w.softcap, chunk_budget=budget,
                    filter_threshold=args.filter_threshold, sort_vocab=args.sort_vocab, compensated=args.compensated)
            else:
                Hx = b[0].detach().requires_grad_(True)
                Wx = b[1].detach().requires_grad_(True)
                loss = F.linear_cross_entropy(Hx, Wx, b[2], w.ignore_index, w.softcap, red, budget,
                                              args.filter_threshold, args.sort_vocab, args.compensated)
                loss.backward()
            freed[i % 2].record(cur)
            loss_host[i % 2].copy_(loss.detach().reshape(1), non_blocking=True)
            loss_ready[i % 2].record(cur)
            used[i % 2] = True

        def read_loss(i):
            loss_ready[i % 2].synchronize()
            return float(loss_host[i % 2][0])

        def run(k):
            losses = []
            enqueue_copy(0)
            for i in range(k):
                if i + 1 < k:
                    enqueue_copy(i + 1)
                compute(i)
                if i > 0:  # step i is enqueued: now wait for step i-1's loss
                    losses.append(read_loss(i - 1))
            losses.append(read_loss(k - 1))
            return losses

        run(3)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(copy_stream)
        enqueue_copy(0)
        c1.record(copy_stream)
        torch.cuda.synchronize()
        h2d_ms = c0.elapsed_time(c1)
        k2 = max(3, args.steps)
        torch.cuda.synchronize()
        with ClockSampler(dev.index) as clk_e2e:
            t0 = time.perf_counter()
            w0 = time.time()
            losses = run(k2)
            torch.cuda.synchronize()
            e2e_ms = 1e3 * (time.perf_counter() - t0) / k2
            w1 = time.time()
        e2e_clocks = clk_e2e.summary(peaks["sm_max"], window=(w0, w1))
        if not all(np.isfinite(losses)):
            raise RuntimeError("non-finite loss in the end-to-end loop")
        if ws > 1:
            t = torch.tensor([e2e_ms], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_ms = float(t.item())
        bi = Hh.numel() * 2 + Wh.numel() * 2 + yh.numel() * 8
        e2e = {"value": ws * N / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": 4, "ms_per_step": e2e_ms, "steps": k2, "h2d_ms_per_step": h2d_ms,
               "clocks": e2e_clocks,
               "path": ("dist.data_parallel_step() (NCCL exchange of counts and loss, dW all-reduce)" if ws > 1 else
                        "linear_cross_entropy() autograd") +
                       "; pinned H, W, labels copied every step by stage_h2d() on a second "
                       "stream (next step's copy overlaps this step's compute); every step's loss copied to pinned host "
                       "memory and read on the host once the next step is enqueued"}

    # peak extra device memory of one forward + backward through the public API
    torch.cuda.synchronize()
    Hx = H.detach().requires_grad_(True)
    Wx = W.detach().requires_grad_(True)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    loss = F.linear_cross_entropy(Hx, Wx, y, w.ignore_index, w.softcap, red, budget, args.filter_threshold,
                                  args.sort_vocab, args.compensated)
    loss.backward()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated(dev) - base
    required = H.numel() * 2 + W.numel() * 2 + 4 * N + 4 + 24  # dH, dW, lse, loss, counts
    peak_extra_mb = (peak - required) / 2**20
    del Hx, Wx, loss

    line = None
    if rank == 0:
        value = ws * N / (ms * 1e-3)
        flops = (2.0 * N + 6.0 * nv_rank) * Hd * V   # useful work: the backward skips rows without a gradient
        flops_nominal = 8.0 * N * Hd * V
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(w), "global_batch": ws * N, "seq_len": 4096 if N >= 4096 else N,
                       "parallelism": "dp%d" % ws if ws > 1 else "single",
                       "l2": "inputs larger than L2 (W %.0f MiB > 129 MB); no flush" % (W.numel() * 2 / 2**20),
                       "chunk_budget_bytes": budget or DEFAULT_CHUNK_BUDGET,
                       "filter_threshold": args.filter_threshold, "sort_vocab": args.sort_vocab,
                       "compensated": args.compensated},
            # useful work of the exact path: the forward over all N rows, the backward over the Nv
            # rows with a valid label (the others have an exactly zero gradient and are skipped);
            # a filtered run skips part of the backward too
            "flops_basis": "(2*N + 6*Nv)*Hd*V, Nv = %d of N = %d rows carry a gradient" % (nv_rank, N)
                           + (" (exact work; filtering skips some)" if args.filter_threshold > 0 else "")
                           + (" (the compensated mode runs (2*N + 10*Nv)*Hd*V)" if args.compensated else ""),
            "pct_bf16_peak": 100.0 * flops / (ms * 1e-3) / (peaks["bf16"] * 1e12),
            "pct_bf16_peak_sustained": 100.0 * flops / (ms * 1e-3) / (peaks["bf16_sus"] * 1e12),
            "pct_bf16_peak_nominal": 100.0 * flops_nominal / (ms * 1e-3) / (peaks["bf16"] * 1e12),
            "peak_extra_mb": peak_extra_mb,
            "workspace_mb": ws_bytes / 2**20,
            "clocks": clocks, "e2e": e2e, "gpu_launches": launches, "roofline": roof,
            "kernel_ms_per_step": {k: v[1] / args.steps for k, v in sorted(per_class.items())},
            "collectives": coll_summary,
            "step_ms": {"median": q(0.5), "q20": q(0.2), "q80": q(0.8),
                        "forward_kernels": fwd_ms, "backward_kernels": bwd_ms},
        }
    if ws > 1:
        torch.distributed.barrier()
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = {k: v for k, v in cpu_baseline(w, args.cpu_sample).items() if k != "seconds"}
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="llama3")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--chunk-budget", type=int, default=0)
    ap.add_argument("--filter-threshold", type=float, default=0.0,
                    help="gradient filtering threshold (0 = exact backward; e.g. 2**-12 = 0.000244140625)")
    ap.add_argument("--sort-vocab", action="store_true",
                    help="backward walks the vocabulary in mean-logit order (pays with --filter-threshold)")
    ap.add_argument("--compensated", action="store_true",
                    help="backward carries dZ's bf16 rounding remainder (twice the dW / dH work)")
    ap.add_argument("--cpu-sample", type=int, default=1024)
    ap.add_argument("--ref-sample", type=int, default=64)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dist-backend", default="nccl", choices=["nccl", "gloo"],
                    help="process-group backend of the data-parallel exchange when N > 1 (gloo: host copies)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    import synthetic as S
    w = S.WORKLOADS[args.config]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
