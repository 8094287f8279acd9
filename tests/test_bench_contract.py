"""The one-line JSON contract of bench.py, run as a subprocess on the small workload.

The reference arm (the fp64 oracle on host cores) runs on CPU; our arm needs the GPU.
Both must print one JSON line as the last line of stdout with the keys the benchmark
driver reads (metric, value, unit, n_gpus, steps, warmup, ms_per_step,
higher_is_better, scaling, vs_baseline, dtype, data, config, e2e, ...)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
          "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline")


def _bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def _common(d, steps, warmup):
    for k in COMMON:
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == "tokens/s" and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["vs_baseline"] is None and "workload" in d["config"] and "model" not in d["config"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert {"h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(e)


def test_reference_arm_line():
    d = _bench("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3", "--ref-sample", "16")
    _common(d, 2, 3)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] == d["value"] and "sample" in c
    assert "cores online" in c["cpu_model"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--warmup", "2"], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


@pytest.mark.gpu
def test_our_arm_line():
    d = _bench("--config", "tiny", "--steps", "5", "--warmup", "3", "--cpu-sample", "32")
    _common(d, 5, 3)
    assert "impl" not in d and d["dtype"] == "bf16"
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0 and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and "traffic" in r
    clk = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)
    assert d["gpu_launches"] >= 5 * 8  # at least the eight kernels of a one-chunk step, per step
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 4
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and "sample" in c
    assert "cores online" in c["cpu_model"]
    assert d["peak_extra_mb"] >= 0


@pytest.mark.gpu
def test_two_rank_data_parallel_line():
    """bench.py's N > 1 path (dist.data_parallel_step with its exchange and dW all-reduce),
    launched the way the driver launches it, with two ranks on the one GPU of this machine.
    The exchange goes through gloo (host copies): NCCL wants one GPU per rank.  The
    kernels of the two ranks never wait on each other; only the host-side collectives
    do.  This checks the code path and the JSON line, not multi-GPU performance."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--steps", "3", "--warmup", "3", "--config", "tiny", "--dist-backend", "gloo",
           "--no-cpu-baseline"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in COMMON:
        assert k in d, k
    assert d["n_gpus"] == 2 and d["scaling"] == "weak" and d["config"]["global_batch"] == 2 * 256
    c = d["collectives"]
    assert set(c["ms_per_step"]) == {"counts", "dW"} and 0 < c["share_of_step"] < 1
    assert d["e2e"]["value"] > 0 and "data_parallel_step" in d["e2e"]["path"]
