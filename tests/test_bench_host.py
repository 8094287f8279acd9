"""Host logic of bench.py that needs no GPU: the nvidia-smi clock summary (median SM
clock over the samples inside the timed region, every throttle reason seen) and the
kernel-source hash that keys the measured DRAM traffic."""
import datetime
import time

import bench


def _line(t, sm, smax=2070, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return "%s, 0, %d, %d, 812.5, 0x0, %s\n" % (stamp, sm, smax, ", ".join(reasons))


def _summary(lines, window):
    c = bench.ClockSampler(0)
    with open(c.path, "w") as f:
        f.writelines(lines)
    c.proc = object()  # as if nvidia-smi had run
    return c.summary(2070, window=window)


def test_clock_median_uses_only_samples_inside_the_timed_region():
    t0 = time.time()
    cap = ("Not Active", "Not Active", "Not Active", "Active")
    lines = [_line(t0 - 0.4, 2070), _line(t0 - 0.2, 2070),           # idle, before the region
             _line(t0 + 0.1, 1500, reasons=cap), _line(t0 + 0.2, 1520, reasons=cap), _line(t0 + 0.3, 1540, reasons=cap),
             _line(t0 + 0.9, 2070)]                                  # after the region
    s = _summary(lines, (t0, t0 + 0.5))
    assert s["sm_mhz"] == 1520 and s["samples"] == 3 and s["samples_all"] == 6
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"


def test_reasons_from_every_sample_and_fallback_to_all_samples():
    t0 = time.time()
    hot = ("Not Active", "Active", "Not Active", "Not Active")
    lines = [_line(t0 - 1.0, 1800, reasons=hot), _line(t0 - 0.9, 1900)]
    s = _summary(lines, (t0, t0 + 0.1))  # no sample inside the window
    assert s["sm_mhz"] == 1850 and s["samples"] == 2
    assert s["reasons"] == ["hw_thermal_slowdown"] and s["window"].startswith("all samples")


def test_unparsable_lines_are_skipped():
    t0 = time.time()
    lines = ["garbage\n", _line(t0 + 0.1, 1600), "0, 0, [N/A], 2070, 1, 0x0, a, b, c, d\n"]
    s = _summary(lines, (t0, t0 + 0.5))
    assert s["sm_mhz"] == 1600 and s["samples_all"] == 1


def test_kernel_source_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash() and len(h) == 16
    # the traffic table is keyed by kernel class, workload, chunk budget and that hash: a
    # stale entry, or a budget never captured, reads as unmeasured (null)
    assert all(len(k) == 4 and isinstance(k[2], int) and len(k[3]) == 16 for k in bench.MEASURED_TRAFFIC)
