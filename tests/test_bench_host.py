"""Host-side logic of the benchmark that needs no GPU: which nvidia-smi
samples count as "during the timed region"."""
import datetime
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def line(t, sm, power, power_cap=False, thermal=False):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    act = "Active" if power_cap else "Not Active"
    th = "Active" if thermal else "Not Active"
    return "%s, %d, 2070, %.1f, 0x0, Not Active, %s, Not Active, %s\n" % (stamp, sm, power, th,
                                                                       act)


class _Done:
    def poll(self):
        return 0


def sampler(bench, rows):
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.lines = [(t + 5.0, line(t, *rest)) for t, *rest in rows]
    return s


def test_window_keeps_only_samples_inside_the_timed_region():
    bench = load_bench()
    t0 = 1_800_000_000.0
    rows = [(t0 - 1.0, 2070, 90.0), (t0 - 0.5, 2070, 95.0, False, True),  # idle, before
            (t0 + 0.05, 1900, 1300.0, True), (t0 + 0.10, 1850, 1390.0, True),
            (t0 + 0.15, 1880, 1350.0, True),
            (t0 + 2.0, 2070, 100.0, False, True)]  # idle, after
    w = sampler(bench, rows).window(t0, t0 + 0.2)
    assert w["samples"] == 3 and w["window"] == "timed region"
    assert w["sm_mhz"] == 1880 and w["sm_max_mhz"] == 2070
    assert w["reasons"] == ["sw_power_cap"]  # the thermal flags outside are not counted
    assert w["power_w_median"] == 1350.0 and w["power_w_max"] == 1390.0


def test_short_region_takes_the_nearest_samples_and_says_so():
    bench = load_bench()
    t0 = 1_800_000_000.0
    rows = [(t0 - 0.1, 1950, 800.0), (t0 + 0.06, 1900, 1200.0, True), (t0 + 1.0, 2070, 90.0)]
    w = sampler(bench, rows).window(t0, t0 + 0.01)
    assert w["samples"] == 2 and w["window"].startswith("timed region +-")
    assert w["reasons"] == ["sw_power_cap"]


def test_no_samples_is_reported_not_invented():
    bench = load_bench()
    w = sampler(bench, [(1_800_000_000.0, 2070, 90.0)]).window(1_900_000_000.0, 1_900_000_001.0)
    assert w["sm_mhz"] is None and w["samples"] == 0


def test_unparseable_timestamp_falls_back_to_arrival_time():
    bench = load_bench()
    s = bench.ClockSampler(0)
    s.proc = _Done()
    t0 = 1_800_000_000.0
    s.lines = [(t0 + 0.1, "12:00:00, 1800, 2070, 1000.0, 0x0, Not Active, Not Active, "
                          "Not Active, Not Active\n")]
    w = s.window(t0, t0 + 0.2)
    assert w["samples"] == 1 and w["sm_mhz"] == 1800 and w["reasons"] == []


def test_roofline_takes_the_binding_bound(monkeypatch):
    """A launch is measured against the tensor peak when its flops take longer
    at peak than its algorithmic bytes at copy bandwidth, else against HBM."""
    bench = load_bench()
    monkeypatch.setattr(bench, "peaks", lambda: ({"bf16_tflops": 2000.0,
                                                   "bf16_tflops_sustained": 1800.0,
                                                   "hbm_gbs": 8000.0}, "measured"))
    # 8192^3 with four 128 MiB inputs and two outputs: 550 us at peak vs 100 us of bytes
    big = bench.roofline(2.0 * 8192 ** 3, 805306368, 0.70, 123)
    assert big["bound"] == "tensor" and big["unit"] == "TFLOP/s" and big["traffic"] == 123
    assert abs(big["achieved"] - 2.0 * 8192 ** 3 / 0.70e-3 / 1e12) < 1e-6
    assert abs(big["frac"] - big["achieved"] / 2000.0) < 1e-12
    assert abs(big["frac_of_sustained"] - big["achieved"] / 1800.0) < 1e-12
    # 1024^3 with 10 MiB of operands: 1.07 us at peak vs 1.31 us of bytes
    small = bench.roofline(2.0 * 1024 ** 3, 10485760, 0.0148, None)
    assert small["bound"] == "hbm" and small["unit"] == "GB/s" and small["peak"] == 8000.0
    assert abs(small["achieved"] - 10485760 / 0.0148e-3 / 1e9) < 1e-6
    assert abs(small["frac"] - small["hbm_frac"]) < 1e-12 and small["tensor_frac"] < small["frac"]


def test_numa_pages_of_a_host_buffer_are_found():
    """The end-to-end leg reports which NUMA nodes hold its pinned buffers;
    on any Linux host a touched buffer's pages are found on some node."""
    import numpy as np
    bench = load_bench()
    if not os.path.exists("/proc/self/numa_maps"):
        return
    a = np.ones(1 << 20)
    nodes = bench._numa_nodes_of(a.ctypes.data, a.ctypes.data + a.nbytes)
    assert nodes and sum(nodes.values()) >= a.nbytes // (1 << 21)
