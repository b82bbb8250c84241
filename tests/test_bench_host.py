"""Host-side logic of the benchmark that needs no GPU: which clock samples
count as "during the timed region"."""
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


def test_nvml_lines_decode_reason_bits():
    """Samples from the NVML child: wall time, SM clock, max, power, reason
    bits (sw_power_cap 0x4, hw_slowdown 0x8, sw_thermal 0x20, hw_thermal
    0x40, from nvml.h); other bits (idle 0x1) are not reasons to report."""
    bench = load_bench()
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.source = "nvml every 2 ms"
    t0 = 1_800_000_000.0
    s.lines = [(t0 + 0.5, "%.6f,1800,2070,900.500,4\n" % (t0 + 0.002)),
               (t0 + 0.5, "%.6f,1700,2070,1200.000,5\n" % (t0 + 0.004)),
               (t0 + 0.5, "%.6f,1600,2070,1300.000,72\n" % (t0 + 0.006)),  # 0x48
               (t0 + 0.5, "%.6f,2070,2070,100.000,1\n" % (t0 + 1.0))]
    w = s.window(t0, t0 + 0.01)
    assert w["samples"] == 3 and w["samples_inside_region"] == 3
    assert w["sm_mhz"] == 1700 and w["power_w_max"] == 1300.0
    assert w["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert w["source"] == "nvml every 2 ms"
    w = s.window(t0 + 0.9, t0 + 1.1)
    assert w["reasons"] == []


def test_sampler_falls_back_when_nvml_cannot_start(monkeypatch):
    """A child that exits without a sample (no NVML, unknown device) leaves
    the sampler on nvidia-smi, or on nothing, never hanging."""
    bench = load_bench()
    s = bench.ClockSampler(0, "ffff:ff:1f.0")
    s.start()
    try:
        assert s.source in (None, "nvidia-smi every 50 ms")
    finally:
        s.stop()


def test_traffic_record_needs_the_same_device_code_and_plan(monkeypatch, tmp_path):
    """A committed ncu traffic figure is reported only for the device code
    and launch configuration it was captured on."""
    import json
    bench = load_bench()
    (tmp_path / "profiles").mkdir()
    rec = {"w": {"kernel_hash": "h1", "dram_bytes_per_launch": 123,
                 "plan": {"cta_group": 2, "tile_n": 256, "raster_group": 16}},
           "old": {"kernel_hash": "h1", "dram_bytes_per_launch": 7}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "h1")
    plan = {"cta_group": 2, "tile_n": 256, "raster_group": 16, "stages": 5}
    assert bench.ncu_traffic("w", plan) == 123
    assert bench.ncu_traffic("w", dict(plan, tile_n=128)) is None
    assert bench.ncu_traffic("w", dict(plan, raster_group=8)) is None
    assert bench.ncu_traffic("w", None) is None
    assert bench.ncu_traffic("old", plan) == 7  # a record without a plan: code only
    assert bench.ncu_traffic("missing", plan) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "h2")
    assert bench.ncu_traffic("w", plan) is None


def test_device_code_hash_ignores_host_only_sources():
    bench = load_bench()
    csrc = os.path.join(ROOT, "dense_gemm_elementwise_gb300", "csrc")
    assert set(bench.HOST_ONLY_SOURCES) <= set(os.listdir(csrc))
    assert len(bench.kernel_source_hash()) == 16


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
