"""bench.py's host-side helpers on the CPU: roofline denominator and its
fallback, the ncu traffic record tied to the kernel source revision, the
clock-record summary, the split workload's CTA model, and the oracle timed
over spawned shards."""

import json

import bench


def test_peak_from_measured_file_or_fallback(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1234.5}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peak_hbm() == (1234.5, "measured")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.peak_hbm() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_traffic_record_only_for_the_profiled_kernel(tmp_path, monkeypatch):
    rec = {"kernel_sha": bench.kernel_sha(),
           "workloads": {"w": {"dram_bytes_per_launch": 157229312}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.ncu_traffic("w") == 157229312
    assert bench.ncu_traffic("other") is None
    rec["kernel_sha"] = "0" * 16          # the kernel changed since the capture
    path.write_text(json.dumps(rec))
    assert bench.ncu_traffic("w") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.ncu_traffic("w") is None


def test_clock_lines_summary():
    lines = [
        "0, 2070, 2070, 480.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 510.3, 0x0, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 505.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    c = bench.parse_clock_lines(lines)
    assert c["samples"] == 3 and c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["power_w_max"] == 510.3 and c["reasons"] == ["sw_power_cap"]
    hot = ["0, 1500, 2070, 900.0, 0x40, Not Active, Active, Not Active, Not Active"]
    assert bench.parse_clock_lines(hot)["reasons"] == ["hw_thermal_slowdown"]
    assert bench.parse_clock_lines([]) is None


def test_clock_sampler_keeps_only_the_timed_region():
    """Samples from before begin() (the warm-up) and after end() are dropped;
    take_now() gives a short region its own sample."""
    clocks = iter([1400.0, 1500.0, 2070.0, 2055.0, 900.0])

    class Fake:
        name = "fake"

        def sample(self):
            return {"sm": next(clocks, 900.0), "max": 2070.0, "power": 500.0,
                    "reasons": ["sw_power_cap"]}

        def close(self):
            pass

    s = bench.ClockSampler(Fake(), period_ms=10 ** 6)   # the thread never fires
    s.take_now()
    s.take_now()                                      # warm-up: 1400, 1500
    s.begin()
    s.take_now()
    s.take_now()                                      # region: 2070, 2055
    s.end()
    s.take_now()                                      # after: 900
    c = s.stop()
    assert c["samples"] == 2 and c["sm_mhz"] == 2062.5 and c["reasons"] == ["sw_power_cap"]
    assert c["source"] == "fake" and c["window"].startswith("timed region")
    assert "edges" not in c
    # edge samples right before and after the region are reported on their own
    e = bench.ClockSampler(Fake(), period_ms=10 ** 6)
    e.take_edge("before")                              # 900
    e.begin()
    e.take_now()                                       # region: 900
    e.end()
    e.take_edge("after")
    c = e.stop()
    assert c["samples"] == 1
    assert set(c["edges"]) == {"before", "after"}
    assert c["edges"]["before"] == {"sm_mhz": 900.0, "reasons": ["sw_power_cap"]}
    empty = bench.ClockSampler(Fake(), period_ms=10 ** 6)
    empty.begin()
    empty.end()
    assert empty.stop() is None


def test_nvml_source_reads_through_a_fake_library(monkeypatch):
    """NvmlSource against a fake libnvidia-ml: handle by UUID, SM clock and
    maximum in MHz, power in mW -> W, and the clock-event reason bits mapped
    to names (0x4 power cap, 0x8 hardware slowdown, 0x20 software thermal,
    0x40 hardware thermal); idle (0x1) is not a reason to report. Only read
    calls exist in the fake, so any attempt to set something would fail."""
    import ctypes
    calls = []

    def out(arg, value):
        arg._obj.value = value
        return 0

    class FakeNvml:
        def nvmlInit_v2(self):
            calls.append("init")
            return 0

        def nvmlShutdown(self):
            calls.append("shutdown")
            return 0

        def nvmlDeviceGetHandleByUUID(self, uuid, handle):
            calls.append(uuid)
            return out(handle, 1234) if uuid == b"GPU-abc" else 999

        def nvmlDeviceGetHandleByIndex_v2(self, index, handle):
            return out(handle, 99)

        def nvmlDeviceGetClockInfo(self, h, kind, v):
            return out(v, 1965 if kind == 1 else 0)

        def nvmlDeviceGetMaxClockInfo(self, h, kind, v):
            return out(v, 2070)

        def nvmlDeviceGetPowerUsage(self, h, v):
            return out(v, 612345)

        def nvmlDeviceGetCurrentClocksEventReasons(self, h, v):
            return out(v, 0x1 | 0x4 | 0x40)

    monkeypatch.setattr(ctypes, "CDLL", lambda name: FakeNvml())
    src = bench.NvmlSource("GPU-abc", 0)
    assert src.h.value == 1234
    s = src.sample()
    assert s == {"sm": 1965.0, "max": 2070.0, "power": 612.345,
                 "reasons": ["sw_power_cap", "hw_thermal_slowdown"]}
    src.close()
    assert calls == ["init", b"GPU-abc", "shutdown"]
    assert bench.NvmlSource("GPU-other", 3).h.value == 99   # falls back to the index


def test_cta_model_of_the_split_workload():
    # ceil(T/128) * (H/128) / 8: the configs' 64 / 128 / 256 / 512 CTAs
    assert [bench.ctas_unsplit(T, 8192) for T in (1024, 2048, 4096, 8192)] == [64, 128, 256, 512]
    assert bench.ctas_unsplit(4864, 8192) == 304


def test_oracle_over_spawned_shards_covers_the_rows():
    # PR1 (T=128): the budget covers every row, split into one contiguous
    # shard per host core (at most 128 non-empty shards)
    import os
    r = bench.cpu_baseline_procs("pr1_t128_h4096_n2", 0, t_row_s=1e-4, budget_s=5.0)
    assert r is not None
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0
    assert r["cores"] == min(len(os.sched_getaffinity(0)), 128)
    assert r["sample"].startswith("128 of 128 token rows")


def test_kernel_fingerprint_ignores_prose_only(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n")
    base = bench.kernel_sha(str(src))
    src.write_text("// header, reworded\n/* a block\n comment */\n__global__ void k(int* p) {\n"
                   "    p[0] = 1;\n}\n")
    assert bench.kernel_sha(str(src)) == base       # comments and layout only
    src.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 2;  // store\n}\n")
    assert bench.kernel_sha(str(src)) != base       # the code changed


def test_reference_arm_line_on_the_oracle():
    """The reference arm times the oracle only: its line carries impl,
    the GPU arm's metric and workload, a cpu_baseline with cores 1, a
    zero-copy e2e and no GPU launches; other ranks return nothing."""
    import argparse
    args = argparse.Namespace(workload="pr1_t128_h4096_n2", tokens=0, steps=3, warmup=3)
    line = bench.reference_arm(args, 0, 1)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == "pr1_t128_h4096_n2"
    assert 1 <= line["config"]["rows_per_step"] <= 128
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["gpu_launches"] == 0 and line["steps"] == 3
    assert bench.reference_arm(args, 1, 2) is None
