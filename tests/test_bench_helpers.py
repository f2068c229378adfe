"""bench.py's measurement helpers on the CPU: the per-launch traffic model,
the lookup of ncu DRAM bytes by kernel-source hash, and the parsing of the
clock samples that decide whether a timed run is accepted."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_and_flops_follow_their_definitions():
    # one m-tile per woken expert at the V4 decode shape: packed rows once per
    # m-tile, each pair's activation row once, the fp32 accumulator read and
    # written once, the fp16 LUT once
    n, k, K, N, L, tiles = 32, 6, 4096, 2048, 16, 137
    want = tiles * N * K // 4 + n * k * K * 2 + n * N * 8 + 2 * (1 << L)
    assert bench.grouped_algorithmic_bytes(tiles, n, k, K, N, L) == want
    assert bench.grouped_flops(n, k, K, N) == 2 * n * k * K * N


def test_recorded_traffic_is_keyed_by_the_kernel_source_hash():
    src = os.path.join(ROOT, "trellis_quantized_moe_sort_gb300", "csrc", "tq_grouped.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    table = open(os.path.join(ROOT, "profiles", "grouped_kernel_traffic.txt")).read()
    for workload in ("v4_decode_n32", "v4_prefill_n8192_up", "v4_prefill_n8192_down"):
        got = bench.recorded_traffic(workload)
        if f"{h} {workload} " in table:
            assert isinstance(got, int) and got > 0
        else:
            assert got is None       # counters taken on another source: not reported
    assert bench.recorded_traffic("no_such_workload") is None


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


@pytest.mark.parametrize("lines,sm,reasons", [
    (["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active"] * 5, 2070.0, []),
    (["0, 1980, 2070, 1390.1, 0x4, Not Active, Not Active, Not Active, Active",
      "0, 2010, 2070, 1391.0, 0x4, Not Active, Not Active, Not Active, Active",
      "0, 1995, 2070, 1389.5, 0x4, Not Active, Not Active, Not Active, Not Active"], 1995.0, ["sw_power_cap"]),
    (["0, 1200, 2070, 500.0, 0x40, Not Active, Active, Not Active, Not Active"], 1200.0, ["hw_thermal_slowdown"]),
])
def test_clock_sampler_parses_median_and_throttle_reasons(tmp_path, monkeypatch, lines, sm, reasons):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    cs = bench.ClockSampler(0)
    f = open(tmp_path / "clocks.csv", "w+")
    f.write("\n".join(lines + ["garbage line", ""]))
    f.flush()
    cs.f, cs.proc = f, _FakeProc()
    out = cs.stop()
    assert out["sm_mhz"] == sm and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == reasons and out["samples"] == len(lines)


def test_clock_sampler_without_samples_reports_none(tmp_path, monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    cs = bench.ClockSampler(0)
    assert cs.stop() is None                 # never started (no nvidia-smi)
    f = open(tmp_path / "empty.csv", "w+")
    cs.f, cs.proc = f, _FakeProc()
    assert cs.stop() is None
