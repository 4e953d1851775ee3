"""Host-side logic of the benchmark, without a GPU: the clock sampler's
summary (which decides whether a run is rejected for throttling), the DRAM
traffic lookup keyed by kernel sources, the peak lookup and the defaults of
the command line."""
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _row(sm, smax, hw="Not Active", hwt="Not Active", swt="Not Active", pcap="Not Active"):
    return ["2026/01/01 00:00:00.000", "0", str(sm), str(smax), "900.0", "0x0", hw, hwt, swt, pcap]


def test_clock_summary_median_max_and_reasons():
    c = bench.Clocks(0)
    c.rows = [(10.0, _row(2070, 2070)), (10.1, _row(1980, 2070, pcap="Active")),
              (10.2, _row(2070, 2070)), (99.0, _row(300, 2070, hw="Active"))]
    s = c.summary(9.0, 11.0)  # the sample outside the timed region is ignored
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_every_throttle_reason():
    c = bench.Clocks(0)
    c.rows = [(1.0, _row(1400, 2070, hw="Active")), (1.1, _row(1400, 2070, hwt="Active")),
              (1.2, _row(1400, 2070, swt="Active"))]
    s = c.summary(0.0, 2.0)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1400.0


def test_clock_summary_without_samples():
    c = bench.Clocks(0)
    c.rows = [(1.0, ["garbage"])]
    s = c.summary(0.0, 2.0)
    assert s == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_lookup_follows_the_kernel_sources(monkeypatch, tmp_path):
    from q8_quantized_gemv_gb300 import build
    key = "gemv_ring_gateup_24576x4096_int8act_b1"
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\n"
                 f"{key}: 109848576 ring={build.sources_digest('ring')}\n"
                 f"other_key: 5 mma={build.sources_digest('mma')}\n")
    got = bench.profile_traffic(key, "ring", str(f))
    assert got == 109848576.0
    assert bench.profile_traffic("no_such_capture", "ring", str(f)) is None
    assert bench.profile_traffic(key, "mma", str(f)) is None  # another family's key
    monkeypatch.setattr(build, "sources_digest", lambda kind=None: "0" * 64)
    assert bench.profile_traffic(key, "ring", str(f)) is None  # sources changed since the capture


def test_committed_traffic_file_parses():
    """profiles/traffic.txt: every line a key, a byte count and a family digest."""
    import os
    with open(os.path.join(bench.ROOT, "profiles", "traffic.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split(":", 1)
            val, tag = v.split()
            fam, sha = tag.split("=")
            assert float(val) > 0 and fam in ("ring", "mma", "chain") and len(sha) == 64


def test_peaks_and_defaults():
    peaks, src = bench.measured_peaks()
    assert peaks["hbm_gbs"] > 1000.0 and src in ("measured", "fallback")
    sys_argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        a = bench.parse()
    finally:
        sys.argv = sys_argv
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1
    assert a.impl != "reference" and a.batch == 1 and a.mode == "int8act"


def test_replica_value():
    assert bench.replica_value(8_041_103_360, 1, 2.0) == pytest.approx(8_041_103_360 / 2e-3 / 1e9)
    assert bench.replica_value(1e9, 4, 1.0) == pytest.approx(4000.0)


def test_host_info():
    h = bench.host_info()
    assert isinstance(h["nproc"], int) and h["nproc"] >= 1 and h["machine"]


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the CPU oracle, no GPU needed) prints one
    JSON line with the contract's keys."""
    import json
    import subprocess
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    import os
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
