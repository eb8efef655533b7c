"""Host-side helpers of bench.py, on the CPU.

* The DRAM-traffic record is used only for the kernel source it was captured
  on: any change to that source turns the bench line's `traffic` into null.
* The clock record keeps only the nvidia-smi samples that fall inside the
  timed region and names every throttle reason that was active there.
* The roofline denominators fall back to the stated figures when the measured
  peaks are absent.
"""

import datetime
import os

import bench


def _write_traffic(path, sha, read, write):
    with open(path, "w") as f:
        f.write("kernel: attn_tc_kernel<128, bf16>\n")
        f.write(f"source_sha256: {sha}\n")
        f.write(f"dram_bytes_read: {read}\n")
        f.write(f"dram_bytes_write: {write}\n")
        f.write(f"dram_bytes_per_launch: {read + write}\n")


def test_traffic_record_is_used_only_for_its_own_kernel_source(tmp_path, monkeypatch):
    path = str(tmp_path / "traffic.txt")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", path)
    assert bench.read_traffic() is None                      # no record
    _write_traffic(path, bench.tc_source_sha(), 1000, 24)
    assert bench.read_traffic() == 1024.0
    _write_traffic(path, "0" * 64, 1000, 24)                 # captured on another source
    assert bench.read_traffic() is None


def test_source_hash_covers_every_kernel_source(tmp_path, monkeypatch):
    # a copy of the sources with one byte changed in any of them hashes differently
    base, root0 = bench.tc_source_sha(), bench.ROOT
    for i, rel in enumerate(bench.TC_SOURCES):
        root = tmp_path / f"copy{i}"
        for other in bench.TC_SOURCES:
            dst = root / other
            dst.parent.mkdir(parents=True, exist_ok=True)
            with open(os.path.join(root0, other), "rb") as f:
                data = f.read()
            dst.write_bytes(data + (b" " if other == rel else b""))
        monkeypatch.setattr(bench, "ROOT", str(root))
        assert bench.tc_source_sha() != base, rel
    monkeypatch.setattr(bench, "ROOT", root0)
    assert bench.tc_source_sha() == base


class _FakeSmi:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _row(t, sm, power, hw="Not Active", thermal="Not Active", cap="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, {sm}, 2070, {power}, 0x0, {hw}, {thermal}, Not Active, {cap}\n"


def _sampler(tmp_path, rows, window):
    s = bench.ClockSampler("0")
    s.out_path = str(tmp_path / "clocks.csv")
    with open(s.out_path, "w") as f:
        f.writelines(rows)
    s.fh = open(os.devnull, "w")
    s.proc = _FakeSmi()
    if window:
        s.mark(*window)
    return s


def test_clock_record_keeps_the_timed_region_only(tmp_path):
    t0 = 1_790_000_000.0
    rows = [_row(t0 - 1.0, 900, 120.0, cap="Active"),        # before the region
            _row(t0 + 0.1, 2070, 950.5),
            _row(t0 + 0.2, 2040, 1210.0, cap="Active"),
            _row(t0 + 0.3, 2010, 1390.0),
            _row(t0 + 2.0, 400, 80.0, hw="Active")]           # after it
    r = _sampler(tmp_path, rows, (t0, t0 + 1.0)).stop()
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2040.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["power_w_median"] == 1210.0 and r["power_w_max"] == 1390.0


def test_clock_record_names_a_slowdown_inside_the_region(tmp_path):
    t0 = 1_790_000_000.0
    rows = [_row(t0 + 0.1, 1500, 700.0, hw="Active"), _row(t0 + 0.2, 1400, 700.0, thermal="Active")]
    r = _sampler(tmp_path, rows, (t0, t0 + 1.0)).stop()
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_record_without_samples(tmp_path):
    t0 = 1_790_000_000.0
    r = _sampler(tmp_path, [_row(t0 - 5.0, 2070, 500.0)], (t0, t0 + 1.0)).stop()
    assert r["samples"] == 0 and r["sm_mhz"] is None
    s = bench.ClockSampler("0")                              # nvidia-smi never started
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.read_peaks()
    assert kind == "fallback" and peaks == bench.FALLBACK_PEAKS
