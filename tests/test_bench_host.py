"""Host helpers of bench.py on CPU: the DRAM-traffic figures are keyed by a hash
of each kernel's own source files (a figure taken before a kernel changed is
not reported), and the roofline peaks fall back to the stated defaults when no
measured peaks are present. The clock record of a timed region is parsed
from nvidia-smi's CSV, and a hardware or thermal slowdown, or a clock held
low with no reason, marks the region for one more measurement."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(kernel, sha, value, operands=None, workload="T16384_C10240"):
    op = f" operands={operands}" if operands else ""
    return (f"kernel={kernel} workload={workload}{op} dram_bytes_per_launch={value} "
            f"src_sha={sha}\n")


def test_traffic_lookup_is_keyed_by_kernel_sources(tmp_path, monkeypatch):
    sha = bench.kernel_sha("gemm_grads")
    path = tmp_path / "traffic.txt"
    path.write_text("# comment line\n"
                    + _line("gemm_grads", sha, 1000)
                    + _line("gemm_grads", sha, 500, operands="fp8_2")
                    + _line("gemm_softmax_grad", "0000000000000000", 700))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.load_traffic("gemm_grads", "T16384_C10240") == 1000.0
    assert bench.load_traffic("gemm_grads", "T16384_C10240", "bf16") == 1000.0
    assert bench.load_traffic("gemm_grads", "T16384_C10240", "fp8_2") == 500.0
    # no line for these operands or this workload
    assert bench.load_traffic("gemm_grads", "T16384_C10240", "fp8_1") is None
    assert bench.load_traffic("gemm_grads", "T32768_C14336") is None
    # a figure whose kernel sources changed since the capture
    assert bench.load_traffic("gemm_softmax_grad", "T16384_C10240") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.load_traffic("gemm_grads", "T16384_C10240") is None


def test_kernel_sha_follows_the_kernel_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    shutil.copytree(bench.CSRC, csrc, ignore=shutil.ignore_patterns("*.o", "*.so"))
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    grads, build = bench.kernel_sha("gemm_grads"), bench.kernel_sha("build_candidates")
    listed = bench.KERNEL_SOURCES["gemm_grads"]
    # a source the kernel does not use leaves its hash alone
    other = next(n for n in bench.KERNEL_SOURCES["build_candidates"] if n not in listed)
    with open(csrc / other, "a") as f:
        f.write("\n// edit\n")
    assert bench.kernel_sha("gemm_grads") == grads
    assert bench.kernel_sha("build_candidates") != build
    # one of its own sources changes it
    with open(csrc / listed[-1], "a") as f:
        f.write("\n// edit\n")
    assert bench.kernel_sha("gemm_grads") != grads
    # a kernel without a source list hashes the whole folder
    whole = bench.kernel_sha("gather_rows")
    (csrc / "extra.cuh").write_text("// new file\n")
    assert bench.kernel_sha("gather_rows") != whole


def test_peaks_fall_back_without_measured_figures(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback"
    assert (p["bf16_tflops"], p["bf16_tflops_sustained"], p["hbm_gbs"]) == (1900.0, 1700.0,
                                                                         6800.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        '{"bf16_tflops": 1950.7, "bf16_tflops_sustained": 1747.9, "hbm_gbs": 6776.6}')
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["bf16_tflops"] == 1950.7 and p["hbm_gbs"] == 6776.6


class _FakeSmi:
    """Stands in for the nvidia-smi process the sampler started."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampled(tmp_path, rows, uuid="GPU-aaaa"):
    s = bench.ClockSampler(uuid)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("".join(r + "\n" for r in rows))
    s.out = open(s.path, "a")
    s.proc = _FakeSmi()
    return s.stop()


def _row(uuid, sm, mx, power, reasons=()):
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    cols = ", ".join("Active" if n in reasons else "Not Active" for n in names)
    return f"0, {uuid}, {sm}, {mx}, {power}, 0x0000000000000000, {cols}"


def test_clock_record_parsing(tmp_path):
    rows = [_row("GPU-aaaa", 1785, 2070, 1200.5),
            _row("GPU-aaaa", 1500, 2070, 1390.0, ("sw_power_cap",)),
            _row("GPU-aaaa", 1900, 2070, 1100.0),
            _row("GPU-bbbb", 300, 2070, 90.0, ("hw_slowdown",)),  # another GPU: ignored
            "garbage line",
            _row("GPU-aaaa", "[N/A]", 2070, 1000.0)]  # no clock reading
    c = _sampled(tmp_path, rows)
    assert c["samples"] == 4
    assert c["sm_mhz"] == 1785.0           # median of 1785, 1500, 1900
    assert c["sm_max_mhz"] == 2070.0
    assert c["power_w_max"] == 1390.0
    assert c["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(str(tmp_path / "clocks.csv"))
    # no sample of this GPU at all
    c = _sampled(tmp_path, [_row("GPU-bbbb", 1800, 2070, 900.0)])
    assert c["samples"] == 0 and c["sm_mhz"] is None


def test_clock_check(tmp_path):
    ok = _sampled(tmp_path, [_row("GPU-aaaa", 2000, 2070, 900.0)])
    assert bench.clock_check(ok) == {"rejected": False, "why": []}
    # the power cap lowers the clock and is kept
    capped = _sampled(tmp_path, [_row("GPU-aaaa", 1400, 2070, 1400.0, ("sw_power_cap",))])
    assert bench.clock_check(capped) == {"rejected": False, "why": []}
    for reason in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        c = _sampled(tmp_path, [_row("GPU-aaaa", 1900, 2070, 900.0, (reason, "sw_power_cap"))])
        assert bench.clock_check(c) == {"rejected": True, "why": [reason]}
    # held well below the maximum with no reason: a leftover clock lock
    low = _sampled(tmp_path, [_row("GPU-aaaa", 1200, 2070, 600.0)])
    assert bench.clock_check(low) == {"rejected": True, "why": ["pinned_low"]}
    # no clock record: nothing to reject on
    assert bench.clock_check({"samples": 0, "sm_mhz": None, "sm_max_mhz": None,
                                "reasons": ["no nvidia-smi"]})["rejected"] is False
