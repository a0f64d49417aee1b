"""Host helpers of bench.py on CPU: the DRAM-traffic figures are keyed by a hash
of each kernel's own source files (a figure taken before a kernel changed is
not reported), and the roofline peaks fall back to the stated defaults when no
measured peaks are present."""
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
