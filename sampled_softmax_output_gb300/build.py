"""Compile the CUDA library libss.so in-tree for sm_103a.

    python -m sampled_softmax_output_gb300.build [--force] [--verbose]

Each translation unit under csrc/ is compiled in parallel with nvcc, then the
objects are linked into ``sampled_softmax_output_gb300/_build/libss.so``. The
CUDA runtime is linked statically, so the library needs only the driver at run
time (the driver API entry point for TMA descriptors is fetched through the
runtime, not linked).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libss.so")
SOURCES = ["ss_api.cu", "ss_candidates.cu", "ss_gemm_logits.cu", "ss_gemm_logits_mtp.cu",
           "ss_gemm_grads.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def _flags(verbose: bool) -> list[str]:
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                "--expt-relaxed-constexpr"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _deps() -> list[str]:
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(ROOT, "include", "ss.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    return _build_into(OUT_DIR, LIB, [], verbose)


def build_variant(out_dir: str, defines: list[str], verbose: bool = False) -> str:
    """Build a copy of the library with extra preprocessor definitions (e.g.
    ``SS_TIE_CAP=0``) into ``out_dir``; returns the path of its libss.so."""
    return _build_into(out_dir, os.path.join(out_dir, "libss.so"), ["-D" + d for d in defines],
                       verbose)


def _build_into(out_dir: str, lib: str, extra: list[str], verbose: bool) -> str:
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = _flags(verbose) + extra

    def compile_one(src: str):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    errors = []
    for src, _, r in results:
        if verbose and (r.stdout or r.stderr):
            print(f"--- {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            errors.append(f"{src}:\n{r.stdout}{r.stderr}")
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for _, o, _ in results] + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
