#!/usr/bin/env python
"""Benchmark of the sampled-softmax CE hot path on GB300.

One step = one pass of the whole path over one synthetic batch: candidate
build, forward (loss + saved lse) and backward (dH, dW candidate rows), i.e.
ss_build_candidates + ss_forward + ss_backward through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 5]
                    [--impl native|reference] [--no-cpu-baseline]

Prints ONE JSON line on rank 0. `value` is tokens/s of the whole job with the
inputs resident in device memory (device-timed with CUDA events, L2 flushed by
a 256 MB write between steps, outside the timed events). `e2e` is the same
metric through the public Python API with the step's inputs (H, targets)
copied from pinned host memory and the per-token loss read back, every step;
`e2e_overlapped` the same with step k+1's copy on a second stream during step
k, as a pipelined training loop runs it. `roofline` is for the kernel with the largest share of the step, timed live
with CUDA events on its launch stream. `cpu_baseline` / `--impl reference`
time the CPU oracle (the plain definition, not tuned) on a bounded sample of
the same workload on this machine's host cores. `clocks` is the SM clock
record of the timed region; a region that saw a hardware or thermal slowdown,
or an SM clock held well below its maximum with no reason active, is taken
once more (the first attempt is kept under `clocks.first_attempt`).

Multi-GPU: the path does not shard across GPUs in this library (one GPU, no
collectives), so N > 1 runs N independent replicas, one per rank (weak
scaling), with a barrier around the timed region and the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sampled-softmax CE fwd+bwd tokens/s; % of GB300 bf16 tensor peak"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
# algorithmic flops per launch of each GEMM kernel, in units of T*C*D: the
# forward (2) and the two gradient GEMMs (4) make the 6*T*C*D of a step; the
# backward's recompute of the logits is work the definition does not ask for
# and counts 0 here (its executed flops are reported beside)
GEMM_FLOPS_TCD = {"gemm_forward_lse": 2, "gemm_softmax_grad": 0, "gemm_grads": 4}
GEMM_EXECUTED_TCD = {"gemm_forward_lse": 2, "gemm_softmax_grad": 2, "gemm_grads": 4}
CSRC = os.path.join(ROOT, "sampled_softmax_output_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for ~3 s of device time)")
    ap.add_argument("--warmup", type=int, default=5)
    # default: the full-vocabulary phase (T=65536, C=V=50304), the largest of
    # the five workloads, which the schedule runs for its final steps
    ap.add_argument("--workload", type=int, default=5, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the workload with this many tokens instead (same seed and "
                         "distributions; for small profiling captures)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU seconds of the oracle sample")
    ap.add_argument("--cap", type=float, default=0.0,
                    help="capped head: logits z = cap / (1 + exp(-s / tau)) (0: plain head)")
    ap.add_argument("--tau", type=float, default=7.5)
    ap.add_argument("--fp8", nargs="?", const="logits", default=None, choices=["logits", "all"],
                    help="the FP8 head: e4m3 operands for the two logit GEMMs ('logits', the "
                         "default), or also e5m2 G for the two gradient GEMMs ('all')")
    ap.add_argument("--targets", type=int, default=1,
                    help="targets per token (multi-token prediction over one set of logits): "
                         "offsets 1..K of one Zipf stream, weights 1, 1/2, 1/4, ...")
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="reference arm: target seconds per step (default: fits the run in ~2.5 min)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


# the source files that define each traced kernel
KERNEL_SOURCES = {
    "gemm_forward_lse": ["ss_internal.h", "ss_ptx.cuh", "ss_gemm.cuh", "ss_gemm2.cuh",
                         "ss_gemm_logits.cuh", "ss_gemm_logits.cu"],
    "gemm_softmax_grad": ["ss_internal.h", "ss_ptx.cuh", "ss_gemm.cuh", "ss_gemm2.cuh",
                          "ss_gemm_logits.cuh", "ss_gemm_logits.cu"],
    "gemm_grads": ["ss_internal.h", "ss_ptx.cuh", "ss_gemm.cuh", "ss_gemm2.cuh",
                   "ss_gemm_grads.cu"],
    "build_candidates": ["ss_internal.h", "ss_ptx.cuh", "ss_candidates.cu"],
}


def kernel_sha(kernel: str) -> str:
    """Hash of the sources of `kernel` (all of csrc/ for kernels not listed)."""
    names = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(CSRC))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, workload: str, operands: str = "bf16"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    if there is none or the kernel sources changed since it was captured.
    `operands`: bf16 (lines without the key), fp8_1 or fp8_2 (the FP8 head)."""
    try:
        with open(TRAFFIC_FILE) as f:
            lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    sha = kernel_sha(kernel)
    for ln in lines:
        parts = dict(kv.split("=", 1) for kv in ln.split())
        if (parts.get("kernel") == kernel and parts.get("workload") == workload
                and parts.get("operands", "bf16") == operands):
            if parts.get("src_sha") != sha:
                return None
            return float(parts["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    QUERY = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 10:  # wait for the first sample
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"samples": 0, "sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 10:
                    continue
                if self.uuid and self.uuid not in c[1]:
                    continue
                rows.append(c)
        os.unlink(self.path)
        if not rows:
            return {"samples": 0, "sm_mhz": None, "sm_max_mhz": None, "reasons": []}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        pw = [num(r[4]) for r in rows if num(r[4]) is not None]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7),
                              ("sw_thermal_slowdown", 8), ("sw_power_cap", 9)):
                if r[col].lower().startswith("active"):
                    reasons.add(name)
        return {"samples": len(rows), "sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons)}


# Throttle reasons that void a timed region. sw_power_cap is the part's usual
# state under a long dense GEMM: it is kept, and listed in `reasons`.
REJECTING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")
# an SM clock median below this fraction of the maximum, with no reason
# active, is taken for a clock lock left by another program
PINNED_LOW_FRAC = 0.8


def clock_check(clocks: dict) -> dict:
    """Whether the clock record of a timed region voids its number, and why:
    a hardware or thermal slowdown, or the SM clock held well below its
    maximum with no reason active ("pinned_low")."""
    reasons = [r for r in clocks.get("reasons", []) if r != "no nvidia-smi"]
    why = [r for r in reasons if r in REJECTING_REASONS]
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm is not None and mx and not reasons and sm < PINNED_LOW_FRAC * mx:
        why.append("pinned_low")
    return {"rejected": bool(why), "why": why}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "native" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def any_rank_rejected(check: dict, world: int, device=None) -> bool:
    """True on every rank if the clock check of any rank rejected its timed
    region, so that all ranks take the region again together."""
    return max_over_ranks(float(check["rejected"]), world, device) > 0


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------- CPU oracle

def fp8_mode(arg) -> int:
    return {None: 0, "logits": 1, "all": 2}[arg]


OPERANDS = {0: "bf16",
            1: "e4m3 (FP8 head) for the logit GEMMs, bf16 for the gradient GEMMs",
            2: "e4m3 (FP8 head) for the logit GEMMs, e5m2 G x e4m3 for the gradient GEMMs"}


def oracle_sample(x: dict, w, T_s: int, scale: float, cap: float = 0.0, tau: float = 1.0,
                  fp8: int = 0):
    """One oracle pass over a bounded sample: the full-batch candidate build
    (and, for the FP8 head, the rounding of H and W[cand]), then forward +
    backward for the first T_s tokens against that candidate set (with the
    same head as the native arm). Returns seconds."""
    import oracle
    t0 = time.perf_counter()
    cand, slot, U = oracle.build_candidates(x["targets"], w.V, w.C, w.seed)
    H, W = x["H"], x["W"]
    if fp8:
        H, W, _, _ = oracle.fp8_inputs(H, W, cand)
    Hs = H[:T_s]
    ss_ = slot[:T_s]
    loss, lse = oracle.forward(Hs, W, cand, ss_, cap=cap, tau=tau)
    if fp8 == 2:  # FP8 gradients: e5m2 G
        oracle.backward_dH_g8(Hs, W, cand, ss_, lse, scale, cap=cap, tau=tau)
        oracle.backward_dWc_g8(Hs, W, cand, ss_, lse, scale, cap=cap, tau=tau)
    else:
        oracle.backward_dH(Hs, W, cand, ss_, lse, scale, cap=cap, tau=tau)
        oracle.backward_dWc(Hs, W, cand, ss_, lse, scale, cap=cap, tau=tau)
    return time.perf_counter() - t0


def cpu_baseline(x: dict, w, target_s: float, cap: float = 0.0, tau: float = 1.0,
                 fp8: int = 0) -> dict:
    import oracle
    oracle.build()
    scale = 1.0 / w.T
    t_small = oracle_sample(x, w, 16, scale, cap, tau, fp8)
    T_s = int(max(16, min(w.T, 16 * target_s / max(t_small, 1e-3))))
    dt = oracle_sample(x, w, T_s, scale, cap, tau, fp8)
    return {"value": T_s / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"{w.name}: full-batch candidate build (T={w.T}) + forward/backward of the "
                       f"first {T_s} tokens against all C={w.C} candidates; {dt:.1f} s"),
            "seconds": dt, "tokens": T_s}


# ------------------------------------------------------------ native arm

def run_native(args, world, rank, local):
    import torch

    import sampled_softmax_output_gb300 as ss

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    if args.tokens is not None:
        import dataclasses
        w = dataclasses.replace(w, T=args.tokens, name=f"{w.name}_T{args.tokens}")
    T, V, C, D = w.T, w.V, w.C, w.D
    x = synth.workload_inputs(w)
    H = torch.from_numpy(x["H"].view(np.int16)).to(dev).view(torch.bfloat16)
    W = torch.from_numpy(x["W"].view(np.int16)).to(dev).view(torch.bfloat16)
    targets = torch.from_numpy(x["targets"]).to(dev)
    ws = ss.workspace(T, V, C, D, device=dev)
    cand = torch.empty(C, dtype=torch.int32, device=dev)
    slot = torch.empty(T, dtype=torch.int32, device=dev)
    loss = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    dH = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    dW = torch.zeros(V, D, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scale = 1.0 / T

    cap, tau, fp8 = args.cap, args.tau, fp8_mode(args.fp8)
    n_tg = args.targets
    mtp_weights = [0.5 ** k for k in range(n_tg)]
    if n_tg > 1:
        extra = synth.zipf_targets(np.random.default_rng(w.seed + 77), n_tg - 1, V, w.zipf_s)
        stream = np.concatenate([x["targets"], extra])
        targets_k = torch.from_numpy(
            np.stack([stream[k:k + T] for k in range(n_tg)]).astype(np.int32)).to(dev)

    def step(h=H, tg=targets):
        if n_tg > 1:
            ss.step_mtp(h, W, targets_k, mtp_weights, C, w.seed, ws, scale=scale, dW=dW, cap=cap,
                        tau=tau)
            return
        ss.step(h, W, tg, C, w.seed, ws, scale=scale, dW=dW, cand=cand, slot=slot, loss=loss,
                lse=lse, dH=dH, cap=cap, tau=tau, fp8=fp8)

    def step_three_calls(h=H, tg=targets):
        ss.build_candidates(tg, V, C, w.seed, ws, cand=cand, slot=slot)
        ss.forward(h, W, cand, slot, ws, loss=loss, lse=lse, cap=cap, tau=tau, fp8=fp8)
        ss.backward(h, W, cand, slot, lse, ws, scale=scale, dH=dH, dW=dW, cap=cap, tau=tau,
                    fp8=fp8)

    for _ in range(max(args.warmup, 1)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st, _ = ss.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    # size the timed region: ~3 s of device time unless --steps is given
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    step()
    e1.record()
    torch.cuda.synchronize()
    est_ms = e0.elapsed_time(e1)
    K = args.steps if args.steps is not None else int(min(3000, max(20, 3000.0 / max(est_ms, 1e-3))))

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass

    def timed_region():
        """K steps, events around each step only (the per-kernel trace below
        would add event records between the kernels), with the clocks sampled
        throughout."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        sampler = ClockSampler(uuid)
        barrier(world)
        torch.cuda.synchronize()
        sampler.start()
        for k in range(K):
            flush.zero_()
            starts[k].record()
            step()
            ends[k].record()
        torch.cuda.synchronize()
        clk = sampler.stop()
        barrier(world)
        clk["check"] = clock_check(clk)
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends)), clk

    total_ms, clocks = timed_region()
    # a slowdown or a held-down clock on any rank voids the number: every rank
    # takes the region once more (the decision is the same on all of them)
    if any_rank_rejected(clocks["check"], world, dev):
        first = {"ms_per_step": total_ms / K, "sm_mhz": clocks.get("sm_mhz"),
                 "reasons": clocks.get("reasons"), "why": clocks["check"]["why"]}
        total_ms, clocks = timed_region()
        clocks["first_attempt"] = first
    total_ms_max = max_over_ranks(total_ms, world, dev)
    st, _ = ss.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")

    # traced region: the same steps with a CUDA event pair around every kernel
    # launch of the library, on its launch stream
    Kt = min(K, 300)
    t_starts = [torch.cuda.Event(enable_timing=True) for _ in range(Kt)]
    t_ends = [torch.cuda.Event(enable_timing=True) for _ in range(Kt)]
    trace = ss.KernelTrace(capacity=16 * Kt)
    torch.cuda.synchronize()
    with trace:
        for k in range(Kt):
            flush.zero_()
            t_starts[k].record()
            step()
            t_ends[k].record()
    torch.cuda.synchronize()
    traced_ms_per_step = sum(s.elapsed_time(e) for s, e in zip(t_starts, t_ends)) / Kt

    # the same steps as three ABI calls (ss_build_candidates, ss_forward,
    # ss_backward), untraced, for comparison
    K3 = min(K, 300) if n_tg == 1 else 0
    s3 = [torch.cuda.Event(enable_timing=True) for _ in range(K3)]
    e3 = [torch.cuda.Event(enable_timing=True) for _ in range(K3)]
    torch.cuda.synchronize()
    for k in range(K3):
        flush.zero_()
        s3[k].record()
        step_three_calls()
        e3[k].record()
    torch.cuda.synchronize()
    three_calls_ms = sum(a.elapsed_time(b) for a, b in zip(s3, e3)) / K3 if K3 else None

    # the same step replayed from a CUDA graph of ss_step (ss_step_graph_*),
    # alternating with direct ss_step calls (graph first on even k, direct
    # first on odd k): under the power cap the clock drifts from region to
    # region, and the two are compared within one region
    graph_ms = beside_graph_ms = None
    if n_tg == 1:
        graph = ss.StepGraph(H, W, targets, C, ws, scale=scale, cand=cand, slot=slot, loss=loss,
                             lse=lse, dH=dH, dW=dW, cap=cap, tau=tau, fp8=fp8)
        graph.launch(w.seed)
        timed = {"graph": [], "direct": []}
        torch.cuda.synchronize()
        for k in range(K3):
            pair = (("graph", lambda: graph.launch(w.seed)), ("direct", step))
            for name, fn in (pair if k % 2 == 0 else pair[::-1]):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                flush.zero_()
                a.record()
                fn()
                b.record()
                timed[name].append((a, b))
        torch.cuda.synchronize()
        graph_ms = sum(a.elapsed_time(b) for a, b in timed["graph"]) / K3
        beside_graph_ms = sum(a.elapsed_time(b) for a, b in timed["direct"]) / K3
        graph.close()
        st, _ = ss.read_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st} after the graph region")

    # per-kernel times from the trace
    per = {}
    for name, ms in trace.timings():
        per.setdefault(name, []).append(ms)
    # kernels the library launched per step (a traced stage may hold several)
    launches_per_step = sum(trace.kernels) / Kt
    launches = int(round(launches_per_step * K))
    kern = {n: {"launches": len(v), "avg_ms": sum(v) / len(v), "total_ms": sum(v)}
            for n, v in per.items()}
    traced_total = sum(k["total_ms"] for k in kern.values())
    for k in kern.values():
        k["share"] = k["total_ms"] / traced_total if traced_total > 0 else None
    dom = max(kern, key=lambda n: kern[n]["total_ms"])
    peaks = load_peaks()
    if dom in GEMM_FLOPS_TCD:
        flops = float(GEMM_FLOPS_TCD[dom]) * T * C * D
        achieved = flops / (kern[dom]["avg_ms"] * 1e-3) / 1e12
        # a kernel on 8-bit operands takes the measured bf16 peak times the
        # nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s dense)
        f8 = (fp8 >= 1 and dom in ("gemm_forward_lse", "gemm_softmax_grad")) or \
             (fp8 == 2 and dom == "gemm_grads")
        ratio = 2.0 if f8 else 1.0
        peak = peaks["bf16_tflops"] * ratio
        src = (f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"
               if peaks["source"] == "measured" else "fallback")
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": load_traffic(dom, w.name, f"fp8_{fp8}" if fp8 else "bf16"),
                "peak_source": src + (" x 2, the nominal e4m3 / bf16 ratio" if f8 else ""),
                "frac_of_sustained": achieved / (peaks["bf16_tflops_sustained"] * ratio),
                "algorithmic_flops_per_launch": flops,
                "executed_flops_per_launch": float(GEMM_EXECUTED_TCD[dom]) * T * C * D}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": None, "traffic": None}

    tokens_per_s = world * T * K / (total_ms_max * 1e-3)
    ms_per_step = total_ms_max / K
    step_tflops = 6.0 * T * C * D / (ms_per_step * 1e-3) / 1e12
    # flops the kernels of one step execute (the traced GEMM launches per
    # step). With the plain head, ss_step's softmax-gradient GEMM is the
    # fallback of the stored-probability backward: a launch that finds its
    # gate shut returns at once, and executes nothing; such launches take a
    # few microseconds where the GEMM takes about as long as the forward.
    def executes(n):
        if n != "gemm_softmax_grad" or "gemm_forward_lse" not in kern:
            return True
        return kern[n]["avg_ms"] > 0.25 * kern["gemm_forward_lse"]["avg_ms"]
    executed_flops_step = sum(float(GEMM_EXECUTED_TCD[n]) * T * C * D * kern[n]["launches"] / Kt
                              for n in kern if n in GEMM_EXECUTED_TCD and executes(n))

    # end to end through the public API: H2D of H and targets from pinned
    # memory, the three calls, D2H of the per-token loss, every step
    H_pin = torch.from_numpy(x["H"].view(np.int16)).pin_memory()
    tg_pin = torch.from_numpy(x["targets"]).pin_memory()
    loss_pin = torch.empty(T, dtype=torch.float32).pin_memory()
    H_dev = torch.empty(T, D, dtype=torch.int16, device=dev)
    tg_dev = torch.empty(T, dtype=torch.int32, device=dev)
    Ke = max(3, min(K, 50))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    barrier(world)
    for k in range(Ke):
        flush.zero_()
        es[k].record()
        H_dev.copy_(H_pin, non_blocking=True)
        tg_dev.copy_(tg_pin, non_blocking=True)
        step(H_dev.view(torch.bfloat16), tg_dev)
        loss_pin.copy_(loss, non_blocking=True)
        ee[k].record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(es, ee)), world, dev)
    e2e = {"value": world * T * Ke / (e2e_ms * 1e-3), "unit": UNIT,
           "h2d_bytes_per_step": int(H_pin.numel() * 2 + tg_pin.numel() * 4),
           "d2h_bytes_per_step": int(loss_pin.numel() * 4), "steps": Ke}

    # the same, pipelined as a training loop would run it: step k + 1's inputs
    # are copied on a second stream while step k computes (two input buffers).
    # Every copy still happens inside a timed span: step 0's in its own, step
    # k + 1's in step k's.
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    Hb = [H_dev, torch.empty_like(H_dev)]
    tb = [tg_dev, torch.empty_like(tg_dev)]
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    es2 = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    ee2 = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]

    def h2d(i, after):
        copy.wait_event(after)
        with torch.cuda.stream(copy):
            Hb[i].copy_(H_pin, non_blocking=True)
            tb[i].copy_(tg_pin, non_blocking=True)
            ready[i].record(copy)

    barrier(world)
    for k in range(Ke):
        flush.zero_()
        es2[k].record(comp)
        cur, nxt = k % 2, (k + 1) % 2
        if k == 0:
            h2d(cur, es2[k])
        if k + 1 < Ke:  # buffer nxt was last read by step k - 1
            h2d(nxt, done[nxt] if k >= 1 else es2[k])
        comp.wait_event(ready[cur])
        step(Hb[cur].view(torch.bfloat16), tb[cur])
        loss_pin.copy_(loss, non_blocking=True)
        done[cur].record(comp)
        ee2[k].record(comp)
    torch.cuda.synchronize()
    e2o_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(es2, ee2)), world, dev)
    e2e_overlapped = {"value": world * T * Ke / (e2o_ms * 1e-3), "unit": UNIT,
                      "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                      "d2h_bytes_per_step": e2e["d2h_bytes_per_step"], "steps": Ke,
                      "note": "step k+1's host-to-device copy runs on a second stream during "
                              "step k (double-buffered inputs)"}

    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "T": T, "V": V, "C": C, "D": D, "zipf_s": w.zipf_s,
                   "seed": w.seed, "parallelism": f"replicas x{world}" if world > 1 else "single",
                   "l2": "flushed between steps (256 MB write, outside the timed events)",
                   "step": "ss_step (= ss_build_candidates + ss_forward + ss_backward in one call)",
                   "head": ({"cap": cap, "tau": tau, "logits": "cap / (1 + exp(-s / tau))"}
                            if cap else "plain"),
                   "targets_per_token": n_tg,
                   "operands": OPERANDS[fp8],
                   **({"target_weights": mtp_weights} if n_tg > 1 else {}),
                   "ms_per_step_three_calls": three_calls_ms,
                   "ms_per_step_graph": graph_ms,
                   "ms_per_step_beside_graph": beside_graph_ms,
                   "step_tflops_algorithmic_6TCD": step_tflops,
                   "pct_bf16_peak_algorithmic": 100.0 * step_tflops / peaks["bf16_tflops"],
                   "step_flops_executed": executed_flops_step,
                   "pct_bf16_peak_executed": 100.0 * executed_flops_step / (ms_per_step * 1e-3)
                                             / 1e12 / peaks["bf16_tflops"],
                   "sm_mhz_median": clocks.get("sm_mhz"),
                   "ms_per_step_x_sm_mhz": (ms_per_step * clocks["sm_mhz"]
                                            if clocks.get("sm_mhz") else None)},
        "roofline": roof,
        "kernels": kern,
        "kernels_note": (f"per-kernel CUDA-event times from a second timed region of {Kt} steps "
                         f"with an event pair around every launch ({traced_ms_per_step:.4f} "
                         "ms/step there)"),
        "gpu_launches": launches,
        "e2e": e2e,
        "e2e_overlapped": e2e_overlapped,
        "clocks": clocks,
    }
    return line, x, w


def run_reference(args, world, rank):
    """The CPU oracle as it stands on this machine's host cores, rank 0 only."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    if args.tokens is not None:
        import dataclasses
        w = dataclasses.replace(w, T=args.tokens, name=f"{w.name}_T{args.tokens}")
    x = synth.workload_inputs(w)
    K = args.steps if args.steps is not None else 3
    W_ = max(args.warmup, 0)
    per_step_s = (args.ref_step_seconds if args.ref_step_seconds is not None
                  else min(5.0, 150.0 / max(K + W_, 1)))
    scale = 1.0 / w.T
    t_small = oracle_sample(x, w, 8, scale, args.cap, args.tau, fp8_mode(args.fp8))
    T_s = int(max(1, min(w.T, 8 * per_step_s / max(t_small, 1e-3))))
    for _ in range(W_):
        oracle_sample(x, w, T_s, scale, args.cap, args.tau, fp8_mode(args.fp8))
    dt = 0.0
    for _ in range(K):
        dt += oracle_sample(x, w, T_s, scale, args.cap, args.tau, fp8_mode(args.fp8))
    value = T_s * K / dt
    cores = oracle.num_threads()
    sample = (f"{w.name}: per step, full-batch candidate build (T={w.T}) + forward/backward of "
              f"the first {T_s} tokens against all C={w.C} candidates")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W_, "ms_per_step": 1e3 * dt / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "V": w.V, "C": w.C, "D": w.D,
                       "sample_tokens_per_step": T_s},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line, x, w = run_native(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(x, w, args.cpu_seconds, args.cap, args.tau,
                                                fp8_mode(args.fp8))
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
