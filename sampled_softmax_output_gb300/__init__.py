"""GB300 sampled-softmax cross-entropy: Python binding of libss (include/ss.h).

Sampled softmax scores only a candidate subset of the vocabulary rows, shared
by the whole batch, in the forward and the backward pass of the lm_head
("KellerJordan/modded-nanogpt" README, technique list; "NanoGPT Training
Record: Technical Optimizations & Speed", section "Key Optimizations and
Ablation Table Results").

This module is argument marshalling only: every step of the computation runs in
the CUDA kernels of ``_build/libss.so``. PyTorch provides device memory and the
current CUDA stream. If the library has not been built, importing the binding
raises -- there is no fallback.

    import sampled_softmax_output_gb300 as ss
    ws = ss.workspace(T, V, C, D)                       # device bytes, reusable
    cand, slot, U = ss.build_candidates(targets, V, C, seed, ws, return_U=True)
    loss, lse = ss.forward(H, W, cand, slot, ws)        # per-token loss, saved lse
    dH, dW = ss.backward(H, W, cand, slot, lse, ws, scale=1.0 / T, dW=dW)
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libss.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "ss.h")

STATUS = {
    0: "SS_OK", 1: "SS_ERR_INVALID", 2: "SS_ERR_UNSUPPORTED", 3: "SS_ERR_CAPACITY",
    4: "SS_ERR_TARGET_RANGE", 5: "SS_ERR_WORKSPACE", 6: "SS_ERR_CUDA", 7: "SS_ERR_TIMEOUT",
    8: "SS_ERR_INDEX",
}
MAX_V = 524288
MAX_D = 16384
NOALLOC_SCRATCH_BYTES = 32 << 20


class Head(ctypes.Structure):
    """ss_head: cap > 0 -> logits z = cap / (1 + exp(-s / tau)); cap = 0 -> plain;
    fp8 = 1 -> the FP8 head (e4m3 logit GEMMs); fp8 = 2 -> FP8 through the
    backward too (e5m2 G in the gradient GEMMs)."""
    _fields_ = [("cap", ctypes.c_float), ("tau", ctypes.c_float), ("fp8", ctypes.c_int)]


def _head(cap: float, tau: float, fp8: int = 0):
    """``fp8``: 0 / False (bf16), 1 / True (FP8 logit GEMMs), 2 (FP8 logit and
    gradient GEMMs)."""
    if cap == 0 and not fp8:
        return None
    return ctypes.byref(Head(float(cap), float(tau), int(fp8)))


class SSError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        self.name = STATUS.get(self.code, str(code))
        msg = _lib.ss_status_string(self.code).decode() if _lib is not None else self.name
        if self.code == 6 and _lib is not None:
            msg += "; " + (_lib.ss_last_error() or b"").decode()
        super().__init__(f"{where}: {self.name} ({msg})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libss.so is not built ({LIB_PATH}); run `python -m sampled_softmax_output_gb300.build` "
            "(or __graft_entry__.build()). There is no non-CUDA fallback.")
    L = ctypes.CDLL(LIB_PATH)
    p, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    L.ss_workspace_size.restype = sz
    L.ss_workspace_size.argtypes = [i64, i64, i64, i64]
    L.ss_build_candidates.restype = ctypes.c_int
    L.ss_build_candidates.argtypes = [p, i64, i64, i64, ctypes.c_uint64, p, p, p, p, sz, p]
    L.ss_forward.restype = ctypes.c_int
    L.ss_forward.argtypes = [p, p, p, p, i64, i64, i64, i64, p, p, p, sz, p]
    L.ss_backward.restype = ctypes.c_int
    L.ss_backward.argtypes = [p, p, p, p, p, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                              p, p, p, sz, p]
    L.ss_read_status.restype = ctypes.c_int
    L.ss_read_status.argtypes = [p, sz, p, p, p]
    L.ss_status_string.restype = ctypes.c_char_p
    L.ss_status_string.argtypes = [ctypes.c_int]
    L.ss_step.restype = ctypes.c_int
    L.ss_step.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_uint64, ctypes.c_float, ctypes.c_int,
                          p, p, p, p, p, p, p, sz, p]
    L.ss_forward_noalloc.restype = ctypes.c_int
    L.ss_forward_noalloc.argtypes = [p, p, p, p, i64, i64, i64, i64, p, p, p, p]
    L.ss_last_error.restype = ctypes.c_char_p
    L.ss_last_error.argtypes = []
    L.ss_trace_begin.restype = ctypes.c_int
    L.ss_trace_begin.argtypes = [p, ctypes.c_int]
    L.ss_trace_end.restype = ctypes.c_int
    L.ss_trace_end.argtypes = []
    L.ss_trace_kernel_name.restype = ctypes.c_char_p
    L.ss_trace_kernel_name.argtypes = [ctypes.c_int]
    L.ss_trace_kernel_launches.restype = ctypes.c_int
    L.ss_trace_kernel_launches.argtypes = [ctypes.c_int]
    hp = ctypes.POINTER(Head)
    L.ss_forward_head.restype = ctypes.c_int
    L.ss_forward_head.argtypes = [p, p, p, p, i64, i64, i64, i64, hp, p, p, p, sz, p]
    L.ss_backward_head.restype = ctypes.c_int
    L.ss_backward_head.argtypes = [p, p, p, p, p, i64, i64, i64, i64, hp, ctypes.c_float,
                                   ctypes.c_int, p, p, p, sz, p]
    L.ss_step_head.restype = ctypes.c_int
    L.ss_step_head.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_uint64, hp, ctypes.c_float,
                               ctypes.c_int, p, p, p, p, p, p, p, sz, p]
    fp = ctypes.POINTER(ctypes.c_float)
    L.ss_forward_mtp.restype = ctypes.c_int
    L.ss_forward_mtp.argtypes = [p, p, p, p, i64, fp, i64, i64, i64, i64, hp, p, p, p, sz, p]
    L.ss_backward_mtp.restype = ctypes.c_int
    L.ss_backward_mtp.argtypes = [p, p, p, p, i64, fp, p, i64, i64, i64, i64, hp, ctypes.c_float,
                                  ctypes.c_int, p, p, p, sz, p]
    L.ss_step_mtp.restype = ctypes.c_int
    L.ss_step_mtp.argtypes = [p, i64, fp, p, p, i64, i64, i64, i64, ctypes.c_uint64, hp,
                              ctypes.c_float, ctypes.c_int, p, p, p, p, p, p, p, sz, p]
    L.ss_quantize_e4m3.restype = ctypes.c_int
    L.ss_quantize_e4m3.argtypes = [p, i64, p, p, p, sz, p]
    L.ss_schedule_candidates.restype = i64
    L.ss_schedule_candidates.argtypes = [i64, i64, i64]
    L.ss_clear_rows.restype = ctypes.c_int
    L.ss_clear_rows.argtypes = [p, i64, i64, i64, p, p, sz, p]
    L.ss_step_graph_create.restype = ctypes.c_int
    L.ss_step_graph_create.argtypes = [p, p, p, i64, i64, i64, i64, hp, ctypes.c_float,
                                       ctypes.c_int, p, p, p, p, p, p, p, sz, ctypes.POINTER(p)]
    L.ss_step_graph_create_mtp.restype = ctypes.c_int
    L.ss_step_graph_create_mtp.argtypes = [p, i64, fp, p, p, i64, i64, i64, i64, hp,
                                           ctypes.c_float, ctypes.c_int, p, p, p, p, p, p, p, sz,
                                           ctypes.POINTER(p)]
    L.ss_step_graph_launch.restype = ctypes.c_int
    L.ss_step_graph_launch.argtypes = [p, ctypes.c_uint64, p]
    L.ss_step_graph_destroy.restype = None
    L.ss_step_graph_destroy.argtypes = [p]
    return L


_lib = None
_lib = _load()


def lib():
    return _lib


def header_symbols(path: str = HEADER) -> list[str]:
    """Names of the functions include/ss.h declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(ss_\w+)\s*\(", text, re.M)))


# ----------------------------------------------------------------- helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check(code: int, where: str):
    if code != 0:
        raise SSError(code, where)


def _bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> the same memory as int16 bit patterns (no copy)."""
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


# --------------------------------------------------------------- public API

def workspace_size(T: int, V: int, C: int, D: int) -> int:
    n = _lib.ss_workspace_size(T, V, C, D)
    if n == 0:
        raise SSError(1, "ss_workspace_size")
    return int(n)


WORKSPACE_HEADER_BYTES = 1024


def workspace(T: int, V: int, C: int, D: int, device=None) -> torch.Tensor:
    """A device byte buffer large enough for one batch of size (T, V, C, D),
    its header (status word) zeroed as include/ss.h requires of a new one."""
    ws = torch.empty(workspace_size(T, V, C, D), dtype=torch.uint8,
                     device=device if device is not None else "cuda")
    ws[:WORKSPACE_HEADER_BYTES].zero_()
    return ws


def build_candidates(targets: torch.Tensor, V: int, C: int, seed: int, ws: torch.Tensor,
                     cand: torch.Tensor | None = None, slot: torch.Tensor | None = None,
                     return_U: bool = False):
    """cand [C] int32 (sorted distinct targets, then seeded negatives by id),
    slot [T] int32 (cand[slot[t]] == targets[t]); U if return_U (synchronises)."""
    _need(targets, "targets", torch.int32)
    dev = targets.device
    T = targets.numel()
    _need(ws, "workspace", torch.uint8, dev)
    if cand is None:
        cand = torch.empty(C, dtype=torch.int32, device=dev)
    if slot is None:
        slot = torch.empty(T, dtype=torch.int32, device=dev)
    _need(cand, "cand", torch.int32, dev, (C,))
    _need(slot, "slot", torch.int32, dev, (T,))
    U = ctypes.c_int32(-1)
    code = _lib.ss_build_candidates(_ptr(targets), T, V, C, seed & (2**64 - 1), _ptr(cand),
                                    _ptr(slot), ctypes.byref(U) if return_U else None, _ptr(ws),
                                    ws.numel(), _stream(dev))
    _check(code, "ss_build_candidates")
    return (cand, slot, int(U.value)) if return_U else (cand, slot)


def forward(H: torch.Tensor, W: torch.Tensor, cand: torch.Tensor, slot: torch.Tensor,
            ws: torch.Tensor, loss: torch.Tensor | None = None, lse: torch.Tensor | None = None,
            cap: float = 0.0, tau: float = 1.0, fp8: int = 0):
    """Per-token loss [T] and log-sum-exp [T] (fp32) over the candidate rows
    (cap > 0: of the capped logits, ss_forward_head)."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    _need(W, "W", torch.bfloat16, dev)
    V = W.shape[0]
    C = cand.numel()
    _need(W, "W", torch.bfloat16, dev, (V, D))
    _need(cand, "cand", torch.int32, dev, (C,))
    _need(slot, "slot", torch.int32, dev, (T,))
    _need(ws, "workspace", torch.uint8, dev)
    if loss is None:
        loss = torch.empty(T, dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty(T, dtype=torch.float32, device=dev)
    _need(loss, "loss", torch.float32, dev, (T,))
    _need(lse, "lse", torch.float32, dev, (T,))
    if cap == 0 and not fp8:
        code = _lib.ss_forward(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), T, V, C, D, _ptr(loss),
                               _ptr(lse), _ptr(ws), ws.numel(), _stream(dev))
    else:
        code = _lib.ss_forward_head(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), T, V, C, D,
                                    _head(cap, tau, fp8), _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(dev))
    _check(code, "ss_forward")
    return loss, lse


def forward_noalloc(H: torch.Tensor, W: torch.Tensor, cand: torch.Tensor, slot: torch.Tensor,
                    loss: torch.Tensor, lse: torch.Tensor, check_status: bool = False):
    """ss_forward_noalloc: the forward pass with no workspace, for callers that
    cannot allocate device memory (the library's fixed scratch array is used
    instead; see include/ss.h). The caller passes the output tensors; this
    wrapper allocates nothing either. check_status=True synchronises and
    raises on a device-side error of this call."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    _need(W, "W", torch.bfloat16, dev)
    V = W.shape[0]
    C = cand.numel()
    _need(W, "W", torch.bfloat16, dev, (V, D))
    _need(cand, "cand", torch.int32, dev, (C,))
    _need(slot, "slot", torch.int32, dev, (T,))
    _need(loss, "loss", torch.float32, dev, (T,))
    _need(lse, "lse", torch.float32, dev, (T,))
    st = ctypes.c_int32(0)
    code = _lib.ss_forward_noalloc(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), T, V, C, D,
                                   _ptr(loss), _ptr(lse), ctypes.byref(st) if check_status else None,
                                   _stream(dev))
    _check(code, "ss_forward_noalloc")
    return loss, lse


def backward(H: torch.Tensor, W: torch.Tensor, cand: torch.Tensor, slot: torch.Tensor,
             lse: torch.Tensor, ws: torch.Tensor, scale: float = 1.0, accumulate: bool = False,
             dH: torch.Tensor | None = None, dW: torch.Tensor | None = None, cap: float = 0.0,
             tau: float = 1.0, fp8: int = 0):
    """dH [T, D] bf16 and dW [V, D] fp32 (only candidate rows written / added to).
    A new dW is zero-filled, so that it is the dense gradient."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    _need(W, "W", torch.bfloat16, dev)
    V = W.shape[0]
    C = cand.numel()
    _need(W, "W", torch.bfloat16, dev, (V, D))
    _need(cand, "cand", torch.int32, dev, (C,))
    _need(slot, "slot", torch.int32, dev, (T,))
    _need(lse, "lse", torch.float32, dev, (T,))
    _need(ws, "workspace", torch.uint8, dev)
    if dH is None:
        dH = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    if dW is None:
        dW = torch.zeros(V, D, dtype=torch.float32, device=dev)
    _need(dH, "dH", torch.bfloat16, dev, (T, D))
    _need(dW, "dW", torch.float32, dev, (V, D))
    if cap == 0 and not fp8:
        code = _lib.ss_backward(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), _ptr(lse), T, V, C, D,
                                float(scale), 1 if accumulate else 0, _ptr(dH), _ptr(dW),
                                _ptr(ws), ws.numel(), _stream(dev))
    else:
        code = _lib.ss_backward_head(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), _ptr(lse), T, V,
                                     C, D, _head(cap, tau, fp8), float(scale),
                                     1 if accumulate else 0,
                                     _ptr(dH), _ptr(dW), _ptr(ws), ws.numel(), _stream(dev))
    _check(code, "ss_backward")
    return dH, dW


def read_status(ws: torch.Tensor) -> tuple[int, int]:
    """(device status code, last U) after synchronising the current stream."""
    _need(ws, "workspace", torch.uint8)
    st = ctypes.c_int32(0)
    U = ctypes.c_int32(0)
    _lib.ss_read_status(_ptr(ws), ws.numel(), _stream(ws.device), ctypes.byref(st), ctypes.byref(U))
    return int(st.value), int(U.value)


class KernelTrace:
    """Per-stage CUDA-event timing of libss launches on this host thread (a
    stage is one kernel or the few kernels of one step of the path; .kernels
    gives the kernel launches of each recorded stage).

        with ss.KernelTrace(capacity=64) as tr:
            ...calls...
        torch.cuda.synchronize()
        for name, ms in tr.timings(): ...
    """

    def __init__(self, capacity: int = 256):
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        # torch creates the CUDA event at its first record: create them all now
        for e in self.events:
            e.record()
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * (2 * capacity))(
            *[ctypes.c_void_p(e.cuda_event) for e in self.events])
        self.count = 0

    def __enter__(self):
        _check(_lib.ss_trace_begin(ctypes.cast(self._handles, ctypes.c_void_p), self.capacity),
               "ss_trace_begin")
        return self

    def __exit__(self, *exc):
        self.count = int(_lib.ss_trace_end())
        if self.count < 0:
            raise RuntimeError("ss_trace: a CUDA event record failed")
        self.names = [(_lib.ss_trace_kernel_name(k) or b"?").decode()
                      for k in range(min(self.count, self.capacity))]
        self.kernels = [int(_lib.ss_trace_kernel_launches(k))
                        for k in range(min(self.count, self.capacity))]
        return False

    def timings(self) -> list[tuple[str, float]]:
        """(kernel name, milliseconds) per recorded launch; call after synchronising."""
        return [(self.names[k], self.events[2 * k].elapsed_time(self.events[2 * k + 1]))
                for k in range(min(self.count, self.capacity))]


def step(H, W, targets, C: int, seed: int, ws, scale: float = 1.0, dW=None, accumulate=False,
         cand=None, slot=None, loss=None, lse=None, dH=None, cap: float = 0.0, tau: float = 1.0,
         fp8: int = 0):
    """One full pass of the path in one call (ss_step): candidates, forward,
    backward, with one gather of the candidate rows shared by both passes."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    V = W.shape[0]
    _need(W, "W", torch.bfloat16, dev, (V, D))
    _need(targets, "targets", torch.int32, dev, (T,))
    _need(ws, "workspace", torch.uint8, dev)
    cand = torch.empty(C, dtype=torch.int32, device=dev) if cand is None else cand
    slot = torch.empty(T, dtype=torch.int32, device=dev) if slot is None else slot
    loss = torch.empty(T, dtype=torch.float32, device=dev) if loss is None else loss
    lse = torch.empty(T, dtype=torch.float32, device=dev) if lse is None else lse
    dH = torch.empty(T, D, dtype=torch.bfloat16, device=dev) if dH is None else dH
    dW = torch.zeros(V, D, dtype=torch.float32, device=dev) if dW is None else dW
    for t, name, dt, shape in ((cand, "cand", torch.int32, (C,)), (slot, "slot", torch.int32, (T,)),
                               (loss, "loss", torch.float32, (T,)), (lse, "lse", torch.float32, (T,)),
                               (dH, "dH", torch.bfloat16, (T, D)), (dW, "dW", torch.float32, (V, D))):
        _need(t, name, dt, dev, shape)
    if cap == 0 and not fp8:
        code = _lib.ss_step(_ptr(targets), _ptr(H), _ptr(W), T, V, C, D, seed & (2**64 - 1),
                            float(scale), 1 if accumulate else 0, _ptr(cand), _ptr(slot),
                            _ptr(loss), _ptr(lse), _ptr(dH), _ptr(dW), _ptr(ws), ws.numel(),
                            _stream(dev))
    else:
        code = _lib.ss_step_head(_ptr(targets), _ptr(H), _ptr(W), T, V, C, D, seed & (2**64 - 1),
                                 _head(cap, tau, fp8), float(scale), 1 if accumulate else 0,
                                 _ptr(cand), _ptr(slot), _ptr(loss), _ptr(lse), _ptr(dH),
                                 _ptr(dW), _ptr(ws), ws.numel(), _stream(dev))
    _check(code, "ss_step")
    return {"cand": cand, "slot": slot, "loss": loss, "lse": lse, "dH": dH, "dW": dW}


def step_separate(H, W, targets, C: int, seed: int, ws, scale: float = 1.0, dW=None,
                  accumulate=False, cap: float = 0.0, tau: float = 1.0, fp8: int = 0):
    """The same pass as three calls: ss_build_candidates, ss_forward, ss_backward."""
    V = W.shape[0]
    cand, slot = build_candidates(targets, V, C, seed, ws)
    loss, lse = forward(H, W, cand, slot, ws, cap=cap, tau=tau, fp8=fp8)
    dH, dW = backward(H, W, cand, slot, lse, ws, scale=scale, accumulate=accumulate, dW=dW,
                      cap=cap, tau=tau, fp8=fp8)
    return {"cand": cand, "slot": slot, "loss": loss, "lse": lse, "dH": dH, "dW": dW}


SCHEDULE_FULL_STEPS = 87


def schedule_candidates(step: int, total_steps: int, V: int) -> int:
    """C of training step `step` under the pages' candidate schedule
    (ss_schedule_candidates)."""
    c = _lib.ss_schedule_candidates(step, total_steps, V)
    if c < 0:
        raise ValueError(f"ss_schedule_candidates({step}, {total_steps}, {V}): invalid arguments")
    return int(c)


def clear_rows(rows: torch.Tensor, dW: torch.Tensor, ws: torch.Tensor):
    """dW[rows] = 0 (ss_clear_rows); rows: distinct int32 ids."""
    _need(rows, "rows", torch.int32)
    dev = rows.device
    _need(dW, "dW", torch.float32, dev)
    _need(ws, "workspace", torch.uint8, dev)
    V, D = dW.shape
    _check(_lib.ss_clear_rows(_ptr(rows), rows.numel(), V, D, _ptr(dW), _ptr(ws), ws.numel(),
                              _stream(dev)), "ss_clear_rows")


class StepGraph:
    """ss_step captured into a CUDA graph (ss_step_graph_*): the buffers are
    fixed at construction and kept alive here; launch(seed) replays the step
    on the current stream. With `weights` (K of them), the step of several
    targets per token (ss_step_mtp): targets and slot are [K, T]."""

    def __init__(self, H, W, targets, C: int, ws, scale: float = 1.0, accumulate=False,
                 cand=None, slot=None, loss=None, lse=None, dH=None, dW=None, cap: float = 0.0,
                 tau: float = 1.0, fp8: int = 0, weights=None):
        _need(H, "H", torch.bfloat16)
        dev = H.device
        T, D = H.shape
        V = W.shape[0]
        tshape = (T,) if weights is None else (len(weights), T)
        _need(W, "W", torch.bfloat16, dev, (V, D))
        _need(targets, "targets", torch.int32, dev, tshape)
        _need(ws, "workspace", torch.uint8, dev)
        self.cand = torch.empty(C, dtype=torch.int32, device=dev) if cand is None else cand
        self.slot = torch.empty(tshape, dtype=torch.int32, device=dev) if slot is None else slot
        self.loss = torch.empty(T, dtype=torch.float32, device=dev) if loss is None else loss
        self.lse = torch.empty(T, dtype=torch.float32, device=dev) if lse is None else lse
        self.dH = torch.empty(T, D, dtype=torch.bfloat16, device=dev) if dH is None else dH
        self.dW = torch.zeros(V, D, dtype=torch.float32, device=dev) if dW is None else dW
        for t, name, dt, shape in ((self.cand, "cand", torch.int32, (C,)),
                                   (self.slot, "slot", torch.int32, tshape),
                                   (self.loss, "loss", torch.float32, (T,)),
                                   (self.lse, "lse", torch.float32, (T,)),
                                   (self.dH, "dH", torch.bfloat16, (T, D)),
                                   (self.dW, "dW", torch.float32, (V, D))):
            _need(t, name, dt, dev, shape)
        self._keep = (H, W, targets, ws)
        self.device = dev
        h = ctypes.c_void_p()
        outs = (_ptr(self.cand), _ptr(self.slot), _ptr(self.loss), _ptr(self.lse), _ptr(self.dH),
                _ptr(self.dW), _ptr(ws), ws.numel(), ctypes.byref(h))
        if weights is None:
            code = _lib.ss_step_graph_create(_ptr(targets), _ptr(H), _ptr(W), T, V, C, D,
                                             _head(cap, tau, fp8), float(scale),
                                             1 if accumulate else 0, *outs)
            _check(code, "ss_step_graph_create")
        else:
            w, K = _weights(weights)
            self._keep_w = w
            code = _lib.ss_step_graph_create_mtp(_ptr(targets), K, w, _ptr(H), _ptr(W), T, V, C,
                                                 D, _head(cap, tau, fp8), float(scale),
                                                 1 if accumulate else 0, *outs)
            _check(code, "ss_step_graph_create_mtp")
        self._h = h

    def launch(self, seed: int):
        if self._h is None:
            raise RuntimeError("StepGraph is closed")
        _check(_lib.ss_step_graph_launch(self._h, seed & (2**64 - 1), _stream(self.device)),
               "ss_step_graph_launch")
        return {"cand": self.cand, "slot": self.slot, "loss": self.loss, "lse": self.lse,
                "dH": self.dH, "dW": self.dW}

    def close(self):
        if self._h is not None:
            _lib.ss_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


MAX_TARGETS = 8


def _weights(weights):
    w = (ctypes.c_float * len(weights))(*[float(v) for v in weights])
    return w, len(weights)


def step_mtp(H, W, targets, weights, C: int, seed: int, ws, scale: float = 1.0, dW=None,
             accumulate=False, cap: float = 0.0, tau: float = 1.0):
    """ss_step_mtp: targets [K, T] int32 (K weighted targets per token), one
    candidate set over all of them; returns slot [K, T]."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    V = W.shape[0]
    K = len(weights)
    _need(W, "W", torch.bfloat16, dev, (V, D))
    _need(targets, "targets", torch.int32, dev, (K, T))
    _need(ws, "workspace", torch.uint8, dev)
    cand = torch.empty(C, dtype=torch.int32, device=dev)
    slot = torch.empty(K, T, dtype=torch.int32, device=dev)
    loss = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    dH = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    dW = torch.zeros(V, D, dtype=torch.float32, device=dev) if dW is None else dW
    _need(dW, "dW", torch.float32, dev, (V, D))
    w, K = _weights(weights)
    code = _lib.ss_step_mtp(_ptr(targets), K, w, _ptr(H), _ptr(W), T, V, C, D, seed & (2**64 - 1),
                            _head(cap, tau), float(scale), 1 if accumulate else 0, _ptr(cand),
                            _ptr(slot), _ptr(loss), _ptr(lse), _ptr(dH), _ptr(dW), _ptr(ws),
                            ws.numel(), _stream(dev))
    _check(code, "ss_step_mtp")
    return {"cand": cand, "slot": slot, "loss": loss, "lse": lse, "dH": dH, "dW": dW}


def forward_mtp(H, W, cand, slot, weights, ws, cap: float = 0.0, tau: float = 1.0):
    """ss_forward_mtp: slot [K, T]; per-token weighted loss [T] and lse [T]."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    V = W.shape[0]
    C = cand.numel()
    K = len(weights)
    _need(W, "W", torch.bfloat16, dev, (V, D))
    _need(cand, "cand", torch.int32, dev, (C,))
    _need(slot, "slot", torch.int32, dev, (K, T))
    _need(ws, "workspace", torch.uint8, dev)
    loss = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    w, K = _weights(weights)
    code = _lib.ss_forward_mtp(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), K, w, T, V, C, D,
                               _head(cap, tau), _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(),
                               _stream(dev))
    _check(code, "ss_forward_mtp")
    return loss, lse


def backward_mtp(H, W, cand, slot, weights, lse, ws, scale: float = 1.0, accumulate=False,
                 dW=None, cap: float = 0.0, tau: float = 1.0):
    """ss_backward_mtp: dH [T, D] bf16 and dW [V, D] fp32 (candidate rows)."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    T, D = H.shape
    V = W.shape[0]
    C = cand.numel()
    K = len(weights)
    _need(slot, "slot", torch.int32, dev, (K, T))
    _need(lse, "lse", torch.float32, dev, (T,))
    dH = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    dW = torch.zeros(V, D, dtype=torch.float32, device=dev) if dW is None else dW
    _need(dW, "dW", torch.float32, dev, (V, D))
    w, K = _weights(weights)
    code = _lib.ss_backward_mtp(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), K, w, _ptr(lse), T, V,
                                C, D, _head(cap, tau), float(scale), 1 if accumulate else 0,
                                _ptr(dH), _ptr(dW), _ptr(ws), ws.numel(), _stream(dev))
    _check(code, "ss_backward_mtp")
    return dH, dW


def quantize_e4m3(x: torch.Tensor, ws: torch.Tensor):
    """ss_quantize_e4m3: the FP8 head's rounding of one bf16 tensor; returns
    (e4m3 codes as uint8, the rounded values as bf16)."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    xq = torch.empty_like(x)
    _check(_lib.ss_quantize_e4m3(_ptr(x), x.numel(), _ptr(q), _ptr(xq), _ptr(ws), ws.numel(),
                                 _stream(dev)), "ss_quantize_e4m3")
    return q, xq
