"""Python face of the CPU oracle (``ss_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline /
reference arms of ``bench.py`` import this package. It never imports the CUDA
library and the CUDA library never imports it.

Every function here is argument marshalling around the C loops; the arithmetic
and its citations live in ``ss_oracle.c``. The one piece of arithmetic done in
Python is the definition's write-back of candidate-row gradients into the full
[V, D] matrix, ``dW[cand[j]] = dWc[j]`` (or ``+=``), which is plain indexing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libss_oracle.so")

ERR = {0: "ok", 1: "invalid", 3: "capacity (U > C)", 4: "target out of range", 8: "out of memory"}


class OracleError(RuntimeError):
    def __init__(self, code: int, U: int | None = None):
        super().__init__(f"oracle: {ERR.get(code, code)}")
        self.code = code
        self.U = U


def build(force: bool = False) -> str:
    """Compile ss_oracle.c with gcc (OpenMP, no fused multiply-add contraction)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def load(path: str):
    """Load an oracle shared library and declare its C signatures."""
    L = ctypes.CDLL(path)
    L.orc_splitmix64_output.restype = ctypes.c_uint64
    L.orc_splitmix64_output.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    L.orc_negative_key.restype = ctypes.c_uint64
    L.orc_negative_key.argtypes = [ctypes.c_uint64, _i64]
    L.orc_build_candidates.restype = ctypes.c_int
    L.orc_build_candidates.argtypes = [_p, _i64, _i64, _i64, ctypes.c_uint64, _p, _p, _p]
    for suf, real in (("f32", ctypes.c_float), ("f64", ctypes.c_double)):
        f = getattr(L, f"orc_forward_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p]
        f = getattr(L, f"orc_backward_dH_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, real, _p, _i64, _p]
        f = getattr(L, f"orc_backward_dW_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, real, _p, _i64, _p]
        f = getattr(L, f"orc_forward_head_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, real, real, _p, _i64, _p, _p]
        f = getattr(L, f"orc_backward_dH_head_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, real, real, real, _p, _i64, _p]
        f = getattr(L, f"orc_backward_dW_head_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, real, real, real, _p, _i64, _p]
    for suf, real in (("f32", ctypes.c_float), ("f64", ctypes.c_double)):
        f = getattr(L, f"orc_forward_mtp_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _i64, _p, _i64, _i64, _i64, real, real, _p, _i64, _p, _p]
        f = getattr(L, f"orc_backward_dH_mtp_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _i64, _p, _p, _i64, _i64, _i64, real, real, real, _p, _i64,
                      _p]
        f = getattr(L, f"orc_backward_dW_mtp_{suf}")
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _i64, _p, _p, _i64, _i64, _i64, real, real, real, _p, _i64,
                      _p]
    L.orc_round_e4m3.restype = ctypes.c_float
    L.orc_round_e4m3.argtypes = [ctypes.c_float]
    L.orc_e4m3_scale_exponent.restype = ctypes.c_int
    L.orc_e4m3_scale_exponent.argtypes = [ctypes.c_float]
    L.orc_quantize_e4m3_bf16.restype = None
    L.orc_quantize_e4m3_bf16.argtypes = [_p, _i64, ctypes.c_int, _p]
    L.orc_round_e5m2.restype = ctypes.c_float
    L.orc_round_e5m2.argtypes = [ctypes.c_float]
    for name in ("orc_backward_dH_g8", "orc_backward_dW_g8"):
        f = getattr(L, name)
        f.restype = None
        f.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_float, ctypes.c_float,
                      ctypes.c_float, _p, _i64, _p]
    L.orc_g8_exponent.restype = ctypes.c_int
    L.orc_g8_exponent.argtypes = [ctypes.c_float, ctypes.c_float]
    L.orc_num_threads.restype = ctypes.c_int
    L.orc_num_threads.argtypes = []
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _real(dtype):
    dtype = np.dtype(dtype)
    if dtype == np.float32:
        return "f32", np.float32
    if dtype == np.float64:
        return "f64", np.float64
    raise ValueError("oracle precision must be float32 or float64")


def _inputs(M, suf):
    """f32 takes bf16 bit patterns (uint16); f64 takes doubles (bf16 patterns are
    widened exactly, other arrays are taken as real values)."""
    M = np.asarray(M)
    if suf == "f32":
        if M.dtype != np.uint16:
            raise TypeError("the fp32 oracle takes bf16 bit patterns (uint16)")
        return np.ascontiguousarray(M)
    if M.dtype == np.uint16:
        return (np.ascontiguousarray(M).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(M, dtype=np.float64)


def num_threads() -> int:
    return int(lib().orc_num_threads())


def splitmix64_output(seed: int, i: int) -> int:
    return int(lib().orc_splitmix64_output(seed & (2**64 - 1), i))


def negative_key(seed: int, v: int) -> int:
    return int(lib().orc_negative_key(seed & (2**64 - 1), v))


def build_candidates(targets: np.ndarray, V: int, C: int, seed: int):
    """Returns (cand[C] int32, slot[T] int32, U). Raises OracleError on bad input."""
    t = np.ascontiguousarray(targets, dtype=np.int32)
    cand = np.empty(C, np.int32)
    slot = np.empty(t.shape[0], np.int32)
    U = ctypes.c_int64(-1)
    rc = lib().orc_build_candidates(_ptr(t), t.shape[0], V, C, seed & (2**64 - 1),
                                    _ptr(cand), _ptr(slot), ctypes.byref(U))
    if rc != 0:
        raise OracleError(rc, U.value if U.value >= 0 else None)
    return cand, slot, int(U.value)


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.shape[0]


def forward(H, W, cand, slot, rows=None, dtype=np.float32, cap=0.0, tau=1.0):
    """Per-token (loss, lse) for all tokens or for the listed token rows.
    cap > 0: the capped head z = cap / (1 + exp(-s / tau)) (cap = 0: plain)."""
    suf, real = _real(dtype)
    H = _inputs(H, suf)
    W = _inputs(W, suf)
    cand = np.ascontiguousarray(cand, np.int32)
    slot = np.ascontiguousarray(slot, np.int32)
    T, D = H.shape
    C = cand.shape[0]
    r, nr = _rows(rows)
    n = nr if r is not None else T
    loss = np.empty(n, real)
    lse = np.empty(n, real)
    getattr(lib(), f"orc_forward_head_{suf}")(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), T, C, D,
                                              cap, tau, _ptr(r), nr, _ptr(loss), _ptr(lse))
    return loss, lse


def backward_dH(H, W, cand, slot, lse_rows, scale=1.0, rows=None, dtype=np.float32, cap=0.0,
                tau=1.0):
    """dH rows [n, D]; lse_rows are the oracle's lse of exactly those rows."""
    suf, real = _real(dtype)
    H = _inputs(H, suf)
    W = _inputs(W, suf)
    cand = np.ascontiguousarray(cand, np.int32)
    slot = np.ascontiguousarray(slot, np.int32)
    lse_rows = np.ascontiguousarray(lse_rows, real)
    T, D = H.shape
    C = cand.shape[0]
    r, nr = _rows(rows)
    n = nr if r is not None else T
    assert lse_rows.shape[0] == n
    dH = np.empty((n, D), real)
    getattr(lib(), f"orc_backward_dH_head_{suf}")(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot),
                                                  _ptr(lse_rows), T, C, D, cap, tau, scale,
                                                  _ptr(r), nr, _ptr(dH))
    return dH


def backward_dWc(H, W, cand, slot, lse, scale=1.0, cols=None, dtype=np.float32, cap=0.0,
                 tau=1.0):
    """Candidate-row gradients dWc [n, D] (row i belongs to vocabulary row cand[cols[i]]).
    `lse` must be the oracle's lse of ALL T tokens."""
    suf, real = _real(dtype)
    H = _inputs(H, suf)
    W = _inputs(W, suf)
    cand = np.ascontiguousarray(cand, np.int32)
    slot = np.ascontiguousarray(slot, np.int32)
    lse = np.ascontiguousarray(lse, real)
    T, D = H.shape
    C = cand.shape[0]
    assert lse.shape[0] == T
    c, nc = _rows(cols)
    n = nc if c is not None else C
    dWc = np.empty((n, D), real)
    getattr(lib(), f"orc_backward_dW_head_{suf}")(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot),
                                                  _ptr(lse), T, C, D, cap, tau, scale, _ptr(c),
                                                  nc, _ptr(dWc))
    return dWc


def loss_and_grads(H, W, targets, C, seed, scale=1.0, dtype=np.float32, dW_init=None,
                   accumulate=False, cap=0.0, tau=1.0):
    """The whole definition on one batch: candidates, per-token loss and lse,
    dH [T, D], and dW [V, D] whose candidate rows are written (or added to)."""
    V = W.shape[0]
    cand, slot, U = build_candidates(targets, V, C, seed)
    loss, lse = forward(H, W, cand, slot, dtype=dtype, cap=cap, tau=tau)
    dH = backward_dH(H, W, cand, slot, lse, scale, dtype=dtype, cap=cap, tau=tau)
    dWc = backward_dWc(H, W, cand, slot, lse, scale, dtype=dtype, cap=cap, tau=tau)
    _, real = _real(dtype)
    dW = np.zeros(W.shape, real) if dW_init is None else np.array(dW_init, dtype=real, copy=True)
    if accumulate:
        dW[cand] += dWc
    else:
        dW[cand] = dWc
    return {"cand": cand, "slot": slot, "U": U, "loss": loss, "lse": lse, "dH": dH, "dW": dW,
            "dWc": dWc}


# -------------------------------------------------- several targets per token

def _mtp_args(slot, weights, real):
    slot = np.ascontiguousarray(slot, np.int32)
    assert slot.ndim == 2, "slot is [K, T]"
    w = np.ascontiguousarray(weights, real)
    assert w.shape == (slot.shape[0],)
    return slot, w


def forward_mtp(H, W, cand, slot, weights, rows=None, dtype=np.float32, cap=0.0, tau=1.0):
    """K targets per token (slot [K, T], weights [K]): per-token
    loss = sum_k w[k] (lse - z[slot[k]]) and lse, for all tokens or the listed rows."""
    suf, real = _real(dtype)
    H = _inputs(H, suf)
    W = _inputs(W, suf)
    cand = np.ascontiguousarray(cand, np.int32)
    slot, w = _mtp_args(slot, weights, real)
    K, T = slot.shape
    D = H.shape[1]
    C = cand.shape[0]
    r, nr = _rows(rows)
    n = nr if r is not None else T
    loss = np.empty(n, real)
    lse = np.empty(n, real)
    getattr(lib(), f"orc_forward_mtp_{suf}")(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), K, _ptr(w),
                                             T, C, D, cap, tau, _ptr(r), nr, _ptr(loss),
                                             _ptr(lse))
    return loss, lse


def backward_dH_mtp(H, W, cand, slot, weights, lse_rows, scale=1.0, rows=None, dtype=np.float32,
                    cap=0.0, tau=1.0):
    suf, real = _real(dtype)
    H = _inputs(H, suf)
    W = _inputs(W, suf)
    cand = np.ascontiguousarray(cand, np.int32)
    slot, w = _mtp_args(slot, weights, real)
    K, T = slot.shape
    D = H.shape[1]
    C = cand.shape[0]
    lse_rows = np.ascontiguousarray(lse_rows, real)
    r, nr = _rows(rows)
    n = nr if r is not None else T
    assert lse_rows.shape[0] == n
    dH = np.empty((n, D), real)
    getattr(lib(), f"orc_backward_dH_mtp_{suf}")(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), K,
                                                 _ptr(w), _ptr(lse_rows), T, C, D, cap, tau,
                                                 scale, _ptr(r), nr, _ptr(dH))
    return dH


def backward_dWc_mtp(H, W, cand, slot, weights, lse, scale=1.0, cols=None, dtype=np.float32,
                     cap=0.0, tau=1.0):
    suf, real = _real(dtype)
    H = _inputs(H, suf)
    W = _inputs(W, suf)
    cand = np.ascontiguousarray(cand, np.int32)
    slot, w = _mtp_args(slot, weights, real)
    K, T = slot.shape
    D = H.shape[1]
    C = cand.shape[0]
    lse = np.ascontiguousarray(lse, real)
    assert lse.shape[0] == T
    c, nc = _rows(cols)
    n = nc if c is not None else C
    dWc = np.empty((n, D), real)
    getattr(lib(), f"orc_backward_dW_mtp_{suf}")(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), K,
                                                 _ptr(w), _ptr(lse), T, C, D, cap, tau, scale,
                                                 _ptr(c), nc, _ptr(dWc))
    return dWc


def loss_and_grads_mtp(H, W, targets, weights, C, seed, scale=1.0, dtype=np.float32, cap=0.0,
                       tau=1.0):
    """targets [K, T]: the candidate set is built over all K*T targets (k-major);
    returns the same keys as loss_and_grads with slot [K, T]."""
    targets = np.ascontiguousarray(targets, np.int32)
    K, T = targets.shape
    V = W.shape[0]
    cand, slot_flat, U = build_candidates(targets.reshape(-1), V, C, seed)
    slot = slot_flat.reshape(K, T)
    loss, lse = forward_mtp(H, W, cand, slot, weights, dtype=dtype, cap=cap, tau=tau)
    dH = backward_dH_mtp(H, W, cand, slot, weights, lse, scale, dtype=dtype, cap=cap, tau=tau)
    dWc = backward_dWc_mtp(H, W, cand, slot, weights, lse, scale, dtype=dtype, cap=cap, tau=tau)
    _, real = _real(dtype)
    dW = np.zeros(W.shape, real)
    dW[cand] = dWc
    return {"cand": cand, "slot": slot, "U": U, "loss": loss, "lse": lse, "dH": dH, "dW": dW,
            "dWc": dWc}


# ------------------------------------------------------------------ FP8 head

def round_e4m3(x: float) -> float:
    return float(lib().orc_round_e4m3(x))


def e4m3_scale_exponent(amax: float) -> int:
    return int(lib().orc_e4m3_scale_exponent(amax))


def quantize_e4m3(bits: np.ndarray, e: int | None = None):
    """bf16 bit patterns -> (rounded bf16 bit patterns, e): every value scaled
    by 2^e (e from the tensor's amax unless given), rounded to e4m3, scaled back."""
    b = np.ascontiguousarray(bits, np.uint16)
    if e is None:
        from synth import bf16_bits_to_f32
        amax = float(np.abs(bf16_bits_to_f32(b)).max()) if b.size else 0.0
        e = e4m3_scale_exponent(amax)
    out = np.empty_like(b)
    lib().orc_quantize_e4m3_bf16(_ptr(b), b.size, e, _ptr(out))
    return out, e


def fp8_inputs(H, W, cand):
    """The FP8 head's operands: H rounded with its own exponent, the candidate
    rows of W rounded with theirs (the other rows of W are never read)."""
    Hq, eH = quantize_e4m3(H)
    Wc_q, eW = quantize_e4m3(np.asarray(W)[cand])
    Wq = np.array(W, copy=True)
    Wq[cand] = Wc_q
    return Hq, Wq, eH, eW


def round_e5m2(x: float) -> float:
    return float(lib().orc_round_e5m2(x))


def g8_exponent(cap: float = 0.0, tau: float = 1.0) -> int:
    return int(lib().orc_g8_exponent(cap, tau))


def backward_dH_g8(H, W, cand, slot, lse_rows, scale=1.0, rows=None, cap=0.0, tau=1.0):
    """FP8 gradients (e5m2 G, one target; cap > 0: the capped head): dH rows
    [n, D] on operands already rounded to e4m3 (bf16 bit patterns)."""
    H = _inputs(H, "f32")
    W = _inputs(W, "f32")
    cand = np.ascontiguousarray(cand, np.int32)
    slot = np.ascontiguousarray(slot, np.int32)
    lse_rows = np.ascontiguousarray(lse_rows, np.float32)
    T, D = H.shape
    r, nr = _rows(rows)
    n = nr if r is not None else T
    assert lse_rows.shape[0] == n
    dH = np.empty((n, D), np.float32)
    lib().orc_backward_dH_g8(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), _ptr(lse_rows), T,
                             cand.shape[0], D, cap, tau, scale, _ptr(r), nr, _ptr(dH))
    return dH


def backward_dWc_g8(H, W, cand, slot, lse, scale=1.0, cols=None, cap=0.0, tau=1.0):
    """FP8 gradients: candidate-row gradients dWc [n, D]; `lse` of ALL T tokens."""
    H = _inputs(H, "f32")
    W = _inputs(W, "f32")
    cand = np.ascontiguousarray(cand, np.int32)
    slot = np.ascontiguousarray(slot, np.int32)
    lse = np.ascontiguousarray(lse, np.float32)
    T, D = H.shape
    C = cand.shape[0]
    assert lse.shape[0] == T
    c, nc = _rows(cols)
    n = nc if c is not None else C
    dWc = np.empty((n, D), np.float32)
    lib().orc_backward_dW_g8(_ptr(H), _ptr(W), _ptr(cand), _ptr(slot), _ptr(lse), T, C, D, cap,
                             tau, scale, _ptr(c), nc, _ptr(dWc))
    return dWc


def loss_and_grads_fp8(H, W, targets, C, seed, scale=1.0, dW_init=None, accumulate=False,
                       grads=False, cap=0.0, tau=1.0):
    """The whole definition with the FP8 head: the single-target loss and its
    gradients on the rounded operands (rows of dW outside cand untouched);
    grads=True: FP8 through the backward too (e5m2 G); cap > 0: the capped
    head on the rounded operands."""
    V = W.shape[0]
    cand, slot, U = build_candidates(targets, V, C, seed)
    Hq, Wq, eH, eW = fp8_inputs(H, W, cand)
    loss, lse = forward(Hq, Wq, cand, slot, cap=cap, tau=tau)
    if grads:
        dH = backward_dH_g8(Hq, Wq, cand, slot, lse, scale, cap=cap, tau=tau)
        dWc = backward_dWc_g8(Hq, Wq, cand, slot, lse, scale, cap=cap, tau=tau)
    else:
        dH = backward_dH(Hq, Wq, cand, slot, lse, scale, cap=cap, tau=tau)
        dWc = backward_dWc(Hq, Wq, cand, slot, lse, scale, cap=cap, tau=tau)
    dW = np.zeros(W.shape, np.float32) if dW_init is None else np.array(dW_init, np.float32)
    if accumulate:
        dW[cand] += dWc
    else:
        dW[cand] = dWc
    return {"cand": cand, "slot": slot, "U": U, "loss": loss, "lse": lse, "dH": dH, "dW": dW,
            "dWc": dWc, "eH": eH, "eW": eW}
