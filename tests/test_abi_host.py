"""Host-side checks of the C ABI: the library loads without a GPU, exports every
function include/ss.h declares, sizes its workspace, and rejects bad arguments
before it touches the device (these paths make no CUDA call, so they run on a
machine without a GPU; the fake device addresses below are never dereferenced)."""
import ctypes

import pytest

import sampled_softmax_output_gb300 as ss  # noqa: E402  (fails loudly if libss.so is missing)

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 5
FAKE = 0x7F0000000000  # 4 KB-aligned address, never dereferenced
p = ctypes.c_void_p


def test_exports_every_declared_symbol():
    names = ss.header_symbols()
    assert set(names) == {"ss_workspace_size", "ss_build_candidates", "ss_forward",
                          "ss_backward", "ss_read_status", "ss_status_string",
                          "ss_trace_begin", "ss_trace_end", "ss_trace_kernel_name",
                          "ss_trace_kernel_launches",
                          "ss_last_error", "ss_forward_noalloc", "ss_step",
                          "ss_schedule_candidates", "ss_clear_rows", "ss_step_graph_create",
                          "ss_step_graph_create_mtp",
                          "ss_step_graph_launch", "ss_step_graph_destroy", "ss_forward_head",
                          "ss_backward_head", "ss_step_head", "ss_forward_mtp", "ss_backward_mtp",
                          "ss_step_mtp", "ss_quantize_e4m3"}
    for n in names:
        assert hasattr(ss.lib(), n), n


def test_status_strings():
    L = ss.lib()
    for code in range(9):
        s = L.ss_status_string(code)
        assert s and s != b"unknown status"
    assert L.ss_status_string(99) == b"unknown status"


def test_workspace_size():
    L = ss.lib()
    T, V, C, D = 16384, 50304, 10240, 768
    n = L.ss_workspace_size(T, V, C, D)
    # at least the bf16 softmax-gradient matrix and the gathered candidate rows
    assert n >= T * C * 2 + C * D * 2
    assert n % 1024 == 0
    assert L.ss_workspace_size(0, V, C, D) > 0             # empty batch is valid
    assert L.ss_workspace_size(T, V, V + 1, D) == 0        # C > V
    assert L.ss_workspace_size(T, V, 0, D) == 0            # C = 0
    assert L.ss_workspace_size(T, V, C, 100) == 0          # D % 64 != 0
    assert L.ss_workspace_size(T, ss.MAX_V + 1, C, D) == 0
    assert L.ss_workspace_size(-1, V, C, D) == 0
    # monotone in every size
    assert L.ss_workspace_size(2 * T, V, C, D) > n and L.ss_workspace_size(T, V, 2 * C, D) > n


def _fwd(**kw):
    a = dict(H=FAKE, W=FAKE, cand=FAKE, slot=FAKE, T=256, V=50304, C=4096, D=768, loss=FAKE,
             lse=FAKE, ws=FAKE, wsb=1 << 40)
    a.update(kw)
    return ss.lib().ss_forward(p(a["H"]), p(a["W"]), p(a["cand"]), p(a["slot"]), a["T"], a["V"],
                               a["C"], a["D"], p(a["loss"]), p(a["lse"]), p(a["ws"]), a["wsb"],
                               None)


def _bwd(**kw):
    a = dict(H=FAKE, W=FAKE, cand=FAKE, slot=FAKE, lse=FAKE, T=256, V=50304, C=4096, D=768,
             scale=1.0, acc=0, dH=FAKE, dW=FAKE, ws=FAKE, wsb=1 << 40)
    a.update(kw)
    return ss.lib().ss_backward(p(a["H"]), p(a["W"]), p(a["cand"]), p(a["slot"]), p(a["lse"]),
                                a["T"], a["V"], a["C"], a["D"], a["scale"], a["acc"], p(a["dH"]),
                                p(a["dW"]), p(a["ws"]), a["wsb"], None)


def _cand(**kw):
    a = dict(targets=FAKE, T=256, V=50304, C=4096, seed=0, cand=FAKE, slot=FAKE, U=None, ws=FAKE,
             wsb=1 << 20)
    a.update(kw)
    return ss.lib().ss_build_candidates(p(a["targets"]), a["T"], a["V"], a["C"], a["seed"],
                                        p(a["cand"]), p(a["slot"]), a["U"], p(a["ws"]), a["wsb"],
                                        None)


@pytest.mark.parametrize("fn", [_fwd, _bwd, _cand])
def test_size_errors(fn):
    assert fn(C=0) == INVALID
    assert fn(C=50305) == INVALID
    assert fn(T=-1) == INVALID
    assert fn(V=ss.MAX_V + 1, C=10) == UNSUPPORTED
    assert fn(T=1 << 31) == UNSUPPORTED


@pytest.mark.parametrize("fn", [_fwd, _bwd])
def test_width_errors(fn):
    assert fn(D=100) == UNSUPPORTED
    assert fn(D=0) == INVALID
    assert fn(D=ss.MAX_D + 64) == UNSUPPORTED


def test_null_and_alignment_errors():
    for k in ("H", "W", "cand", "slot", "loss", "lse", "ws"):
        assert _fwd(**{k: 0}) == INVALID, k
    for k in ("H", "W", "ws"):
        assert _fwd(**{k: FAKE + 8}) == INVALID, k      # 16-byte alignment
    for k in ("cand", "slot", "loss", "lse"):
        assert _fwd(**{k: FAKE + 2}) == INVALID, k      # 4-byte alignment
    for k in ("H", "W", "cand", "slot", "lse", "dH", "dW", "ws"):
        assert _bwd(**{k: 0}) == INVALID, k
    assert _bwd(dH=FAKE + 8) == INVALID and _bwd(dW=FAKE + 4) == INVALID
    assert _bwd(acc=2) == INVALID
    for k in ("targets", "cand", "slot", "ws"):
        assert _cand(**{k: 0}) == INVALID, k
    assert _cand(targets=FAKE + 1) == INVALID


def _step(**kw):
    a = dict(targets=FAKE, H=FAKE, W=FAKE, T=256, V=50304, C=4096, D=768, seed=0, scale=1.0, acc=0,
             cand=FAKE, slot=FAKE, loss=FAKE, lse=FAKE, dH=FAKE, dW=FAKE, ws=FAKE, wsb=1 << 40)
    a.update(kw)
    return ss.lib().ss_step(p(a["targets"]), p(a["H"]), p(a["W"]), a["T"], a["V"], a["C"], a["D"],
                            a["seed"], a["scale"], a["acc"], p(a["cand"]), p(a["slot"]),
                            p(a["loss"]), p(a["lse"]), p(a["dH"]), p(a["dW"]), p(a["ws"]),
                            a["wsb"], None)


def test_step_argument_errors():
    assert _step(C=0) == INVALID and _step(D=100) == UNSUPPORTED
    for k in ("targets", "H", "W", "cand", "slot", "loss", "lse", "dH", "dW", "ws"):
        assert _step(**{k: 0}) == INVALID, k
    assert _step(H=FAKE + 8) == INVALID and _step(acc=3) == INVALID
    need = ss.lib().ss_workspace_size(256, 50304, 4096, 768)
    assert _step(wsb=need - 1) == WORKSPACE


def test_workspace_too_small():
    L = ss.lib()
    need = L.ss_workspace_size(256, 50304, 4096, 768)
    assert _fwd(wsb=need - 1) == WORKSPACE
    assert _bwd(wsb=need - 1) == WORKSPACE
    assert _cand(wsb=16) == WORKSPACE
    assert L.ss_read_status(p(FAKE), 16, None, None, None) == WORKSPACE
    assert L.ss_read_status(None, 1 << 20, None, None, None) == INVALID


def test_trace_bookkeeping_without_launches():
    L = ss.lib()
    assert L.ss_trace_begin(None, -1) == INVALID
    assert L.ss_trace_begin(None, 4) == INVALID
    assert L.ss_trace_begin(None, 0) == OK
    assert L.ss_trace_end() == 0
    assert L.ss_trace_kernel_name(0) is None


def test_empty_batch_forward_is_a_no_op():
    # T = 0: nothing to compute, returns before any device work
    assert _fwd(T=0, H=0, slot=0, loss=0, lse=0) == OK


def test_schedule_candidates():
    """The pages' schedule: 10,240 / 14,336 / 24,576 candidates in three equal
    phases, then all V rows for the final 87 steps."""
    V = 50304
    for total in (87, 88, 100, 3000, 5960):
        cs = [ss.schedule_candidates(s, total, V) for s in range(total)]
        assert cs[-87:] == [V] * 87
        head = cs[:total - 87]
        assert head == sorted(head)                       # phases in order
        counts = [head.count(c) for c in (10240, 14336, 24576)]
        assert sum(counts) == len(head)
        assert max(counts) - min(counts) <= 1             # equal phases (+-1 step)
    assert ss.schedule_candidates(0, 3000, 8000) == 8000  # capped at V
    L = ss.lib()
    for args in ((-1, 10, V), (10, 10, V), (0, 0, V), (0, 10, 0), (0, 10, (1 << 19) + 1)):
        assert L.ss_schedule_candidates(*args) == -1, args


def test_clear_rows_argument_errors():
    L = ss.lib()

    def clear(rows=FAKE, n=16, V=50304, D=768, dW=FAKE, ws=FAKE, wsb=1 << 20):
        return L.ss_clear_rows(p(rows), n, V, D, p(dW), p(ws), wsb, None)

    assert clear(n=0) == OK                        # nothing to do, nothing enqueued
    assert clear(n=-1) == INVALID and clear(n=50305) == INVALID and clear(V=0) == INVALID
    assert clear(V=(1 << 19) + 1, n=1) == UNSUPPORTED and clear(D=100) == UNSUPPORTED
    assert clear(rows=0) == INVALID and clear(dW=0) == INVALID and clear(ws=0) == INVALID
    assert clear(rows=FAKE + 2) == INVALID and clear(dW=FAKE + 8) == INVALID
    assert clear(wsb=16) == WORKSPACE


def test_step_graph_argument_errors():
    L = ss.lib()
    h = ctypes.c_void_p()

    def create(**kw):
        a = dict(targets=FAKE, H=FAKE, W=FAKE, T=256, V=50304, C=4096, D=768, scale=1.0, acc=0,
                 cand=FAKE, slot=FAKE, loss=FAKE, lse=FAKE, dH=FAKE, dW=FAKE, ws=FAKE,
                 wsb=1 << 40)
        a.update(kw)
        return L.ss_step_graph_create(p(a["targets"]), p(a["H"]), p(a["W"]), a["T"], a["V"],
                                      a["C"], a["D"], a.get("head"), a["scale"], a["acc"],
                                      p(a["cand"]),
                                      p(a["slot"]), p(a["loss"]), p(a["lse"]), p(a["dH"]),
                                      p(a["dW"]), p(a["ws"]), a["wsb"], ctypes.byref(h))

    assert create(C=0) == INVALID and create(D=100) == UNSUPPORTED and create(acc=2) == INVALID
    assert create(H=0) == INVALID and create(dW=FAKE + 4) == INVALID
    need = L.ss_workspace_size(256, 50304, 4096, 768)
    assert create(wsb=need - 1) == WORKSPACE
    assert h.value is None                          # nothing was created
    assert L.ss_step_graph_launch(None, 0, None) == INVALID
    L.ss_step_graph_destroy(None)                   # a no-op


def test_several_targets_step_graph_argument_errors():
    L = ss.lib()
    h = ctypes.c_void_p()

    def create(K=2, w=(1.0, 0.5), head=None, wsb=1 << 40, C=4096, out=True):
        wa = (ctypes.c_float * max(len(w), 1))(*w)
        return L.ss_step_graph_create_mtp(p(FAKE), K, wa, p(FAKE), p(FAKE), 256, 50304, C, 768,
                                          head, 1.0, 0, p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                                          p(FAKE), p(FAKE), p(FAKE), wsb,
                                          ctypes.byref(h) if out else None)

    assert create(K=0, w=()) == INVALID and create(K=9, w=(1.0,) * 9) == INVALID
    assert create(w=(1.0, -0.5)) == INVALID and create(w=(0.0, 0.0)) == INVALID
    assert create(head=ctypes.byref(ss.Head(0.0, 1.0, 1))) == UNSUPPORTED  # no FP8 path
    assert create(C=0) == INVALID and create(out=False) == INVALID
    need = L.ss_workspace_size(256, 50304, 4096, 768)
    assert create(wsb=need - 1) == WORKSPACE
    assert h.value is None


def test_head_argument_errors():
    """Head options: cap 0 (or NULL) is the plain head; a negative or
    non-finite cap, or a capped head without a positive finite tau, is invalid."""
    L = ss.lib()
    a = dict(H=FAKE, W=FAKE, cand=FAKE, slot=FAKE, T=256, V=50304, C=4096, D=768)

    def fwd(head, wsb=1 << 40):
        return L.ss_forward_head(p(a["H"]), p(a["W"]), p(a["cand"]), p(a["slot"]), 0, a["V"],
                                 a["C"], a["D"], head, p(FAKE), p(FAKE), p(FAKE), wsb, None)

    def step(head):
        return L.ss_step_head(p(FAKE), p(FAKE), p(FAKE), 0, 50304, 4096, 768, 0, head, 1.0, 0,
                              p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                              16, None)

    assert fwd(None) == OK and fwd(ctypes.byref(ss.Head(0.0, 0.0))) == OK  # T = 0: no-op
    for cap, tau in ((-1.0, 1.0), (30.0, 0.0), (30.0, -2.0), (float("inf"), 1.0),
                     (float("nan"), 1.0), (30.0, float("nan"))):
        h = ctypes.byref(ss.Head(cap, tau))
        assert fwd(h) == INVALID, (cap, tau)
        assert step(h) == INVALID, (cap, tau)
        bwd = L.ss_backward_head(p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), 0, 50304, 4096, 768,
                                 h, 1.0, 0, p(FAKE), p(FAKE), p(FAKE), 1 << 40, None)
        assert bwd == INVALID, (cap, tau)
    assert fwd(ctypes.byref(ss.Head(30.0, 7.5)), wsb=16) == WORKSPACE


def test_several_targets_argument_errors():
    """K in [1, SS_MAX_TARGETS]; weights finite, >= 0, with a positive sum."""
    L = ss.lib()

    def step(weights, K=None, T=0, wsb=1 << 40):
        w = (ctypes.c_float * max(1, len(weights)))(*weights) if weights else None
        K = len(weights) if K is None else K
        return L.ss_step_mtp(p(FAKE), K, w, p(FAKE), p(FAKE), T, 50304, 4096, 768, 0, None, 1.0, 0,
                             p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), wsb,
                             None)

    for bad in ([], [0.0], [0.0, 0.0], [-1.0, 2.0], [float("nan")], [float("inf"), 1.0],
                [1.0] * 9):
        assert step(bad) == INVALID, bad
    assert step([1.0], K=0) == INVALID
    need = L.ss_workspace_size(256, 50304, 4096, 768)
    assert step([1.0, 0.5], T=256, wsb=need - 1) == WORKSPACE
    w = (ctypes.c_float * 2)(1.0, -0.5)
    assert L.ss_forward_mtp(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 2, w, 0, 50304, 4096, 768, None,
                            p(FAKE), p(FAKE), p(FAKE), 1 << 40, None) == INVALID
    assert L.ss_backward_mtp(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 2, w, p(FAKE), 0, 50304, 4096,
                             768, None, 1.0, 0, p(FAKE), p(FAKE), p(FAKE), 1 << 40,
                             None) == INVALID


def test_fp8_head_argument_errors():
    """The FP8 head (capped or not) needs D % 128 == 0; the
    several-targets entry points have no FP8 path; fp8 must be 0, 1 or 2."""
    L = ss.lib()

    def step(head, D=768, T=256):  # a workspace too small: accepted arguments say so
        return L.ss_step_head(p(FAKE), p(FAKE), p(FAKE), T, 50304, 4096, D, 0, head, 1.0, 0,
                              p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                              16, None)

    assert step(ctypes.byref(ss.Head(0.0, 1.0, 1))) == WORKSPACE       # the FP8 head is accepted
    assert step(ctypes.byref(ss.Head(30.0, 7.5, 1))) == WORKSPACE      # capped FP8 head
    assert step(ctypes.byref(ss.Head(0.0, 1.0, 1)), D=192) == UNSUPPORTED
    assert step(ctypes.byref(ss.Head(0.0, 1.0, 2))) == WORKSPACE       # FP8 gradients too
    assert step(ctypes.byref(ss.Head(30.0, 7.5, 2))) == WORKSPACE
    assert step(ctypes.byref(ss.Head(-1.0, 7.5, 2))) == INVALID
    assert step(ctypes.byref(ss.Head(0.0, 1.0, 2)), D=192) == UNSUPPORTED
    assert step(ctypes.byref(ss.Head(0.0, 1.0, 3))) == INVALID
    assert step(ctypes.byref(ss.Head(0.0, 1.0, -1))) == INVALID
    w = (ctypes.c_float * 1)(1.0)
    assert L.ss_step_mtp(p(FAKE), 1, w, p(FAKE), p(FAKE), 0, 50304, 4096, 768, 0,
                         ctypes.byref(ss.Head(0.0, 1.0, 1)), 1.0, 0, p(FAKE), p(FAKE), p(FAKE),
                         p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1 << 40, None) == UNSUPPORTED
    q = L.ss_quantize_e4m3
    assert q(p(FAKE), 0, p(FAKE), p(FAKE), p(FAKE), 1024, None) == OK
    assert q(p(FAKE), 12, p(FAKE), p(FAKE), p(FAKE), 1024, None) == INVALID    # n % 8
    assert q(p(FAKE + 8), 16, p(FAKE), p(FAKE), p(FAKE), 1024, None) == INVALID
    assert q(p(FAKE), 16, p(FAKE), p(FAKE), p(FAKE), 16, None) == WORKSPACE
