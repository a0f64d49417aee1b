"""A device-side wait that runs out returns SS_ERR_TIMEOUT, and the library
stays usable.

Every wait in the library's kernels is bounded: after its limit the kernel
records SS_ERR_TIMEOUT in the workspace status word and returns, instead of
spinning forever or trapping. This test reaches that path without a fault:
it builds a copy of the library whose grid barrier (the one of the FP8 head's
H preparation beside the candidate build, a plain spin on a counter with no
copies or tensor-core work in flight) waits for one more arrival than its grid
has blocks, with a 1 ms limit. An FP8 ss_step through that copy must then
report SS_ERR_TIMEOUT and leave its outputs untouched, and the next step on
the same workspace (plain head, which has no such barrier) must succeed and
match the oracle.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_util import GRAD_RTOL, assert_loss_close, rel_fro, to_dev_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import sampled_softmax_output_gb300 as ss  # noqa: E402  (fails loudly if libss.so is missing)


@pytest.fixture(scope="module")
def short_wait_lib(tmp_path_factory):
    from sampled_softmax_output_gb300 import build as b
    out = str(tmp_path_factory.mktemp("ss_short_wait"))
    lib = ctypes.CDLL(b.build_variant(out, ["SS_BESIDE_EXTRA_ARRIVALS=1",
                                            "SS_BESIDE_WAIT_NS=1000000ull"]))
    p, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.ss_step_head.restype = ctypes.c_int
    lib.ss_step_head.argtypes = [p, p, p, i64, i64, i64, i64, ctypes.c_uint64,
                                 ctypes.POINTER(ss.Head), ctypes.c_float, ctypes.c_int, p, p, p,
                                 p, p, p, p, sz, p]
    lib.ss_read_status.restype = ctypes.c_int
    lib.ss_read_status.argtypes = [p, sz, p, ctypes.POINTER(ctypes.c_int32),
                                   ctypes.POINTER(ctypes.c_int32)]
    return lib


def _step(lib, H, W, tg, C, seed, ws, out, head):
    T, D = H.shape
    V = W.shape[0]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = lib.ss_step_head(ptr(tg), ptr(H), ptr(W), T, V, C, D, seed,
                            ctypes.byref(head) if head is not None else None, 1.0 / T, 0,
                            ptr(out["cand"]), ptr(out["slot"]), ptr(out["loss"]),
                            ptr(out["lse"]), ptr(out["dH"]), ptr(out["dW"]), ptr(ws),
                            ws.numel(), stream)
    st, U = ctypes.c_int32(0), ctypes.c_int32(0)
    lib.ss_read_status(ptr(ws), ws.numel(), stream, ctypes.byref(st), ctypes.byref(U))
    return code, st.value


def test_barrier_wait_runs_out_then_the_next_step_succeeds(short_wait_lib, orc):
    T, V, D, C, seed = 300, 3000, 256, 517, 4
    x = synth.make_inputs(T, V, D, 1.1, seed)
    C = max(C, len(np.unique(x["targets"])))
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    out = {"cand": torch.empty(C, dtype=torch.int32, device="cuda"),
           "slot": torch.empty(T, dtype=torch.int32, device="cuda"),
           "loss": torch.full((T,), -5.0, device="cuda"),
           "lse": torch.full((T,), -5.0, device="cuda"),
           "dH": torch.full((T, D), 3.0, dtype=torch.bfloat16, device="cuda"),
           "dW": torch.full((V, D), 7.0, device="cuda")}
    # 1: the FP8 step's barrier waits 1 ms for an arrival that never comes
    code, st = _step(short_wait_lib, H, W, tg, C, seed, ws, out, ss.Head(0.0, 1.0, 1))
    assert code == 0          # enqueued; the error is the device's
    assert st == 7            # SS_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert torch.all(out["loss"] == -5.0) and torch.all(out["lse"] == -5.0)
    assert torch.all(out["dH"].float() == 3.0) and torch.all(out["dW"] == 7.0)
    # 2: the same library and workspace, plain head: the candidate build clears
    # the status word and the step succeeds
    code, st = _step(short_wait_lib, H, W, tg, C, seed, ws, out, None)
    assert code == 0 and st == 0
    ref = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, seed, 1.0 / T)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out["cand"].cpu().numpy(), ref["cand"])
    assert_loss_close(out["loss"].cpu().numpy(), ref["loss"])
    assert rel_fro(out["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL
    c = ref["cand"]
    dW = out["dW"].cpu().numpy()
    assert rel_fro(dW[c], ref["dW"][c]) < GRAD_RTOL
    assert np.all(np.delete(dW, c, axis=0) == 7.0)  # rows outside the set untouched
