"""The allocation-free forward entry point, ss_forward_noalloc.

Some callers cannot allocate device memory: a plugin inside a host program
that owns and has planned all device memory gets only its input and output
buffers, and some latency-critical paths cannot afford a cudaMalloc, which may
synchronise the device. They cannot provide the workspace that ss_forward
needs, so ss_forward_noalloc keeps its scratch in a fixed array inside the
library's device data instead.

These tests call it through the C ABI and check its loss and lse against the
ordinary ss_forward (itself checked here against the CPU oracle), within the
tolerance the other parity tests use, on calls
in a row on the shared array: a larger batch first, then a call with a
candidate id out of range (the gather's bounds check reports SS_ERR_INDEX
without touching memory outside W), then a smaller valid batch, which must
return SS_OK (each call clears the status word) and must not read the larger
call's leftover partials or target logits. Also its size limit. This file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import LOSS_RTOL, to_dev_bf16

import sampled_softmax_output_gb300 as ss  # noqa: E402  (fails loudly if libss.so is missing)

pytestmark = pytest.mark.gpu


def _batch(T, V, D, C, seed, orc):
    x = synth.make_inputs(T, V, D, 1.1, seed)
    C = max(C, len(np.unique(x["targets"])))
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    targets = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    cand, slot = ss.build_candidates(targets, V, C, seed, ws)
    ref_loss, ref_lse = ss.forward(H, W, cand, slot, ws)
    # the ordinary forward itself against the CPU oracle
    o_loss, o_lse = orc.forward(x["H"], x["W"], cand.cpu().numpy(), slot.cpu().numpy())
    _close(ref_loss, torch.from_numpy(o_loss))
    _close(ref_lse, torch.from_numpy(o_lse))
    return H, W, cand, slot, ref_loss, ref_lse


def _close(got, ref):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= LOSS_RTOL * np.abs(ref) + 1e-5)


def _run(H, W, cand, slot):
    T = H.shape[0]
    loss = torch.full((T,), float("nan"), device="cuda")
    lse = torch.full((T,), float("nan"), device="cuda")
    ss.forward_noalloc(H, W, cand, slot, loss, lse, check_status=True)
    torch.cuda.synchronize()
    return loss, lse


def test_noalloc_forward_matches_forward_calls_in_a_row(orc):
    big = _batch(1000, 8000, 768, 2000, 5, orc)
    small = _batch(300, 3000, 768, 517, 4, orc)
    # 1: the larger batch fills more of the shared array
    H, W, cand, slot, ref_loss, ref_lse = big
    loss, lse = _run(H, W, cand, slot)
    _close(loss, ref_loss)
    _close(lse, ref_lse)
    # 2: an out-of-range candidate id: the error comes back through status_host
    H, W, cand, slot, _, _ = small
    bad = cand.clone()
    bad[7] = W.shape[0] + 11
    with pytest.raises(ss.SSError) as e:
        _run(H, W, bad, slot)
    assert e.value.name == "SS_ERR_INDEX"
    # 3, 4: the smaller valid batch, twice: SS_OK again, and the same values
    H, W, cand, slot, ref_loss, ref_lse = small
    for _ in range(2):
        loss, lse = _run(H, W, cand, slot)
        _close(loss, ref_loss)
        _close(lse, ref_lse)


def test_noalloc_forward_rejects_sizes_beyond_its_scratch():
    T, V, C, D = 65536, 50304, 24576, 768  # needs far more than the fixed array
    L = ss.lib()
    p = ctypes.c_void_p
    fake = p(0x7F0000000000)
    code = L.ss_forward_noalloc(fake, fake, fake, fake, T, V, C, D, fake, fake, None, None)
    assert code == 2  # SS_ERR_UNSUPPORTED
    assert b"needs" in L.ss_last_error()
