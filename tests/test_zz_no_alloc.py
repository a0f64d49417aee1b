"""The allocation-free forward entry point, ss_forward_noalloc.

Some callers cannot allocate device memory: a plugin inside a host program
that owns and has planned all device memory gets only its input and output
buffers, and some latency-critical paths cannot afford a cudaMalloc, which may
synchronise the device. They cannot provide the workspace that ss_forward
needs, so ss_forward_noalloc keeps its scratch in a fixed array inside the
library's device data instead.

These tests call it through the C ABI and check its loss and lse against the
ordinary ss_forward, within the tolerance the other parity tests use, on two
calls in a row with different batch sizes (the shared array keeps the first
call's contents, so the second call must not depend on them), plus its size
limit. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import LOSS_RTOL, to_dev_bf16

import sampled_softmax_output_gb300 as ss  # noqa: E402  (fails loudly if libss.so is missing)

pytestmark = pytest.mark.gpu


def _batch(T, V, D, C, seed):
    x = synth.make_inputs(T, V, D, 1.1, seed)
    C = max(C, len(np.unique(x["targets"])))
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    targets = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    cand, slot = ss.build_candidates(targets, V, C, seed, ws)
    ref_loss, ref_lse = ss.forward(H, W, cand, slot, ws)
    return H, W, cand, slot, ref_loss, ref_lse


def _close(got, ref):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= LOSS_RTOL * np.abs(ref) + 1e-5)


def test_noalloc_forward_matches_forward_two_calls():
    cases = [(300, 3000, 768, 517, 4), (1000, 8000, 768, 2000, 5)]
    for T, V, D, C, seed in cases:  # two calls in a row on the shared array
        H, W, cand, slot, ref_loss, ref_lse = _batch(T, V, D, C, seed)
        loss = torch.full((T,), float("nan"), device="cuda")
        lse = torch.full((T,), float("nan"), device="cuda")
        ss.forward_noalloc(H, W, cand, slot, loss, lse, check_status=True)
        torch.cuda.synchronize()
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
