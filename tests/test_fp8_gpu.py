"""The FP8 head on the GPU, against the oracle ("KellerJordan/modded-nanogpt"
README, technique list: FP8 for the head).

H and the candidate rows W_c are each scaled by 2^e (e the largest integer
with max|x| 2^e <= 448), rounded to e4m3 and used in that form by both logit
GEMMs (tcgen05 kind::f8f6f4). fp8 = 1: the gradient GEMMs use the same rounded
operands in bf16, and the oracle is the plain definition on the rounded
operands. fp8 = 2 (FP8 through the backward pass, the record page): G is
scaled by 2^15 and rounded to e5m2, and the gradient GEMMs run on e5m2 x e4m3;
the oracle rounds G the same way.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import GRAD_RTOL, assert_loss_close, rel_fro, to_dev_bf16

import sampled_softmax_output_gb300 as ss  # noqa: E402

pytestmark = pytest.mark.gpu


def test_quantizer_bit_exact(orc):
    """ss_quantize_e4m3: the e4m3 codes equal torch's float8_e4m3fn conversion
    of x * 2^e, the rounded values equal the oracle's, bit for bit (values
    spread over many binades, exact grid points and midpoints among them)."""
    rng = np.random.default_rng(30)
    x = (rng.standard_normal(1 << 16) * np.exp2(rng.uniform(-8, 8, 1 << 16))).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    bits[:8] = synth.f32_to_bf16_bits(np.array([0, -0.0, 1.0, 1.0625, 232.0, 2**-9, 3.0, -448.0],
                                               np.float32))
    ws = ss.workspace(256, 1000, 256, 128)
    q, xq = ss.quantize_e4m3(to_dev_bf16(bits), ws)
    torch.cuda.synchronize()
    ref_bits, e = orc.quantize_e4m3(bits)
    np.testing.assert_array_equal(xq.view(torch.int16).cpu().numpy().view(np.uint16), ref_bits)
    scaled = torch.from_numpy(synth.bf16_bits_to_f32(bits) * np.float32(2.0 ** e))
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q.cpu().numpy(), codes)


CASES = [
    # T, V, D, C, seed, scale
    (300, 3000, 768, 517, 1, 1.0),     # ragged T and C tails
    (257, 2000, 128, 1000, 2, 0.5),    # one k-block of 128
    (500, 1000, 256, 1000, 3, 1.0 / 500),  # C = V
    (1, 64, 128, 1, 4, 1.0),           # a single candidate
]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("T,V,D,C,seed,scale", CASES)
def test_fp8_head_parity(orc, T, V, D, C, seed, scale, mode):
    x = synth.make_inputs(T, V, D, 1.1, seed)
    C = max(C, len(np.unique(x["targets"])))
    ref = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, seed, scale, grads=mode == 2)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    got = ss.step(H, W, tg, C, seed, ws, scale=scale, fp8=mode)
    sep = ss.step_separate(H, W, tg, C, seed, ss.workspace(T, V, C, D), scale=scale, fp8=mode)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
        assert torch.equal(got[k], sep[k]), k
    np.testing.assert_array_equal(got["cand"].cpu().numpy(), ref["cand"])
    assert_loss_close(got["loss"].cpu().numpy(), ref["loss"])
    assert_loss_close(got["lse"].cpu().numpy(), ref["lse"])
    assert rel_fro(got["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"].cpu().numpy(), ref["dW"]) < GRAD_RTOL
    if C > 1:  # and it is not the bf16 head
        plain = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, seed, scale)
        assert np.abs(plain["loss"] - ref["loss"]).max() > 1e-4


def test_fp8_gradients_accumulate_and_scale_sign(orc):
    """FP8 gradients with accumulate = 1 into a non-zero dW and a negative
    scale: dW rows += the oracle's e5m2-gradient rows, other rows untouched."""
    T, V, D, C, seed, scale = 300, 3000, 256, 700, 8, -0.25
    x = synth.make_inputs(T, V, D, 1.1, seed)
    C = max(C, len(np.unique(x["targets"])))
    dW0 = np.random.default_rng(9).standard_normal((V, D)).astype(np.float32)
    ref = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, seed, scale, dW_init=dW0,
                                 accumulate=True, grads=True)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    dW = torch.from_numpy(dW0).cuda()
    ws = ss.workspace(T, V, C, D)
    got = ss.step(H, W, tg, C, seed, ws, scale=scale, fp8=2, accumulate=True, dW=dW)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    other = np.setdiff1d(np.arange(V), ref["cand"])
    np.testing.assert_array_equal(got["dW"].cpu().numpy()[other], dW0[other])
    assert rel_fro(got["dW"].cpu().numpy()[ref["cand"]] - dW0[ref["cand"]], ref["dWc"]) < GRAD_RTOL
    assert rel_fro(got["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL


@pytest.mark.parametrize("mode", [1, 2])
def test_fp8_head_full_size(orc, mode):
    """T16384_C10240 with the FP8 head: cand bit-exact, sampled token rows of
    loss, lse and dH, and exact candidate rows of dW, against the oracle."""
    w = synth.WORKLOADS[2]
    x = synth.workload_inputs(w)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(w.T, w.V, w.C, w.D)
    scale = 1.0 / w.T
    got = ss.step(H, W, tg, w.C, w.seed, ws, scale=scale, fp8=mode)
    got = {k: v.clone() for k, v in got.items()}
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    # ss_step makes H's e4m3 codes beside the candidate build (several tiles
    # per block at this size); the separate calls make them after the gather
    sep = ss.step_separate(H, W, tg, w.C, w.seed, ws, scale=scale, fp8=mode)
    torch.cuda.synchronize()
    for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
        assert torch.equal(got[k], sep[k]), k
    del sep
    cand, slot, _ = orc.build_candidates(x["targets"], w.V, w.C, w.seed)
    np.testing.assert_array_equal(got["cand"].cpu().numpy(), cand)
    Hq, Wq, _, _ = orc.fp8_inputs(x["H"], x["W"], cand)
    rng = np.random.default_rng(31)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.integers(0, w.T, 40)]))
    l_ref, s_ref = orc.forward(Hq, Wq, cand, slot, rows=rows)
    assert_loss_close(got["loss"].cpu().numpy()[rows], l_ref)
    assert_loss_close(got["lse"].cpu().numpy()[rows], s_ref)
    dH_fn = orc.backward_dH_g8 if mode == 2 else orc.backward_dH
    dH_ref = dH_fn(Hq, Wq, cand, slot, s_ref, scale, rows=rows)
    assert rel_fro(got["dH"].float().cpu().numpy()[rows], dH_ref) < GRAD_RTOL
    _, lse_all = orc.forward(Hq, Wq, cand, slot)
    cols = np.array([0, 1, w.C // 2, w.C - 1])
    dW_fn = orc.backward_dWc_g8 if mode == 2 else orc.backward_dWc
    ref_rows = dW_fn(Hq, Wq, cand, slot, lse_all, scale, cols=cols)
    assert rel_fro(got["dW"].cpu().numpy()[cand[cols]], ref_rows) < GRAD_RTOL


@pytest.mark.parametrize("mode", [1, 2])
def test_fp8_graph_replay_equals_direct_step(mode):
    """A captured FP8 step replayed with new seeds gives the bits of ss_step."""
    T, V, D, C = 700, 6000, 768, 1500
    x = synth.make_inputs(T, V, D, 1.1, 41)
    C = max(C, len(np.unique(x["targets"])))
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    g = ss.StepGraph(H, W, tg, C, ws, scale=0.25, fp8=mode)
    ws2 = ss.workspace(T, V, C, D)
    for seed in (5, 9):
        g.dW.zero_()
        got = g.launch(seed)
        ref = ss.step(H, W, tg, C, seed, ws2, scale=0.25, fp8=mode)
        torch.cuda.synchronize()
        assert ss.read_status(ws)[0] == 0
        for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
            assert torch.equal(got[k], ref[k]), (seed, k)
    g.close()


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("cap,tau", [(30.0, 7.5), (6.0, 0.7)])
def test_capped_fp8_head_parity(orc, mode, cap, tau):
    """The pages' head, FP8 and soft-capped: z = cap / (1 + exp(-s / tau)) of
    the e4m3 logits, and (mode 2) G8 = e5m2(2^e (P - Y) dz/ds), e from the
    bound cap / (4 tau), against the oracle of the same head."""
    T, V, D, C, seed, scale = 300, 3000, 768, 517, 11, 0.5
    x = synth.make_inputs(T, V, D, 1.1, seed)
    C = max(C, len(np.unique(x["targets"])))
    ref = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, seed, scale, grads=mode == 2,
                                 cap=cap, tau=tau)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    got = ss.step(H, W, tg, C, seed, ws, scale=scale, fp8=mode, cap=cap, tau=tau)
    sep = ss.step_separate(H, W, tg, C, seed, ss.workspace(T, V, C, D), scale=scale, fp8=mode,
                           cap=cap, tau=tau)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
        assert torch.equal(got[k], sep[k]), k
    assert_loss_close(got["loss"].cpu().numpy(), ref["loss"])
    assert_loss_close(got["lse"].cpu().numpy(), ref["lse"])
    assert rel_fro(got["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"].cpu().numpy(), ref["dW"]) < GRAD_RTOL
    plain = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, seed, scale, grads=mode == 2)
    assert np.abs(plain["loss"] - ref["loss"]).max() > 1e-3  # and the cap is applied


def test_capped_fp8_gradients_full_size(orc):
    """T16384_C10240 with the capped FP8 head and FP8 gradients (cap 30, tau
    7.5): cand bit-exact, sampled token rows of loss, lse and dH, and exact
    candidate rows of dW, against the oracle."""
    w = synth.WORKLOADS[2]
    cap, tau = 30.0, 7.5
    x = synth.workload_inputs(w)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(w.T, w.V, w.C, w.D)
    scale = 1.0 / w.T
    got = ss.step(H, W, tg, w.C, w.seed, ws, scale=scale, fp8=2, cap=cap, tau=tau)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    cand, slot, _ = orc.build_candidates(x["targets"], w.V, w.C, w.seed)
    np.testing.assert_array_equal(got["cand"].cpu().numpy(), cand)
    Hq, Wq, _, _ = orc.fp8_inputs(x["H"], x["W"], cand)
    rng = np.random.default_rng(32)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.integers(0, w.T, 40)]))
    l_ref, s_ref = orc.forward(Hq, Wq, cand, slot, rows=rows, cap=cap, tau=tau)
    assert_loss_close(got["loss"].cpu().numpy()[rows], l_ref)
    assert_loss_close(got["lse"].cpu().numpy()[rows], s_ref)
    dH_ref = orc.backward_dH_g8(Hq, Wq, cand, slot, s_ref, scale, rows=rows, cap=cap, tau=tau)
    assert rel_fro(got["dH"].float().cpu().numpy()[rows], dH_ref) < GRAD_RTOL
    _, lse_all = orc.forward(Hq, Wq, cand, slot, cap=cap, tau=tau)
    cols = np.array([0, 1, w.C // 2, w.C - 1])
    ref_rows = orc.backward_dWc_g8(Hq, Wq, cand, slot, lse_all, scale, cols=cols, cap=cap, tau=tau)
    assert rel_fro(got["dW"].cpu().numpy()[cand[cols]], ref_rows) < GRAD_RTOL
