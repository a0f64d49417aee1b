"""Several weighted targets per token over one set of logits, on the GPU,
against the oracle ("KellerJordan/modded-nanogpt" README, technique list:
multi-token prediction and a prefix-token prediction auxiliary loss).

Token t has K targets (k-major [K, T]) with weights w[k]; the candidate set
covers all K*T targets; loss[t] = sum_k w[k] (lse[t] - z[t, slot[k, t]]) and
G = scale (W P - sum_k w[k] Y_k) (times dz/ds with the capped head).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import GRAD_RTOL, assert_loss_close, rel_fro, to_dev_bf16

import sampled_softmax_output_gb300 as ss  # noqa: E402

pytestmark = pytest.mark.gpu


def _mtp_inputs(T, V, D, K, seed, w_std=0.02):
    x = synth.make_inputs(T, V, D, 1.1, seed, w_std=w_std)
    # targets of offsets 1..K: the next tokens of one Zipf stream
    stream = synth.zipf_targets(np.random.default_rng(seed + 1000), T + K, V, 1.1)
    tg = np.stack([stream[k:k + T] for k in range(K)]).astype(np.int32)
    return x, tg


def _run(x, tg, weights, C, seed, scale, cap=0.0, tau=1.0):
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    T, D = H.shape
    V = W.shape[0]
    ws = ss.workspace(T, V, C, D)
    out = ss.step_mtp(H, W, torch.from_numpy(tg).cuda(), weights, C, seed, ws, scale=scale,
                      cap=cap, tau=tau)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    return {k: (v.float() if v.dtype == torch.bfloat16 else v).cpu().numpy() for k, v in out.items()}


CASES = [
    # T, V, D, C, K, weights, seed, scale, cap, tau
    (300, 3000, 768, 700, 2, [1.0, 0.5], 1, 1.0, 0.0, 1.0),
    (257, 2000, 192, 1200, 3, [1.0, 0.3, 0.2], 2, 0.5, 0.0, 1.0),
    (100, 1500, 128, 1500, 8, [1.0, 0.5, 0.25, 0.125, 0.1, 0.1, 0.05, 0.05], 3, 1.0, 0.0, 1.0),
    (300, 3000, 768, 700, 2, [0.7, 0.3], 4, 1.0, 30.0, 7.5),
    (7, 300, 64, 40, 2, [1.0, 1.0], 5, 1.0, 0.0, 1.0),
]


@pytest.mark.parametrize("T,V,D,C,K,weights,seed,scale,cap,tau", CASES)
def test_several_targets_parity(orc, T, V, D, C, K, weights, seed, scale, cap, tau):
    x, tg = _mtp_inputs(T, V, D, K, seed)
    C = max(C, len(np.unique(tg)))
    ref = orc.loss_and_grads_mtp(x["H"], x["W"], tg, weights, C, seed, scale, cap=cap, tau=tau)
    got = _run(x, tg, weights, C, seed, scale, cap, tau)
    np.testing.assert_array_equal(got["cand"], ref["cand"])
    np.testing.assert_array_equal(got["slot"], ref["slot"])
    assert_loss_close(got["loss"], ref["loss"])
    assert_loss_close(got["lse"], ref["lse"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL


def test_one_target_equals_the_single_target_step():
    T, V, D, C, seed = 500, 4000, 768, 1000, 6
    x, tg = _mtp_inputs(T, V, D, 1, seed)
    C = max(C, len(np.unique(tg)))
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    t1 = torch.from_numpy(tg).cuda()
    a = ss.step_mtp(H, W, t1, [1.0], C, seed, ss.workspace(T, V, C, D), scale=0.5)
    b = ss.step(H, W, t1[0].contiguous(), C, seed, ss.workspace(T, V, C, D), scale=0.5)
    torch.cuda.synchronize()
    assert torch.equal(a["slot"][0], b["slot"])
    for k in ("cand", "loss", "lse", "dH", "dW"):
        assert torch.equal(a[k], b[k]), k


def test_repeated_target_rows_add_their_weights(orc):
    T, V, D, C, seed = 300, 3000, 256, 700, 7
    x, tg = _mtp_inputs(T, V, D, 1, seed)
    C = max(C, len(np.unique(tg)))
    two = np.concatenate([tg, tg])
    got = _run(x, two, [0.25, 0.5], C, seed, 1.0)
    ref = orc.loss_and_grads_mtp(x["H"], x["W"], tg, [0.75], C, seed)
    assert_loss_close(got["loss"], ref["loss"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL


def test_several_targets_full_size(orc):
    """T16384_C10240 with targets at offsets 1 and 2 (weights 1, 0.5): cand and
    slot bit-exact; sampled token rows of loss, lse and dH against the oracle;
    <dW_c, W_c> = <dH, H>."""
    w = synth.WORKLOADS[2]
    x = synth.workload_inputs(w)
    stream = np.concatenate([x["targets"],
                             synth.zipf_targets(np.random.default_rng(9), 1, w.V, 1.1)])
    tg = np.stack([stream[:w.T], stream[1:w.T + 1]]).astype(np.int32)
    weights, scale = [1.0, 0.5], 1.0 / w.T
    C = max(w.C, len(np.unique(tg)))
    got = _run(x, tg, weights, C, w.seed, scale)
    cand_ref, slot_flat, _ = orc.build_candidates(tg.reshape(-1), w.V, C, w.seed)
    slot_ref = slot_flat.reshape(tg.shape)
    np.testing.assert_array_equal(got["cand"], cand_ref)
    np.testing.assert_array_equal(got["slot"], slot_ref)
    rng = np.random.default_rng(10)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.integers(0, w.T, 40)]))
    l_ref, s_ref = orc.forward_mtp(x["H"], x["W"], cand_ref, slot_ref, weights, rows=rows)
    assert_loss_close(got["loss"][rows], l_ref)
    assert_loss_close(got["lse"][rows], s_ref)
    dH_ref = orc.backward_dH_mtp(x["H"], x["W"], cand_ref, slot_ref, weights, s_ref, scale,
                                 rows=rows)
    assert rel_fro(got["dH"][rows], dH_ref) < GRAD_RTOL
    dWc = got["dW"][cand_ref].astype(np.float64)
    W64 = synth.bf16_bits_to_f32(x["W"]).astype(np.float64)
    H64 = synth.bf16_bits_to_f32(x["H"]).astype(np.float64)
    lhs = float((dWc * W64[cand_ref]).sum())
    rhs = float((got["dH"].astype(np.float64) * H64).sum())
    assert abs(lhs - rhs) <= 0.02 * abs(rhs)


@pytest.mark.parametrize("cap,tau", [(0.0, 1.0), (30.0, 7.5)])
def test_several_targets_graph_replay_equals_step(cap, tau):
    """ss_step_graph_create_mtp: replays with new seeds give the bits of
    ss_step_mtp."""
    T, V, D, C = 500, 4000, 768, 1200
    x, tg = _mtp_inputs(T, V, D, 2, 12)
    C = max(C, len(np.unique(tg)))
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    t = torch.from_numpy(tg).cuda()
    weights = [1.0, 0.5]
    ws = ss.workspace(T, V, C, D)
    g = ss.StepGraph(H, W, t, C, ws, scale=0.5, weights=weights, cap=cap, tau=tau)
    ws2 = ss.workspace(T, V, C, D)
    for seed in (3, 8):
        g.dW.zero_()
        got = g.launch(seed)
        ref = ss.step_mtp(H, W, t, weights, C, seed, ws2, scale=0.5, cap=cap, tau=tau)
        torch.cuda.synchronize()
        assert ss.read_status(ws)[0] == 0
        for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
            assert torch.equal(got[k], ref[k]), (seed, k)
    g.close()
