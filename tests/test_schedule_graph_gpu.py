"""The step driver of the pages' training loop, on the GPU, against the oracle.

- the candidate schedule (10,240 / 14,336 / 24,576 candidates, then all rows
  for the final 87 steps: "NanoGPT Training Record: Technical Optimizations &
  Speed", "Key Optimizations and Ablation Table Results");
- lm_head gradients accumulated over windows of 2 steps ("KellerJordan/
  modded-nanogpt" README, technique list), with the rows a window wrote
  cleared before the next window (ss_clear_rows);
- each step replayed from a CUDA graph of ss_step (ss_step_graph_*; the same
  record page: training-step graph capture), one graph per candidate count,
  the seed patched per launch.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import GRAD_RTOL, assert_loss_close, rel_fro, to_dev_bf16

import sampled_softmax_output_gb300 as ss  # noqa: E402

pytestmark = pytest.mark.gpu


def test_graph_replay_equals_direct_step(orc):
    """Replays with new seeds and new input contents give the bits of ss_step."""
    T, V, D, C = 700, 6000, 768, 1500
    x1 = synth.make_inputs(T, V, D, 1.1, 31)
    x2 = synth.make_inputs(T, V, D, 1.1, 32)
    C = max(C, len(np.unique(x1["targets"])), len(np.unique(x2["targets"])))
    H = to_dev_bf16(x1["H"])
    W = to_dev_bf16(x1["W"])
    tg = torch.from_numpy(x1["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    g = ss.StepGraph(H, W, tg, C, ws, scale=0.25)
    ws2 = ss.workspace(T, V, C, D)
    for x, seed in ((x1, 5), (x2, 9), (x2, 5)):
        H.copy_(to_dev_bf16(x["H"]))
        tg.copy_(torch.from_numpy(x["targets"]).cuda())
        g.dW.zero_()  # rows outside this step's candidates keep what they held
        got = g.launch(seed)
        ref = ss.step(H, W, tg, C, seed, ws2, scale=0.25)
        torch.cuda.synchronize()
        assert ss.read_status(ws)[0] == 0
        for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
            assert torch.equal(got[k], ref[k]), (seed, k)
    # and the oracle agrees with the last replay
    cand_ref, slot_ref, _ = orc.build_candidates(x2["targets"], V, C, 5)
    np.testing.assert_array_equal(got["cand"].cpu().numpy(), cand_ref)
    l_ref, _ = orc.forward(x2["H"], x1["W"], cand_ref, slot_ref)
    assert_loss_close(got["loss"].cpu().numpy(), l_ref)
    g.close()


def test_schedule_accumulation_windows_from_graphs(orc):
    """Steps 0..4 of a 91-step schedule (C = 10240, 10240, 14336, 24576, 50304)
    in accumulation windows (0, 1), (2, 3), (4): per-step loss and, at each
    window's end, the accumulated dW rows against the oracle's sum; clearing a
    window's rows leaves dW all zero."""
    T, V, D, total = 512, 50304, 768, 91
    Cs = [ss.schedule_candidates(s, total, V) for s in range(5)]
    assert Cs == [10240, 10240, 14336, 24576, 50304]
    W_bits = synth.make_inputs(1, V, D, 1.1, 40)["W"]
    W = to_dev_bf16(W_bits)
    H = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    tg = torch.empty(T, dtype=torch.int32, device="cuda")
    dW = torch.zeros(V, D, dtype=torch.float32, device="cuda")
    ws = ss.workspace(T, V, V, D)  # the largest C of the schedule
    graphs = {}  # one graph per candidate count, all accumulating into dW
    window, scale = [], 1.0 / T
    for step, C in enumerate(Cs):
        x = synth.make_inputs(T, V, D, 1.1, 100 + step)
        x["W"] = W_bits
        H.copy_(to_dev_bf16(x["H"]))
        tg.copy_(torch.from_numpy(x["targets"]).cuda())
        if C not in graphs:
            graphs[C] = ss.StepGraph(H, W, tg, C, ws, scale=scale, accumulate=True, dW=dW)
        seed = 1000 + step
        out = graphs[C].launch(seed)
        torch.cuda.synchronize()
        assert ss.read_status(ws)[0] == 0
        cand_ref, slot_ref, _ = orc.build_candidates(x["targets"], V, C, seed)
        np.testing.assert_array_equal(out["cand"].cpu().numpy(), cand_ref)
        np.testing.assert_array_equal(out["slot"].cpu().numpy(), slot_ref)
        l_ref, lse_ref = orc.forward(x["H"], W_bits, cand_ref, slot_ref)
        assert_loss_close(out["loss"].cpu().numpy(), l_ref)
        window.append((x, cand_ref, slot_ref, lse_ref, out["cand"].clone()))
        if step % 2 == 1 or step == len(Cs) - 1:  # window end: check, then clear its rows
            rng = np.random.default_rng(step)
            touched = np.unique(np.concatenate([w[1] for w in window]))
            rows = np.unique(np.concatenate([rng.choice(touched, 48, replace=False),
                                             rng.integers(0, V, 16)]))
            expect = np.zeros((rows.size, D))
            for xs, cr, sr, lr, _ in window:
                pos = {int(v): j for j, v in enumerate(cr)}
                hit = [i for i, v in enumerate(rows) if int(v) in pos]
                if hit:
                    cols = np.array([pos[int(rows[i])] for i in hit])
                    expect[hit] += orc.backward_dWc(xs["H"], W_bits, cr, sr, lr, scale, cols=cols)
            got = dW[torch.from_numpy(rows).cuda()].cpu().numpy()
            assert rel_fro(got, expect) < GRAD_RTOL
            outside = np.setdiff1d(rows, touched)
            assert np.all(got[np.isin(rows, outside)] == 0)
            for *_, cand_dev in window:
                ss.clear_rows(cand_dev, dW, ws)
            torch.cuda.synchronize()
            assert ss.read_status(ws)[0] == 0
            assert torch.count_nonzero(dW).item() == 0
            window = []
    for g in graphs.values():
        g.close()
