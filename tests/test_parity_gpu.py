"""GPU path vs the CPU oracle, through the C ABI.

Both entry-point sequences are checked: the three calls (ss_build_candidates,
ss_forward, ss_backward, whose backward recomputes the logits) and the
one-call ss_step (whose plain head keeps the forward's probabilities for the
backward, with the recompute as its fallback).

* small and ragged sizes (several tiles plus a ragged tail in T, C and D, the
  degenerate cases C = 1, U = C, C = V, T = 1): every output element compared;
* the five full-size workloads, in the launch configuration the benchmark
  times: candidates bit-exact, sampled tokens and candidate rows against the
  oracle computed one by one, and properties that hold at any size;
* device-side error paths and the write-back contract of dW.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import GRAD_RTOL, assert_loss_close, rel_fro, run_gpu, run_gpu_step, to_dev_bf16

pytestmark = pytest.mark.gpu

import sampled_softmax_output_gb300 as ss  # noqa: E402  (fails loudly if libss.so is missing)


def _case(T, V, D, C, seed, s=1.1, w_std=0.02):
    x = synth.make_inputs(T, V, D, s, seed, w_std=w_std)
    U = len(np.unique(x["targets"]))
    return x, max(C, U)


def _full_oracle(orc, x, C, seed, scale=1.0, dW0=None, accumulate=False, cap=0.0, tau=1.0):
    return orc.loss_and_grads(x["H"], x["W"], x["targets"], C, seed, scale, dW_init=dW0,
                              accumulate=accumulate, cap=cap, tau=tau)


SMALL = [
    # T, V, D, C, seed, scale
    (1, 64, 64, 1, 1, 1.0),          # a single candidate: loss = 0
    (7, 300, 64, 37, 2, 1.0),
    (128, 1000, 768, 256, 3, 1.0),   # exactly one tile each way
    (300, 3000, 768, 517, 4, 1.0),   # ragged T and C tails
    (257, 2000, 192, 1000, 5, 0.5),  # D not a multiple of the 256-wide gradient tile
    (500, 1000, 128, 1000, 6, 1.0 / 500),  # C = V: full vocabulary
    (200, 5000, 1024, 130, 7, 1.0),  # U close to C
    (64, 4096, 768, 4096, 8, 1.0),   # C = V, one partial token tile
]


RUNS = {"calls": run_gpu, "step": run_gpu_step}


@pytest.mark.parametrize("path", ["calls", "step"])
@pytest.mark.parametrize("T,V,D,C,seed,scale", SMALL)
def test_small_parity(orc, T, V, D, C, seed, scale, path):
    x, C = _case(T, V, D, C, seed)
    ref = _full_oracle(orc, x, C, seed, scale)
    got = RUNS[path](ss, x, C, seed, scale)
    assert got["status"] == 0
    assert got["U"] == ref["U"]
    np.testing.assert_array_equal(got["cand"], ref["cand"])
    np.testing.assert_array_equal(got["slot"], ref["slot"])
    assert_loss_close(got["loss"], ref["loss"])
    assert_loss_close(got["lse"], ref["lse"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL
    outside = np.setdiff1d(np.arange(V), ref["cand"])
    assert np.all(got["dW"][outside] == 0)


@pytest.mark.parametrize("path", ["calls", "step"])
def test_pair_kernels_ragged(orc, path):
    """A batch large enough that the logit GEMMs run on CTA pairs (more
    256 x 256 tiles than SM pairs) while H and W_c stay in L2, with ragged
    token and candidate tails (the last pair's second CTA holds no valid
    row, the last logit tile 135 valid columns): every output element
    against the oracle."""
    T, V, D, C, seed = 2049, 8000, 128, 4999, 21
    x, C = _case(T, V, D, C, seed)
    assert (T + 255) // 256 * ((C + 255) // 256 - 1) >= 76
    ref = _full_oracle(orc, x, C, seed, 1.0 / T)
    got = RUNS[path](ss, x, C, seed, 1.0 / T)
    assert got["status"] == 0
    np.testing.assert_array_equal(got["cand"], ref["cand"])
    np.testing.assert_array_equal(got["slot"], ref["slot"])
    assert_loss_close(got["loss"], ref["loss"])
    assert_loss_close(got["lse"], ref["lse"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL
    outside = np.setdiff1d(np.arange(V), ref["cand"])
    assert np.all(got["dW"][outside] == 0)


@pytest.mark.parametrize("path", ["calls", "step"])
def test_accumulate_and_untouched_rows(orc, path):
    T, V, D, C, seed = 300, 2500, 256, 700, 11
    x, C = _case(T, V, D, C, seed)
    dW0 = np.random.default_rng(3).standard_normal((V, D)).astype(np.float32)
    for acc in (False, True):
        ref = _full_oracle(orc, x, C, seed, 0.25, dW0=dW0, accumulate=acc)
        got = RUNS[path](ss, x, C, seed, 0.25, dW0=dW0, accumulate=acc)
        assert got["status"] == 0
        outside = np.setdiff1d(np.arange(V), ref["cand"])
        np.testing.assert_array_equal(got["dW"][outside], dW0[outside])
        c = ref["cand"]
        assert rel_fro(got["dW"][c] - (dW0[c] if acc else 0), ref["dW"][c] - (dW0[c] if acc else 0)) < GRAD_RTOL


def test_workspace_reused_across_shapes(orc):
    """One workspace serves problems of other shapes one after another (one
    logit tile per row, many, a ragged token tail), each matching the oracle."""
    cases = [(900, 4000, 256, 2000, 11), (129, 4000, 256, 200, 12), (900, 4000, 256, 2000, 13),
             (300, 4000, 256, 517, 14)]
    ws = ss.workspace(1000, 4000, 2100, 256)
    for T, V, D, C, seed in cases:
        x, C = _case(T, V, D, C, seed)
        ref = _full_oracle(orc, x, C, seed)
        got = run_gpu(ss, x, C, seed, ws=ws)
        assert got["status"] == 0
        assert_loss_close(got["loss"], ref["loss"])
        assert_loss_close(got["lse"], ref["lse"])
        assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
        assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL


def test_repeated_calls_are_deterministic(orc):
    T, V, D, C, seed = 400, 3000, 768, 1200, 12
    x, C = _case(T, V, D, C, seed)
    ws = ss.workspace(T, V, C, D)
    a = run_gpu(ss, x, C, seed, ws=ws)
    b = run_gpu(ss, x, C, seed, ws=ws)
    for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_uniform_logits_ln_C(orc):
    # H = 0: every logit is 0, loss = ln C for every token
    T, V, D, C = 300, 5000, 768, 2500
    x, C = _case(T, V, D, C, 13)
    x["H"] = np.zeros_like(x["H"])
    got = run_gpu(ss, x, C, 13)
    np.testing.assert_allclose(got["loss"], np.log(C), rtol=1e-6)


# ------------------------------------------------------------- full sizes

def _check_sampled(orc, x, T, V, D, C, seed, rng_seed, exact_cols, cap=0.0, tau=1.0):
    """The whole path on one batch: candidates bit-exact, sampled token rows of
    loss/lse/dH against the oracle, dW rows outside the candidate set
    untouched, two identities of the gradients, and (exact_cols) some dW
    candidate rows and the whole lse against the oracle."""
    cand_ref, slot_ref, U_ref = orc.build_candidates(x["targets"], V, C, seed)
    H = to_dev_bf16(x["H"])
    W = to_dev_bf16(x["W"])
    targets = torch.from_numpy(x["targets"]).cuda()
    ws = ss.workspace(T, V, C, D)
    cand, slot, U = ss.build_candidates(targets, V, C, seed, ws, return_U=True)
    assert U == U_ref
    np.testing.assert_array_equal(cand.cpu().numpy(), cand_ref)
    np.testing.assert_array_equal(slot.cpu().numpy(), slot_ref)
    loss, lse = ss.forward(H, W, cand, slot, ws, cap=cap, tau=tau)
    canary = 7.0
    dW = torch.full((V, D), canary, dtype=torch.float32, device="cuda")
    scale = 1.0 / T
    dH, dW = ss.backward(H, W, cand, slot, lse, ws, scale=scale, dW=dW, cap=cap, tau=tau)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    loss, lse = loss.cpu().numpy(), lse.cpu().numpy()
    dH = dH.float().cpu().numpy()
    dW = dW.cpu().numpy()
    # sampled tokens, including both ends and the last partial tile
    rng = np.random.default_rng(rng_seed)
    rows = np.unique(np.concatenate([[0, T - 1, (T // 128) * 128 - 1, (T // 256) * 256],
                                     rng.integers(0, T, 45)]))
    rows = rows[(rows >= 0) & (rows < T)]
    l_ref, s_ref = orc.forward(x["H"], x["W"], cand_ref, slot_ref, rows=rows, cap=cap, tau=tau)
    assert_loss_close(loss[rows], l_ref)
    assert_loss_close(lse[rows], s_ref)
    dH_ref = orc.backward_dH(x["H"], x["W"], cand_ref, slot_ref, s_ref, scale, rows=rows, cap=cap,
                             tau=tau)
    assert rel_fro(dH[rows], dH_ref) < GRAD_RTOL
    # rows of dW outside the candidate set keep the canary bit for bit
    outside = np.setdiff1d(np.arange(V), cand_ref)
    assert outside.size == V - C
    assert np.all(dW[outside] == canary)
    dWc = dW[cand_ref].astype(np.float64)
    # rows of P - Y sum to zero, so the candidate-row gradients sum to zero
    # (not with a capped head: G carries the per-logit factor dz/ds)
    if cap == 0:
        assert np.linalg.norm(dWc.sum(0)) <= 0.02 * np.linalg.norm(dWc)
    # <dW_c, W_c> = sum_tj G_tj S_tj = <dH, H>
    W64 = synth.bf16_bits_to_f32(x["W"]).astype(np.float64)
    H64 = synth.bf16_bits_to_f32(x["H"]).astype(np.float64)
    lhs = float((dWc * W64[cand_ref]).sum())
    rhs = float((dH.astype(np.float64) * H64).sum())
    assert abs(lhs - rhs) <= 0.02 * abs(rhs)
    # the one-call entry point on the same batch: bit-exact candidates, and
    # the same oracle checks (with the plain head its backward reads the
    # forward's stored probabilities instead of recomputing the logits)
    fused = ss.step(H, W, targets, C, seed, ws, scale=scale, cap=cap, tau=tau,
                    dW=torch.full((V, D), canary, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    np.testing.assert_array_equal(fused["cand"].cpu().numpy(), cand_ref)
    np.testing.assert_array_equal(fused["slot"].cpu().numpy(), slot_ref)
    f_loss, f_lse = fused["loss"].cpu().numpy(), fused["lse"].cpu().numpy()
    f_dH = fused["dH"].float().cpu().numpy()
    f_dW = fused["dW"].cpu().numpy()
    del fused
    assert_loss_close(f_loss[rows], l_ref)
    assert_loss_close(f_lse[rows], s_ref)
    assert rel_fro(f_dH[rows], dH_ref) < GRAD_RTOL
    assert np.all(f_dW[outside] == canary)
    # and it agrees with the three calls over every token and candidate row
    assert_loss_close(f_loss, loss)
    assert rel_fro(f_dH, dH) < GRAD_RTOL
    assert rel_fro(f_dW[cand_ref], dWc) < GRAD_RTOL
    del f_dH
    if exact_cols:
        _, lse_all = orc.forward(x["H"], x["W"], cand_ref, slot_ref, cap=cap, tau=tau)
        cols = np.unique(np.array([0, U_ref - 1, min(U_ref, C - 1), C - 1, C // 2, 1,
                                   (C // 256) * 256]))
        cols = cols[cols < C]
        ref_rows = orc.backward_dWc(x["H"], x["W"], cand_ref, slot_ref, lse_all, scale, cols=cols,
                                    cap=cap, tau=tau)
        assert rel_fro(dW[cand_ref[cols]], ref_rows) < GRAD_RTOL
        assert rel_fro(f_dW[cand_ref[cols]], ref_rows) < GRAD_RTOL
        assert_loss_close(lse, lse_all)
        assert_loss_close(f_lse, lse_all)
    return {"lse": lse, "loss": loss, "dW": dW, "f_lse": f_lse, "f_loss": f_loss, "f_dW": f_dW,
            "cand": cand_ref, "U": U_ref}


def _golden_dw(name):
    """The stored oracle values of a large workload (tests/golden/, written by
    tests/golden/make_full_size_dw.py from the CPU oracle alone)."""
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "make_full_size_dw.py")
    spec = importlib.util.spec_from_file_location("_golden_dw", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.read(name)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_full_size_workload(orc, wid):
    w = synth.WORKLOADS[wid]
    x = synth.workload_inputs(w)
    # exact candidate rows computed here where the oracle's full-batch lse is
    # affordable; for the three large workloads, stored oracle rows instead
    small = w.T * w.C <= 16384 * 10240
    got = _check_sampled(orc, x, w.T, w.V, w.D, w.C, w.seed, 100 + wid, exact_cols=small)
    if small:
        return
    g = _golden_dw(w.name)
    meta = g["meta"]
    assert int(meta["T"][0]) == w.T and int(meta["C"][0]) == w.C and int(meta["seed"][0]) == w.seed
    assert int(meta["U"][0]) == got["U"]
    cols = g["cols"]
    np.testing.assert_array_equal(got["cand"][cols], [int(c) for c in meta["cand_of_columns"]])
    # candidate rows of dW (both entry points) against the oracle's, and the
    # mean loss and lse over every token
    for dW in (got["dW"], got["f_dW"]):
        assert rel_fro(dW[got["cand"][cols]], g["rows"]) < GRAD_RTOL
    for loss, lse in ((got["loss"], got["lse"]), (got["f_loss"], got["f_lse"])):
        ml, ms = float(np.mean(loss.astype(np.float64))), float(np.mean(lse.astype(np.float64)))
        assert abs(ml - float(meta["mean_loss"][0])) <= 1e-4 * abs(float(meta["mean_loss"][0]))
        assert abs(ms - float(meta["mean_lse"][0])) <= 1e-4 * abs(float(meta["mean_lse"][0]))


def test_operands_beyond_l2_ragged(orc):
    """H and W_c together above 96 MB (bf16): the softmax-gradient GEMM runs on CTA pairs
    and the gradient GEMMs in two launches. Ragged T (not a multiple of the
    256-row pair tile) and C."""
    T, V, D, C, seed = 9001, 20000, 4096, 4001, 21
    assert (T + C) * D * 2 > 96 * 2**20
    x, C = _case(T, V, D, C, seed)
    _check_sampled(orc, x, T, V, D, C, seed, 7, exact_cols=True)


def test_step_accumulate_beyond_l2():
    """ss_step with accumulate = 1 where H and W_c exceed L2 (the forward on
    CTA pairs, dH and dW_c as two launches, dW_c not waiting for dH): every
    candidate row of dW is the previous row plus what the non-accumulating
    step writes (to an ulp), and every other row is untouched."""
    T, V, D, C, seed = 20001, 30000, 2048, 12001, 33
    assert (T + C) * D * 2 > 96 * 2**20
    x, C = _case(T, V, D, C, seed)
    H, W, tg = to_dev_bf16(x["H"]), to_dev_bf16(x["W"]), _dev(x["targets"])
    ws = ss.workspace(T, V, C, D)
    dW0 = torch.from_numpy(np.random.default_rng(5).standard_normal((V, D)).astype(np.float32)).cuda()
    plain = ss.step(H, W, tg, C, seed, ws, scale=1.0 / T, dW=torch.zeros_like(dW0))
    plain = {k: v.clone() for k, v in plain.items()}
    acc = ss.step(H, W, tg, C, seed, ws, scale=1.0 / T, dW=dW0.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    c = plain["cand"].long()
    assert torch.equal(acc["cand"], plain["cand"])
    # (the epilogue may fuse the scale and the add into one FMA: one rounding
    # instead of two, so allow an ulp of the operands)
    want = dW0[c] + plain["dW"][c]
    tol = 2.0 ** -22 * (dW0[c].abs() + plain["dW"][c].abs()) + 1e-30
    assert torch.all((acc["dW"][c] - want).abs() <= tol)
    outside = torch.ones(V, dtype=torch.bool, device="cuda")
    outside[c] = False
    assert torch.equal(acc["dW"][outside], dW0[outside])
    assert torch.equal(acc["dH"], plain["dH"]) and torch.equal(acc["loss"], plain["loss"])


# ------------------------------------------------------------ error paths

def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_target_out_of_range_is_reported_and_blocks_later_calls():
    T, V, D, C = 100, 1000, 64, 200
    x = synth.make_inputs(T, V, D, 1.1, 1)
    x["targets"][17] = V  # out of range
    ws = ss.workspace(T, V, C, D)
    with pytest.raises(ss.SSError) as e:
        ss.build_candidates(_dev(x["targets"]), V, C, 1, ws, return_U=True)
    assert e.value.name == "SS_ERR_TARGET_RANGE"
    # the sticky status makes the forward a no-op: outputs keep their sentinel
    cand = torch.arange(C, dtype=torch.int32, device="cuda")
    slot = torch.zeros(T, dtype=torch.int32, device="cuda")
    loss = torch.full((T,), -5.0, device="cuda")
    lse = torch.full((T,), -5.0, device="cuda")
    ss.forward(to_dev_bf16(x["H"]), to_dev_bf16(x["W"]), cand, slot, ws, loss=loss, lse=lse)
    assert ss.read_status(ws)[0] == 4
    assert torch.all(loss == -5.0) and torch.all(lse == -5.0)
    # a fresh candidate build clears it
    x["targets"][17] = 3
    ss.build_candidates(_dev(x["targets"]), V, C, 1, ws, return_U=True)
    assert ss.read_status(ws)[0] == 0


def test_capacity_error():
    T, V, D = 50, 1000, 64
    targets = np.arange(T, dtype=np.int32)
    ws = ss.workspace(T, V, 40, D)
    with pytest.raises(ss.SSError) as e:
        ss.build_candidates(_dev(targets), V, 40, 0, ws, return_U=True)
    assert e.value.name == "SS_ERR_CAPACITY"
    assert ss.read_status(ws) == (3, T)


def test_bad_cand_and_slot_are_reported():
    T, V, D, C = 64, 500, 64, 100
    x = synth.make_inputs(T, V, D, 1.1, 2)
    ws = ss.workspace(T, V, C, D)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    cand, slot, U = ss.build_candidates(_dev(x["targets"]), V, C, 2, ws, return_U=True)
    bad = cand.clone()
    bad[5] = V + 3
    ss.forward(H, W, bad, slot, ws)
    assert ss.read_status(ws)[0] == 8
    ss.build_candidates(_dev(x["targets"]), V, C, 2, ws)
    bslot = slot.clone()
    bslot[3] = C
    ss.forward(H, W, cand, bslot, ws)
    assert ss.read_status(ws)[0] == 8


def test_empty_batch():
    V, D, C = 500, 64, 100
    ws = ss.workspace(0, V, C, D)
    targets = torch.empty(0, dtype=torch.int32, device="cuda")
    cand, slot, U = ss.build_candidates(targets, V, C, 5, ws, return_U=True)
    assert U == 0
    c = cand.cpu().numpy()
    assert np.all(np.diff(c) > 0) and c.min() >= 0 and c.max() < V
    H = torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(V, D, device="cuda").to(torch.bfloat16)
    loss, lse = ss.forward(H, W, cand, slot, ws)
    assert loss.numel() == 0
    dW = torch.full((V, D), 3.0, device="cuda")
    ss.backward(H, W, cand, slot, lse, ws, dW=dW)
    torch.cuda.synchronize()
    d = dW.cpu().numpy()
    assert np.all(d[c] == 0)
    assert np.all(d[np.setdiff1d(np.arange(V), c)] == 3.0)


def test_fused_step_against_oracle_and_separate_calls(orc):
    # ss_step (stored probabilities) and the three calls (recompute) on the
    # same batch: identical candidates, both within tolerance of the oracle
    T, V, D, C, seed = 700, 6000, 768, 1500, 21
    x, C = _case(T, V, D, C, seed)
    H, W, tg = to_dev_bf16(x["H"]), to_dev_bf16(x["W"]), _dev(x["targets"])
    ws = ss.workspace(T, V, C, D)
    a = ss.step(H, W, tg, C, seed, ws, scale=0.5)
    a = {k: v.clone() for k, v in a.items()}
    b = ss.step_separate(H, W, tg, C, seed, ws, scale=0.5)
    torch.cuda.synchronize()
    for k in ("cand", "slot"):
        assert torch.equal(a[k], b[k]), k
    ref = _full_oracle(orc, x, C, seed, 0.5)
    for r in (a, b):
        assert_loss_close(r["loss"].cpu().numpy(), ref["loss"])
        assert_loss_close(r["lse"].cpu().numpy(), ref["lse"])
        assert rel_fro(r["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL
        assert rel_fro(r["dW"].cpu().numpy(), ref["dW"]) < GRAD_RTOL


def test_step_is_deterministic():
    T, V, D, C, seed = 900, 5000, 256, 2100, 23
    x, C = _case(T, V, D, C, seed)
    H, W, tg = to_dev_bf16(x["H"]), to_dev_bf16(x["W"]), _dev(x["targets"])
    ws = ss.workspace(T, V, C, D)
    a = {k: v.clone() for k, v in ss.step(H, W, tg, C, seed, ws, scale=0.5).items()}
    b = ss.step(H, W, tg, C, seed, ws, scale=0.5)
    torch.cuda.synchronize()
    for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
        assert torch.equal(a[k], b[k]), k


def _stored_fallback_case(T, V, D, C, seed, far):
    """Inputs on which the first logit tile of every row lies far below the
    row's largest logits: H = 6 u + noise, W rows of the ids in the first tile
    (the smallest targets, all below V / 4) = -far/6 u, every other row
    = +far/6 u plus noise, u a unit vector. Then lse - r is about 2 far."""
    x = synth.make_inputs(T, V, D, 1.1, seed)
    rng = np.random.default_rng(seed + 1)
    u = rng.standard_normal(D)
    u /= np.linalg.norm(u)
    H = 6.0 * u[None, :] + 0.3 * rng.standard_normal((T, D))
    Wf = 0.02 * rng.standard_normal((V, D))
    Wf[: V // 4] -= (far / 6.0) * u
    Wf[V // 4:] += (far / 6.0) * u
    x["H"] = synth.f32_to_bf16_bits(H.astype(np.float32))
    x["W"] = synth.f32_to_bf16_bits(Wf.astype(np.float32))
    x["targets"] = np.minimum(x["targets"], V // 4 - 1).astype(np.int32)
    return x


@pytest.mark.parametrize("far", [5.0, 200.0])
def test_step_stored_several_targets_far_below(orc, far):
    """Two weighted targets per token (weights 1 and 0.5, so G carries their
    sum W = 1.5) on the stored-probability step: with the reference inside
    the stored range (far 5) and beyond it (far 200, the recompute fallback,
    whose G is scaled by 1 / W and whose row factors become scale W), every
    element against the oracle."""
    T, V, D, C, seed = 300, 4000, 256, 1700, 32
    x = _stored_fallback_case(T, V, D, C, seed, far)
    tg = np.stack([x["targets"], np.roll(x["targets"], 1)]).astype(np.int32)
    weights = [1.0, 0.5]
    C = max(C, len(np.unique(tg)))
    ref = orc.loss_and_grads_mtp(x["H"], x["W"], tg, weights, C, seed, 1.0 / T)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    ws = ss.workspace(T, V, C, D)
    got = ss.step_mtp(H, W, torch.from_numpy(tg).cuda(), weights, C, seed, ws, scale=1.0 / T)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    np.testing.assert_array_equal(got["cand"].cpu().numpy(), ref["cand"])
    assert_loss_close(got["loss"].cpu().numpy(), ref["loss"])
    assert rel_fro(got["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"].cpu().numpy(), ref["dW"]) < GRAD_RTOL


@pytest.mark.parametrize("far", [5.0, 25.0, 40.0, 200.0])
def test_step_stored_reference_far_below(orc, far):
    """The per-row reference r (largest logit of the first tile) far below the
    row's lse: at 2 far = 10, 50 the stored probabilities stay in bf16's
    range (alpha = exp(r - lse) down to e^-50); at 80 and 400 the merge raises
    the fallback flag (at 400 exp(S - r) overflows) and the backward
    recomputes the logits. Every case matches the oracle."""
    T, V, D, C, seed = 300, 4000, 256, 1700, 31
    x = _stored_fallback_case(T, V, D, C, seed, far)
    C = max(C, len(np.unique(x["targets"])))
    ref = _full_oracle(orc, x, C, seed, 1.0 / T)
    got = run_gpu_step(ss, x, C, seed, 1.0 / T)
    assert got["status"] == 0
    np.testing.assert_array_equal(got["cand"], ref["cand"])
    # the first tile lies below the others: the case does what it says
    assert np.all(ref["cand"][:256] < V // 4) and ref["U"] <= 256
    assert_loss_close(got["loss"], ref["loss"])
    assert_loss_close(got["lse"], ref["lse"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL


def test_step_fallback_beyond_l2(orc):
    """The stored-probability step's fallback where H and W_c exceed L2: the
    gated recompute runs on CTA pairs and resets Hs and the row factors. The
    first logit tile lies ~400 below the rest (exp(S - r) overflows), so the
    fallback must run; the step then matches the three calls (which always
    recompute) over every token and candidate row, and the oracle on sampled
    token rows."""
    T, V, D, C, seed = 20001, 30000, 2048, 12001, 35
    assert (T + C) * D * 2 > 96 * 2**20
    x = _stored_fallback_case(T, V, D, C, seed, 200.0)
    C = max(C, len(np.unique(x["targets"])))
    H, W, tg = to_dev_bf16(x["H"]), to_dev_bf16(x["W"]), _dev(x["targets"])
    ws = ss.workspace(T, V, C, D)
    a = {k: v.clone() for k, v in ss.step(H, W, tg, C, seed, ws, scale=1.0 / T).items()}
    b = ss.step_separate(H, W, tg, C, seed, ws, scale=1.0 / T)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    cand = a["cand"].cpu().numpy()
    assert np.all(cand[:256] < V // 4)
    assert torch.equal(a["cand"], b["cand"]) and torch.equal(a["slot"], b["slot"])
    assert_loss_close(a["loss"].cpu().numpy(), b["loss"].cpu().numpy())
    assert_loss_close(a["lse"].cpu().numpy(), b["lse"].cpu().numpy())
    assert rel_fro(a["dH"].float().cpu().numpy(), b["dH"].float().cpu().numpy()) < GRAD_RTOL
    c = a["cand"].long()
    assert rel_fro(a["dW"][c].cpu().numpy(), b["dW"][c].cpu().numpy()) < GRAD_RTOL
    rows = np.array([0, 1, T // 2, T - 1])
    slot = a["slot"].cpu().numpy()
    l_ref, s_ref = orc.forward(x["H"], x["W"], cand, slot, rows=rows)
    assert_loss_close(a["loss"].cpu().numpy()[rows], l_ref)
    dH_ref = orc.backward_dH(x["H"], x["W"], cand, slot, s_ref, 1.0 / T, rows=rows)
    assert rel_fro(a["dH"].float().cpu().numpy()[rows], dH_ref) < GRAD_RTOL


def test_step_single_target_weight_half_merge_beside_softmax_grad(orc):
    # one target with weight 1/2 (ss_step_mtp) keeps the recompute, with the
    # LSE merge on two blocks per SM (several passes of its grid-stride loop
    # at this T) while the softmax-gradient GEMM's mainloop starts beside it
    T, V, D, C, seed = 20000, 3000, 64, 2000, 22
    x, C = _case(T, V, D, C, seed)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    tg = _dev(x["targets"][None, :].copy())
    ws = ss.workspace(T, V, C, D)
    a = ss.step_mtp(H, W, tg, [0.5], C, seed, ws, scale=1.0 / T)
    torch.cuda.synchronize()
    assert ss.read_status(ws)[0] == 0
    ref = orc.loss_and_grads_mtp(x["H"], x["W"], x["targets"][None, :], [0.5], C, seed, 1.0 / T)
    assert_loss_close(a["loss"].cpu().numpy(), ref["loss"])
    assert rel_fro(a["dH"].float().cpu().numpy(), ref["dH"]) < GRAD_RTOL
    assert rel_fro(a["dW"].cpu().numpy(), ref["dW"]) < GRAD_RTOL


def test_kernel_trace_records_every_launch():
    T, V, D, C = 300, 3000, 768, 517
    x, C = _case(T, V, D, C, 4)
    H, W = to_dev_bf16(x["H"]), to_dev_bf16(x["W"])
    ws = ss.workspace(T, V, C, D)
    with ss.KernelTrace(capacity=16) as tr:
        ss.step_separate(H, W, _dev(x["targets"]), C, 4, ws)
    torch.cuda.synchronize()
    names = [n for n, _ in tr.timings()]
    assert names == ["build_candidates", "gather_rows", "gemm_forward_lse", "lse_merge",
                     "gather_rows", "gemm_softmax_grad", "gemm_grads"]
    assert tr.kernels == [1] * 7
    with ss.KernelTrace(capacity=16) as tr:
        ss.step(H, W, _dev(x["targets"]), C, 4, ws)
    torch.cuda.synchronize()
    # one gather shared by the forward and the backward; the recompute is
    # launched (as the fallback) but finds its gate shut
    assert [n for n, _ in tr.timings()] == ["build_candidates", "gather_rows", "gemm_forward_lse",
                                           "lse_merge", "gemm_softmax_grad", "gemm_grads"]
    # the forward is two launches (first logit tile, the other tiles)
    assert tr.kernels == [1, 1, 2, 1, 1, 1]
    assert all(ms > 0 for _, ms in tr.timings())


# ------------------------------------------------------------ capped head

CAPPED = [
    # T, V, D, C, seed, scale, cap, tau
    (1, 64, 64, 1, 1, 1.0, 30.0, 7.5),
    (300, 3000, 768, 517, 4, 1.0, 30.0, 7.5),     # ragged T and C tails
    (257, 2000, 192, 1000, 5, 0.5, 6.0, 0.7),     # strongly saturated cap
    (500, 1000, 128, 1000, 6, 1.0 / 500, 15.0, 3.0),  # C = V
    (300, 3000, 768, 517, 9, 1.0, 80.0, 20.0),    # above the stored step's cap limit
]


@pytest.mark.parametrize("path", ["calls", "step"])
@pytest.mark.parametrize("T,V,D,C,seed,scale,cap,tau", CAPPED)
def test_capped_head_parity(orc, T, V, D, C, seed, scale, cap, tau, path):
    """z = cap / (1 + exp(-s / tau)) before the softmax: every element against
    the oracle of the same head, through the three calls (the backward
    recomputes the logits) and through ss_step (which keeps exp(z - cap) dz/ds
    from the forward)."""
    x, C = _case(T, V, D, C, seed)
    x["W"] = synth.make_inputs(1, V, D, 1.1, seed + 50, w_std=0.2)["W"]  # wide logits
    ref = _full_oracle(orc, x, C, seed, scale, cap=cap, tau=tau)
    got = RUNS[path](ss, x, C, seed, scale, cap=cap, tau=tau)
    assert got["status"] == 0
    np.testing.assert_array_equal(got["cand"], ref["cand"])
    assert_loss_close(got["loss"], ref["loss"])
    assert_loss_close(got["lse"], ref["lse"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL
    # and it differs from the plain head (the cap is really applied)
    plain = _full_oracle(orc, x, C, seed, scale)
    if C > 1:
        assert not np.allclose(plain["loss"], ref["loss"], rtol=1e-2)


@pytest.mark.parametrize("wid", [2, 4])
def test_full_size_capped_head(orc, wid):
    """Workloads T16384_C10240 (single-CTA tiles) and T65536_C24576 (CTA-pair
    softmax-gradient tiles) with the capped head, as in the plain full-size check."""
    w = synth.WORKLOADS[wid]
    x = synth.workload_inputs(w)
    _check_sampled(orc, x, w.T, w.V, w.D, w.C, w.seed, 200 + wid, exact_cols=wid == 2, cap=30.0,
                   tau=7.5)


def test_capped_graph_replay_equals_step():
    T, V, D, C, seed = 700, 6000, 768, 1500, 33
    x, C = _case(T, V, D, C, seed)
    H, W, tg = to_dev_bf16(x["H"]), to_dev_bf16(x["W"]), _dev(x["targets"])
    ws, ws2 = ss.workspace(T, V, C, D), ss.workspace(T, V, C, D)
    g = ss.StepGraph(H, W, tg, C, ws, scale=0.5, cap=15.0, tau=2.0)
    got = g.launch(seed)
    ref = ss.step(H, W, tg, C, seed, ws2, scale=0.5, cap=15.0, tau=2.0)
    plain = ss.step(H, W, tg, C, seed, ss.workspace(T, V, C, D), scale=0.5)
    torch.cuda.synchronize()
    for k in ("cand", "slot", "loss", "lse", "dH", "dW"):
        assert torch.equal(got[k], ref[k]), k
    assert not torch.equal(got["loss"], plain["loss"])
    g.close()


def test_permuted_ids_parity(orc):
    """The robustness variant of the synthetic inputs: the token ids of the
    Zipf law permuted by a fixed seed, so that the frequent ids (and with them
    the unique targets) are spread over the whole vocabulary instead of
    filling its first rows. Every element against the oracle."""
    T, V, D, C, seed = 500, 6000, 768, 1400, 12
    x = synth.make_inputs(T, V, D, 1.1, seed, permute_seed=99)
    C = max(C, len(np.unique(x["targets"])))
    assert x["targets"].max() > V // 2  # the frequent ids are no longer the first rows
    ref = _full_oracle(orc, x, C, seed, 1.0 / T)
    got = run_gpu(ss, x, C, seed, 1.0 / T)
    assert got["status"] == 0
    assert got["U"] == ref["U"]
    np.testing.assert_array_equal(got["cand"], ref["cand"])
    np.testing.assert_array_equal(got["slot"], ref["slot"])
    assert_loss_close(got["loss"], ref["loss"])
    assert rel_fro(got["dH"], ref["dH"]) < GRAD_RTOL
    assert rel_fro(got["dW"], ref["dW"]) < GRAD_RTOL


def test_permuted_ids_full_size(orc):
    """T16384_C10240 with permuted ids: cand and slot bit-exact, sampled rows
    and the gradient identities (as for the benchmark workload)."""
    w = synth.WORKLOADS[2]
    x = synth.make_inputs(w.T, w.V, w.D, w.zipf_s, w.seed, permute_seed=7)
    _check_sampled(orc, x, w.T, w.V, w.D, w.C, w.seed, 21, exact_cols=False)
