"""Pins for the CPU oracle, against facts that do not come from the oracle itself.

* candidate set: published SplitMix64 outputs, set invariants, brute force over
  every k-subset on tiny vocabularies, and a chi-square test of uniformity;
* forward: the full-vocabulary case equals dense cross-entropy (torch), any
  candidate set equals torch's cross-entropy on the candidate columns, zero
  logits give ln C, and a two-candidate case has a closed form;
* backward: torch autograd in fp64, central finite differences in fp64, closed
  forms with H = 0 and with W = 0, and the invariants of P - Y;
* a mutation check: planting plausible mistakes in the oracle's C source makes
  at least one of these checks fail.
"""
import itertools
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _vectors():
    out = []
    with open(os.path.join(GOLDEN, "splitmix64_vectors.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                s, i, o = (int(x) for x in line.split())
                out.append((s, i, o))
    return out


# ----------------------------------------------------------------- generator

def test_splitmix64_published_vectors(orc):
    vec = _vectors()
    assert len(vec) >= 6
    for seed, i, out in vec:
        assert orc.splitmix64_output(seed, i) == out


def test_negative_key_layout(orc):
    # high half = high 32 bits of the published output number v; low half = v
    for seed, i, out in _vectors():
        key = orc.negative_key(seed, i)
        assert key >> 32 == out >> 32
        assert key & 0xFFFFFFFF == i


# ------------------------------------------------------------ candidate set

def check_candidates(targets, V, C, cand, slot, U):
    t = np.asarray(targets)
    u = np.unique(t)
    assert U == len(u)
    assert cand.shape == (C,) and cand.dtype == np.int32
    assert np.array_equal(cand[:U], u), "targets first, ascending"
    neg = cand[U:]
    assert np.all(np.diff(neg) > 0), "negatives ascending and distinct"
    assert not np.isin(neg, u).any(), "no target among negatives"
    assert np.all((neg >= 0) & (neg < V))
    assert np.array_equal(cand[slot], t), "cand[slot[t]] == target[t]"
    assert np.all((slot >= 0) & (slot < U))


@pytest.mark.parametrize("T,V,C,s,seed", [
    (1, 10, 1, 1.1, 0),
    (1, 10, 10, 1.1, 1),
    (64, 300, 64, 1.1, 2),
    (256, 50304, 4096, 1.1, 0),
    (2000, 5000, 5000, 1.0, 5),     # full vocabulary
    (5000, 700, 700, 0.5, 6),       # nearly every id is a target
])
def test_candidate_invariants(orc, T, V, C, s, seed):
    rng = np.random.default_rng(seed)
    targets = synth.zipf_targets(rng, T, V, s)
    U = len(np.unique(targets))
    if U > C:
        C = U
    cand, slot, U2 = orc.build_candidates(targets, V, C, seed)
    check_candidates(targets, V, C, cand, slot, U2)
    if C == V:
        assert np.array_equal(np.sort(cand), np.arange(V))


def test_candidates_exact_fill(orc):
    # U == C: no negatives at all
    targets = np.array([5, 3, 3, 9, 0, 5], np.int32)
    cand, slot, U = orc.build_candidates(targets, 12, 4, 1)
    assert U == 4 and list(cand) == [0, 3, 5, 9]
    assert list(slot) == [2, 1, 1, 3, 0, 2]


def test_candidates_bruteforce_tiny(orc):
    # the chosen negatives are the k-subset of non-targets whose sorted key
    # tuple is smallest, found by enumerating every k-subset
    rng = np.random.default_rng(11)
    cases = 0
    for V in range(2, 10):
        for _ in range(6):
            T = int(rng.integers(1, V + 1))
            targets = rng.integers(0, V, size=T).astype(np.int32)
            U = len(np.unique(targets))
            for C in range(U, V + 1):
                seed = int(rng.integers(0, 2**63))
                cand, slot, U2 = orc.build_candidates(targets, V, C, seed)
                non = [v for v in range(V) if v not in set(targets.tolist())]
                k = C - U
                best = None
                for sub in itertools.combinations(non, k):
                    key = tuple(sorted(orc.negative_key(seed, v) for v in sub))
                    if best is None or key < best[0]:
                        best = (key, sorted(sub))
                assert list(cand[U:]) == best[1]
                check_candidates(targets, V, C, cand, slot, U2)
                cases += 1
    assert cases > 100


def test_candidates_uniform_chi2(orc):
    # V = 6, targets {0, 2}: 4 non-targets, k = 2 -> 6 equally likely subsets
    targets = np.array([0, 2, 2], np.int32)
    counts = {}
    n = 6000
    for seed in range(n):
        cand, _, U = orc.build_candidates(targets, 6, 4, seed)
        counts[tuple(cand[U:])] = counts.get(tuple(cand[U:]), 0) + 1
    assert len(counts) == 6
    exp = n / 6
    chi2 = sum((c - exp) ** 2 / exp for c in counts.values())
    assert chi2 < 20.52  # 5 degrees of freedom, p = 0.001


def test_candidates_errors(orc):
    with pytest.raises(orc.OracleError) as e:
        orc.build_candidates(np.array([1, 10], np.int32), 10, 5, 0)
    assert e.value.code == 4
    with pytest.raises(orc.OracleError) as e:
        orc.build_candidates(np.array([1, -1], np.int32), 10, 5, 0)
    assert e.value.code == 4
    with pytest.raises(orc.OracleError) as e:
        orc.build_candidates(np.array([1, 2, 3, 4], np.int32), 10, 3, 0)
    assert e.value.code == 3 and e.value.U == 4


def test_seed_changes_negatives(orc):
    targets = np.array([1, 2, 3], np.int32)
    a, _, _ = orc.build_candidates(targets, 1000, 50, 1)
    b, _, _ = orc.build_candidates(targets, 1000, 50, 2)
    assert np.array_equal(a[:3], b[:3]) and not np.array_equal(a[3:], b[3:])


# ------------------------------------------------------------------ forward

def _case(T, V, D, C, seed, w_std=0.3, s=1.1):
    x = synth.make_inputs(T, V, D, s, seed, w_std=w_std)
    U = len(np.unique(x["targets"]))
    C = max(C, U)
    return x, C


def _torch_ref(H64, W64, cand, slot, scale=1.0, cap=0.0, tau=1.0):
    """torch autograd of the loss; cap > 0 applies cap * sigmoid(logits / tau)
    (torch's own sigmoid) to the logits first."""
    Ht = torch.tensor(H64, requires_grad=True)
    Wt = torch.tensor(W64, requires_grad=True)
    logits = Ht @ Wt[torch.from_numpy(cand.astype(np.int64))].T
    if cap > 0:
        logits = cap * torch.sigmoid(logits / tau)
    y = torch.from_numpy(slot.astype(np.int64))
    loss = F.cross_entropy(logits, y, reduction="none")
    (scale * loss.sum()).backward()
    return (loss.detach().numpy(), torch.logsumexp(logits, 1).detach().numpy(),
            Ht.grad.numpy(), Wt.grad.numpy())


def test_forward_full_vocab_equals_dense_ce(orc):
    T, V, D = 40, 300, 32
    x = synth.make_inputs(T, V, D, 1.1, 3, w_std=0.3)
    cand, slot, U = orc.build_candidates(x["targets"], V, V, 3)
    H64, W64 = _f64(x["H"]), _f64(x["W"])
    dense = F.cross_entropy(torch.tensor(H64 @ W64.T), torch.from_numpy(x["targets"].astype(np.int64)),
                            reduction="none").numpy()
    l64, _ = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64)
    l32, _ = orc.forward(x["H"], x["W"], cand, slot)
    np.testing.assert_allclose(l64, dense, rtol=1e-12, atol=0)
    np.testing.assert_allclose(l32, dense, rtol=2e-5, atol=0)


@pytest.mark.parametrize("T,V,D,C,seed", [(33, 200, 24, 50, 1), (7, 64, 8, 9, 2), (100, 1000, 64, 300, 3)])
def test_forward_equals_ce_on_candidate_columns(orc, T, V, D, C, seed):
    x, C = _case(T, V, D, C, seed)
    cand, slot, U = orc.build_candidates(x["targets"], V, C, seed)
    loss, lse, _, _ = _torch_ref(_f64(x["H"]), _f64(x["W"]), cand, slot)
    l64, s64 = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64)
    np.testing.assert_allclose(l64, loss, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s64, lse, rtol=1e-12, atol=1e-13)
    l32, s32 = orc.forward(x["H"], x["W"], cand, slot)
    np.testing.assert_allclose(l32, loss, rtol=1e-5, atol=1e-6)
    assert np.all(l64 >= 0)


@pytest.mark.parametrize("C", [1, 5, 4096, 10240])
def test_uniform_logits_give_ln_C(orc, C):
    T, V, D = 6, max(C, 16), 16
    x = synth.make_inputs(T, V, D, 1.1, 4)
    cand, slot, U = orc.build_candidates(x["targets"] % C if C < 16 else x["targets"], V, C, 4)
    for H, W in ((np.zeros_like(x["H"]), x["W"]), (x["H"], np.zeros_like(x["W"]))):
        loss, lse = orc.forward(H, W, cand, slot)
        assert np.all(np.abs(loss - math.log(C)) <= 2e-7 * max(1.0, math.log(C)))
        np.testing.assert_array_equal(loss, lse)


def test_two_candidate_closed_form(orc):
    # every target is id 1 of V = 3, C = 2: one negative n; with logits a (target)
    # and b (negative), loss = log(1 + e^(b - a)) and dL/dh = sigmoid(b - a) (w_n - w_1)
    W = synth.f32_to_bf16_bits(np.array([[0.5, -1.25], [2.0, 0.75], [-0.5, 1.5]], np.float32))
    H = synth.f32_to_bf16_bits(np.array([[1.0, 0.0], [0.0, 1.0], [2.0, -1.0], [0.25, 0.5]], np.float32))
    targets = np.ones(4, np.int32)
    cand, slot, U = orc.build_candidates(targets, 3, 2, 9)
    assert U == 1 and cand[0] == 1 and cand[1] in (0, 2)
    w = synth.bf16_bits_to_f32(W).astype(np.float64)
    h = synth.bf16_bits_to_f32(H).astype(np.float64)
    a, b = h @ w[1], h @ w[cand[1]]
    loss = np.log1p(np.exp(b - a))
    sig = 1 / (1 + np.exp(-(b - a)))
    l, lse = orc.forward(H, W, cand, slot, dtype=np.float64)
    np.testing.assert_allclose(l, loss, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse, a + loss, rtol=1e-14)
    dH = orc.backward_dH(H, W, cand, slot, lse, dtype=np.float64)
    np.testing.assert_allclose(dH, sig[:, None] * (w[cand[1]] - w[1])[None, :], rtol=1e-13, atol=1e-15)
    dWc = orc.backward_dWc(H, W, cand, slot, lse, dtype=np.float64)
    np.testing.assert_allclose(dWc[0], -(sig[:, None] * h).sum(0), rtol=1e-13)
    np.testing.assert_allclose(dWc[1], (sig[:, None] * h).sum(0), rtol=1e-13)


# ----------------------------------------------------------------- backward

@pytest.mark.parametrize("T,V,D,C,seed,scale", [(33, 200, 24, 50, 1, 1.0), (50, 120, 16, 120, 2, 0.02),
                                                (100, 1000, 64, 300, 3, 1.0 / 100)])
def test_backward_matches_torch_autograd(orc, T, V, D, C, seed, scale):
    x, C = _case(T, V, D, C, seed)
    cand, slot, U = orc.build_candidates(x["targets"], V, C, seed)
    _, _, gH, gW = _torch_ref(_f64(x["H"]), _f64(x["W"]), cand, slot, scale)
    r64 = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, seed, scale, dtype=np.float64)
    np.testing.assert_allclose(r64["dH"], gH, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(r64["dW"], gW, rtol=1e-10, atol=1e-13)
    r32 = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, seed, scale)
    for k, ref in (("dH", gH), ("dW", gW)):
        err = np.linalg.norm(r32[k] - ref) / np.linalg.norm(ref)
        assert err < 1e-5, (k, err)


def test_backward_finite_differences(orc):
    rng = np.random.default_rng(21)
    T, V, D, C, scale = 3, 9, 6, 5, 0.7
    H = rng.standard_normal((T, D))
    W = rng.standard_normal((V, D)) * 0.8
    targets = np.array([4, 1, 4], np.int32)
    cand, slot, U = orc.build_candidates(targets, V, C, 5)

    def L(H_, W_):
        loss, _ = orc.forward(H_, W_, cand, slot, dtype=np.float64)
        return scale * loss.sum()

    _, lse = orc.forward(H, W, cand, slot, dtype=np.float64)
    dH = orc.backward_dH(H, W, cand, slot, lse, scale, dtype=np.float64)
    dWc = orc.backward_dWc(H, W, cand, slot, lse, scale, dtype=np.float64)
    dW = np.zeros_like(W)
    dW[cand] = dWc
    eps = 1e-6
    for M, G in ((H, dH), (W, dW)):
        num = np.zeros_like(M)
        for idx in np.ndindex(M.shape):
            keep = M[idx]
            M[idx] = keep + eps
            lp = L(H, W)
            M[idx] = keep - eps
            lm = L(H, W)
            M[idx] = keep
            num[idx] = (lp - lm) / (2 * eps)
        assert np.linalg.norm(num - G) <= 1e-6 * np.linalg.norm(G) + 1e-9
    # rows of W outside the candidate set carry no gradient
    outside = np.setdiff1d(np.arange(V), cand)
    assert outside.size == V - C and np.all(dW[outside] == 0)


def test_backward_W_zero_closed_form(orc):
    # W = 0: P is uniform 1/C, so dH = 0 and dWc[j] = scale * sum_t (1/C - [slot_t == j]) H[t]
    T, V, D, C, scale = 20, 50, 8, 12, 0.5
    x, C = _case(T, V, D, C, 8, w_std=0.02)
    W0 = np.zeros_like(x["W"])
    r = orc.loss_and_grads(x["H"], W0, x["targets"], C, 8, scale, dtype=np.float64)
    assert np.all(r["dH"] == 0)
    Y = np.zeros((T, C))
    Y[np.arange(T), r["slot"]] = 1
    ref = scale * (1.0 / C - Y).T @ _f64(x["H"])
    np.testing.assert_allclose(r["dWc"], ref, rtol=1e-12, atol=1e-14)


def test_backward_H_zero_closed_form(orc):
    # H = 0: dWc = 0 and dH[t] = scale * (mean_j W[cand[j]] - W[target_t])
    T, V, D, C, scale = 20, 50, 8, 12, 2.0
    x, C = _case(T, V, D, C, 9, w_std=0.5)
    H0 = np.zeros_like(x["H"])
    r = orc.loss_and_grads(H0, x["W"], x["targets"], C, 9, scale, dtype=np.float64)
    assert np.all(r["dWc"] == 0)
    W64 = _f64(x["W"])
    ref = scale * (W64[r["cand"]].mean(0)[None, :] - W64[x["targets"]])
    np.testing.assert_allclose(r["dH"], ref, rtol=1e-12, atol=1e-14)


def test_backward_invariants(orc):
    T, V, D, C = 64, 500, 32, 100
    x, C = _case(T, V, D, C, 12, w_std=0.2)
    rng = np.random.default_rng(0)
    dW0 = rng.standard_normal((V, D)).astype(np.float32)
    r = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, 12, dW_init=dW0)
    # rows of P - Y sum to zero -> candidate-row gradients sum to zero
    colsum = np.abs(r["dWc"].astype(np.float64).sum(0)).max()
    assert colsum <= 1e-5 * np.abs(r["dWc"]).max()
    # <dWc, W_c> = sum G*S = <dH, H>
    lhs = float((r["dWc"].astype(np.float64) * _f64(x["W"])[r["cand"]]).sum())
    rhs = float((r["dH"].astype(np.float64) * _f64(x["H"])).sum())
    assert abs(lhs - rhs) <= 1e-4 * (abs(lhs) + 1e-3)
    # rows outside the candidate set are left as given
    outside = np.setdiff1d(np.arange(V), r["cand"])
    assert np.array_equal(r["dW"][outside], dW0[outside])
    # accumulate adds instead of overwriting
    ra = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, 12, dW_init=dW0, accumulate=True)
    np.testing.assert_allclose(ra["dW"][r["cand"]], dW0[r["cand"]] + r["dWc"], rtol=1e-6, atol=1e-7)
    assert np.array_equal(ra["dW"][outside], dW0[outside])


def test_row_subsets_match_full(orc):
    T, V, D, C = 40, 400, 32, 90
    x, C = _case(T, V, D, C, 13)
    cand, slot, U = orc.build_candidates(x["targets"], V, C, 13)
    loss, lse = orc.forward(x["H"], x["W"], cand, slot)
    rows = np.array([39, 0, 17, 17, 5])
    l2, s2 = orc.forward(x["H"], x["W"], cand, slot, rows=rows)
    assert np.array_equal(l2, loss[rows]) and np.array_equal(s2, lse[rows])
    dH = orc.backward_dH(x["H"], x["W"], cand, slot, lse)
    dH2 = orc.backward_dH(x["H"], x["W"], cand, slot, lse[rows], rows=rows)
    assert np.array_equal(dH2, dH[rows])
    dWc = orc.backward_dWc(x["H"], x["W"], cand, slot, lse)
    cols = np.array([C - 1, 0, 3])
    assert np.array_equal(orc.backward_dWc(x["H"], x["W"], cand, slot, lse, cols=cols), dWc[cols])


# ------------------------------------------------------ planted mistakes

MUTATIONS = [
    ("drop one-hot term in dH", "REAL g = scale * (wsum * EXP(z - lse_rows[i]) - y) *",
     "REAL g = scale * (wsum * EXP(z - lse_rows[i])) *"),
    ("capped head: dz/ds factor dropped in dW",
     "REAL g = scale * (wsum * EXP(z - lse[t]) - y) * head_dz_##SUF(z, cap, tau);",
     "REAL g = scale * (wsum * EXP(z - lse[t]) - y);"),
    ("several targets: weights ignored in the loss", "acc += w[k] * (l - s[slot[k * T + t]]);",
     "acc += (l - s[slot[k * T + t]]);"),
    ("several targets: weight sum missing in dH", "REAL g = scale * (wsum * EXP(z - lse_rows[i]) - y)",
     "REAL g = scale * (EXP(z - lse_rows[i]) - y)"),
    ("several targets: only the first target in G", "if (slot[k * T + t] == j) y += w[k];",
     "if (k == 0 && slot[k * T + t] == j) y += w[k];"),
    ("capped head: logistic of +s", "cap / ((REAL)1 + EXP(-s / tau))", "cap / ((REAL)1 + EXP(s / tau))"),
    ("capped head: dz/ds without (A - z)", "z * (cap - z) / (cap * tau)", "z / tau"),
    ("sign of the log-sum", "REAL l = m + LOG(sum);", "REAL l = m - LOG(sum);"),
    ("transposed operand in dW", "for (int64_t d = 0; d < D; ++d) out[d] += g * (REAL)LOAD(h[d]);",
     "for (int64_t d = 0; d < D; ++d) out[d] += g * (REAL)LOAD(w[d]);"),
    ("wrong target index", "s[slot[k * T + t]]", "s[0]"),
    ("dropped term of the dot product", "for (int64_t d = 0; d < D; ++d) acc +=",
     "for (int64_t d = 1; d < D; ++d) acc +="),
    ("negatives left in key order", "qsort(neg, (size_t)k, sizeof(int32_t), cmp_i32);", ""),
    ("targets not deduplicated", "if (U == 0 || u[U - 1] != u[i]) u[U++] = u[i];", "u[U++] = u[i];"),
    ("wrong hash constant", "0xBF58476D1CE4E5B9ull", "0xBF58476D1CE4E5B8ull"),
    ("FP8 head: e4m3 grid one bit too fine", "const float q = ldexpf(1.0f, E - 3);",
     "const float q = ldexpf(1.0f, E - 4);"),
    ("FP8 head: scale exponent one too large", "return m <= 0.875f ? 9 - k : 8 - k;",
     "return m <= 0.875f ? 10 - k : 9 - k;"),
    ("FP8 gradients: e5m2 grid one bit too fine", "const float q = ldexpf(1.0f, E - 2);",
     "const float q = ldexpf(1.0f, E - 3);"),
    ("FP8 gradients: G not rounded",
     "return orc_round_e5m2(ldexpf((expf(z - lse) - y) * head_dz_f32(z, cap, tau), e));",
     "return ldexpf((expf(z - lse) - y) * head_dz_f32(z, cap, tau), e);"),
    ("FP8 gradients: wrong power-of-two scale", "const float f = ldexpf(scale, -e);\n#pragma omp parallel\n",
     "const float f = ldexpf(scale, 1 - e);\n#pragma omp parallel\n"),
    ("FP8 gradients: capped dz/ds dropped", "* head_dz_f32(z, cap, tau), e));", ", e));"),
    ("FP8 gradients: exponent bound doubled", "while (B * ldexp(1.0, e + 1) <= 57344.0) ++e;",
     "while (B * ldexp(1.0, e + 1) <= 114688.0) ++e;"),
]


def _battery(orc):
    """Run a compact set of the pins above; return the names of those that fail."""
    failed = []
    try:
        for seed, i, out in _vectors():
            assert orc.splitmix64_output(seed, i) == out
    except AssertionError:
        failed.append("vectors")
    T, V, D, C = 30, 150, 16, 40
    x, C = _case(T, V, D, C, 31)
    try:
        cand, slot, U = orc.build_candidates(x["targets"], V, C, 31)
        check_candidates(x["targets"], V, C, cand, slot, U)
    except (AssertionError, Exception):
        failed.append("candidates")
        return failed
    _, _, gH, gW = _torch_ref(_f64(x["H"]), _f64(x["W"]), cand, slot)
    loss, lse, _, _ = _torch_ref(_f64(x["H"]), _f64(x["W"]), cand, slot)
    l64, s64 = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64)
    if not np.allclose(l64, loss, rtol=1e-10):
        failed.append("forward")
    dH = orc.backward_dH(x["H"], x["W"], cand, slot, s64, dtype=np.float64)
    dWc = orc.backward_dWc(x["H"], x["W"], cand, slot, s64, dtype=np.float64)
    if not np.allclose(dH, gH, rtol=1e-8, atol=1e-12):
        failed.append("dH")
    if not np.allclose(dWc, gW[cand], rtol=1e-8, atol=1e-12):
        failed.append("dW")
    # the capped head against torch autograd of cap * sigmoid(logits / tau)
    cap, tau = 6.0, 0.7
    loss, _, gH, gW = _torch_ref(_f64(x["H"]), _f64(x["W"]), cand, slot, cap=cap, tau=tau)
    l64, s64 = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64, cap=cap, tau=tau)
    if not np.allclose(l64, loss, rtol=1e-10):
        failed.append("capped forward")
    dH = orc.backward_dH(x["H"], x["W"], cand, slot, s64, dtype=np.float64, cap=cap, tau=tau)
    dWc = orc.backward_dWc(x["H"], x["W"], cand, slot, s64, dtype=np.float64, cap=cap, tau=tau)
    if not np.allclose(dH, gH, rtol=1e-8, atol=1e-12):
        failed.append("capped dH")
    if not np.allclose(dWc, gW[cand], rtol=1e-8, atol=1e-12):
        failed.append("capped dW")
    # two weighted targets per token against torch autograd
    try:
        bad = _mtp_mismatch(orc, 12, 80, 8, 30, 32, [1.0, 0.5], 0.0, 1.0)
    except Exception:
        bad = ["mtp crashed"]
    failed += bad
    # the FP8 roundings against torch's float8 conversions, and the closed form
    # of the FP8 gradients at H = 0
    if _fp8_rounding_mismatch(orc, 2000):
        failed.append("fp8 rounding")
    if _e4m3_exponent_mismatch(orc):
        failed.append("e4m3 scale exponent")
    if _fp8_grad_closed_form_mismatch(orc):
        failed.append("fp8 gradients")
    if _g8_exponent_mismatch(orc):
        failed.append("fp8 gradient exponent")
    for k in (4.0, 8.0):
        if _fp8_grad_closed_form_mismatch(orc, cap_over_tau=k):
            failed.append(f"capped fp8 gradients {k}")
    return failed


def _battery_in_subprocess(so_path):
    """Run the battery against another build of the oracle in a child process, so
    that a planted mistake which corrupts memory cannot take the test run down."""
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import json, sys; sys.path[:0] = [%r, %r]; import oracle, test_oracle as t; "
            "oracle._lib = oracle.load(%r); print('BATTERY', json.dumps(t._battery(oracle)))"
            % (os.path.dirname(here), here, str(so_path)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    for line in r.stdout.splitlines():
        if line.startswith("BATTERY "):
            return json.loads(line[len("BATTERY "):])
    return [f"crashed (exit {r.returncode})"]


def test_pins_catch_planted_mistakes(orc, tmp_path):
    src = open(orc._SRC).read()
    assert _battery(orc) == []
    for i, (name, old, new) in enumerate(MUTATIONS):
        assert src.count(old) >= 1, name
        mut = tmp_path / f"mut{i}.c"
        mut.write_text(src.replace(old, new))
        so = tmp_path / f"mut{i}.so"
        subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                        "-o", str(so), str(mut), "-lm"], check=True)
        failed = _battery_in_subprocess(so)
        assert failed, f"planted mistake not caught: {name}"


# ----------------------------------------------------- the capped head variant

CAPS = [(30.0, 7.5), (6.0, 0.7), (15.0, 3.0)]


@pytest.mark.parametrize("cap,tau", CAPS)
def test_capped_head_against_torch_autograd(orc, cap, tau):
    """z = cap * sigmoid(s / tau), the loss and both gradients, against torch
    (its sigmoid, its cross-entropy, its autograd) in fp64; the fp32 oracle
    within fp32 rounding of it."""
    T, V, D, C = 30, 400, 24, 90
    x, C = _case(T, V, D, C, 7, w_std=0.3)
    cand, slot, _ = orc.build_candidates(x["targets"], V, C, 7)
    loss, lse, gH, gW = _torch_ref(_f64(x["H"]), _f64(x["W"]), cand, slot, scale=0.5, cap=cap,
                                   tau=tau)
    l64, s64 = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64, cap=cap, tau=tau)
    np.testing.assert_allclose(l64, loss, rtol=1e-12)
    np.testing.assert_allclose(s64, lse, rtol=1e-12)
    dH = orc.backward_dH(x["H"], x["W"], cand, slot, s64, 0.5, dtype=np.float64, cap=cap, tau=tau)
    dWc = orc.backward_dWc(x["H"], x["W"], cand, slot, s64, 0.5, dtype=np.float64, cap=cap,
                           tau=tau)
    np.testing.assert_allclose(dH, gH, rtol=1e-9, atol=1e-13)
    np.testing.assert_allclose(dWc, gW[cand], rtol=1e-9, atol=1e-13)
    l32, _ = orc.forward(x["H"], x["W"], cand, slot, cap=cap, tau=tau)
    np.testing.assert_allclose(l32, loss, rtol=2e-5, atol=1e-6)


def test_capped_head_is_a_shifted_tanh_softcap(orc):
    """cap * sigmoid(s / tau) = cap/2 + (cap/2) tanh(s / (2 tau)), and softmax
    ignores the shift: the loss equals cross-entropy of the symmetric softcap
    (cap/2) tanh(s / (2 tau)), written here with numpy's tanh."""
    T, V, D, C = 25, 300, 16, 70
    x, C = _case(T, V, D, C, 8, w_std=0.5)
    cand, slot, _ = orc.build_candidates(x["targets"], V, C, 8)
    cap, tau = 20.0, 2.5
    S = _f64(x["H"]) @ _f64(x["W"])[cand].T
    z = (cap / 2) * np.tanh(S / (2 * tau))
    m = z.max(1, keepdims=True)
    lse = (m + np.log(np.exp(z - m).sum(1, keepdims=True)))[:, 0]
    expect = lse - z[np.arange(T), slot]
    l64, _ = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64, cap=cap, tau=tau)
    np.testing.assert_allclose(l64, expect, rtol=1e-12)


def test_capped_head_uniform_logits_closed_form(orc):
    """W = 0: every z = cap / 2, so loss = ln C, dH = 0, and
    dW[cand[j]] = scale * cap / (4 tau) * sum_t (1/C - [slot[t] = j]) H[t]."""
    T, V, D, C = 20, 100, 8, 37
    x, C = _case(T, V, D, C, 9)
    x["W"] = np.zeros_like(x["W"])
    cand, slot, _ = orc.build_candidates(x["targets"], V, C, 9)
    cap, tau, scale = 12.0, 1.5, 0.3
    l64, s64 = orc.forward(x["H"], x["W"], cand, slot, dtype=np.float64, cap=cap, tau=tau)
    np.testing.assert_allclose(l64, np.log(C), rtol=1e-14)
    dH = orc.backward_dH(x["H"], x["W"], cand, slot, s64, scale, dtype=np.float64, cap=cap, tau=tau)
    assert np.all(dH == 0)
    dWc = orc.backward_dWc(x["H"], x["W"], cand, slot, s64, scale, dtype=np.float64, cap=cap,
                           tau=tau)
    H64 = _f64(x["H"])
    Y = np.zeros((T, C))
    Y[np.arange(T), slot] = 1
    expect = scale * cap / (4 * tau) * ((1.0 / C - Y).T @ H64)
    np.testing.assert_allclose(dWc, expect, rtol=1e-10, atol=1e-14)


def test_capped_head_finite_differences(orc):
    """Central differences in fp64 over every element of H and of the candidate
    rows of W, with the capped head."""
    T, V, D, C = 3, 12, 5, 6
    rng = np.random.default_rng(10)
    H = rng.normal(size=(T, D))
    W = rng.normal(size=(V, D))
    targets = rng.integers(0, V, T).astype(np.int32)
    cand, slot, _ = orc.build_candidates(targets, V, C, 10)
    cap, tau, scale = 5.0, 0.8, 1.0
    _, lse = orc.forward(H, W, cand, slot, dtype=np.float64, cap=cap, tau=tau)
    dH = orc.backward_dH(H, W, cand, slot, lse, scale, dtype=np.float64, cap=cap, tau=tau)
    dWc = orc.backward_dWc(H, W, cand, slot, lse, scale, dtype=np.float64, cap=cap, tau=tau)

    def total(Hx, Wx):
        return orc.forward(Hx, Wx, cand, slot, dtype=np.float64, cap=cap, tau=tau)[0].sum()

    eps = 1e-6
    for (t, d) in np.ndindex(T, D):
        Hp, Hm = H.copy(), H.copy()
        Hp[t, d] += eps
        Hm[t, d] -= eps
        fd = (total(Hp, W) - total(Hm, W)) / (2 * eps)
        assert abs(fd - dH[t, d]) <= 1e-6 * max(1.0, abs(fd))
    for (j, d) in np.ndindex(C, D):
        Wp, Wm = W.copy(), W.copy()
        Wp[cand[j], d] += eps
        Wm[cand[j], d] -= eps
        fd = (total(H, Wp) - total(H, Wm)) / (2 * eps)
        assert abs(fd - dWc[j, d]) <= 1e-6 * max(1.0, abs(fd))


# ------------------------------------------------ several targets per token

def _torch_ref_mtp(H64, W64, cand, slot, weights, scale=1.0, cap=0.0, tau=1.0):
    """torch autograd of sum_k w[k] * CE(logits, slot[k]) (slot [K, T])."""
    Ht = torch.tensor(H64, requires_grad=True)
    Wt = torch.tensor(W64, requires_grad=True)
    logits = Ht @ Wt[torch.from_numpy(cand.astype(np.int64))].T
    if cap > 0:
        logits = cap * torch.sigmoid(logits / tau)
    loss = 0
    for k, wk in enumerate(weights):
        loss = loss + wk * F.cross_entropy(logits, torch.from_numpy(slot[k].astype(np.int64)),
                                           reduction="none")
    (scale * loss.sum()).backward()
    return (loss.detach().numpy(), torch.logsumexp(logits, 1).detach().numpy(),
            Ht.grad.numpy(), Wt.grad.numpy())


def _mtp_case(T, V, D, C, seed, K, w_std=0.3):
    rng = np.random.default_rng(seed)
    x = synth.make_inputs(T, V, D, 1.1, seed, w_std=w_std)
    tg = np.stack([x["targets"]] + [synth.zipf_targets(rng, T, V, 1.1) for _ in range(K - 1)])
    C = max(C, len(np.unique(tg)))
    return x, tg.astype(np.int32), C


def _mtp_mismatch(orc, T, V, D, C, seed, weights, cap, tau):
    """Names of the quantities where the fp64 oracle disagrees with torch."""
    x, tg, C = _mtp_case(T, V, D, C, seed, len(weights))
    cand, slot_flat, _ = orc.build_candidates(tg.reshape(-1), V, C, seed)
    slot = slot_flat.reshape(tg.shape)
    loss, lse, gH, gW = _torch_ref_mtp(_f64(x["H"]), _f64(x["W"]), cand, slot, weights, 0.7, cap,
                                       tau)
    l64, s64 = orc.forward_mtp(x["H"], x["W"], cand, slot, weights, dtype=np.float64, cap=cap,
                               tau=tau)
    dH = orc.backward_dH_mtp(x["H"], x["W"], cand, slot, weights, s64, 0.7, dtype=np.float64,
                             cap=cap, tau=tau)
    dWc = orc.backward_dWc_mtp(x["H"], x["W"], cand, slot, weights, s64, 0.7, dtype=np.float64,
                               cap=cap, tau=tau)
    bad = []
    if not np.allclose(l64, loss, rtol=1e-11):
        bad.append("mtp forward")
    if not np.allclose(s64, lse, rtol=1e-12):
        bad.append("mtp lse")
    if not np.allclose(dH, gH, rtol=1e-9, atol=1e-13):
        bad.append("mtp dH")
    if not np.allclose(dWc, gW[cand], rtol=1e-9, atol=1e-13):
        bad.append("mtp dW")
    return bad


@pytest.mark.parametrize("weights,cap,tau", [([1.0, 0.5], 0.0, 1.0), ([1.0, 0.3, 0.2], 0.0, 1.0),
                                             ([0.6, 0.4], 20.0, 4.0), ([2.0], 0.0, 1.0)])
def test_several_targets_against_torch_autograd(orc, weights, cap, tau):
    """sum_k w[k] * CE over the same logits, both gradients, against torch in
    fp64, with and without the capped head."""
    assert _mtp_mismatch(orc, 40, 500, 24, 120, 11, weights, cap, tau) == []


def test_single_weight_one_target_is_the_plain_loss(orc):
    """K = 1, w = 1 gives the single-target results bit for bit."""
    x, tg, C = _mtp_case(50, 700, 32, 200, 12, 1)
    cand, slot, _ = orc.build_candidates(tg[0], 700, C, 12)
    for dt in (np.float32, np.float64):
        l1, s1 = orc.forward(x["H"], x["W"], cand, slot, dtype=dt)
        lk, sk = orc.forward_mtp(x["H"], x["W"], cand, slot[None], [1.0], dtype=dt)
        np.testing.assert_array_equal(l1, lk)
        np.testing.assert_array_equal(s1, sk)
        d1 = orc.backward_dWc(x["H"], x["W"], cand, slot, s1, 0.5, dtype=dt)
        dk = orc.backward_dWc_mtp(x["H"], x["W"], cand, slot[None], [1.0], sk, 0.5, dtype=dt)
        np.testing.assert_array_equal(d1, dk)


def test_repeated_target_counts_its_weights(orc):
    """Two target rows equal to each other with weights a and b give the loss of
    one target row with weight a + b (a weighted one-hot term adds up)."""
    x, tg, C = _mtp_case(30, 400, 16, 100, 13, 1)
    cand, slot, _ = orc.build_candidates(tg[0], 400, C, 13)
    two = np.stack([slot, slot])
    l2, s2 = orc.forward_mtp(x["H"], x["W"], cand, two, [0.25, 0.5], dtype=np.float64)
    l1, _ = orc.forward_mtp(x["H"], x["W"], cand, slot[None], [0.75], dtype=np.float64)
    np.testing.assert_allclose(l2, l1, rtol=1e-14)
    d2 = orc.backward_dH_mtp(x["H"], x["W"], cand, two, [0.25, 0.5], s2, dtype=np.float64)
    d1 = orc.backward_dH_mtp(x["H"], x["W"], cand, slot[None], [0.75], s2, dtype=np.float64)
    np.testing.assert_allclose(d2, d1, rtol=1e-12, atol=1e-15)


def test_several_targets_loss_and_grads_builds_over_all_targets(orc):
    x, tg, C = _mtp_case(60, 900, 16, 150, 14, 3)
    ref = orc.loss_and_grads_mtp(x["H"], x["W"], tg, [1.0, 0.5, 0.25], C, 14)
    allt = np.unique(tg)
    assert ref["U"] == allt.size
    np.testing.assert_array_equal(ref["cand"][:allt.size], allt)
    np.testing.assert_array_equal(ref["cand"][ref["slot"]], tg)


# ------------------------------------------------------------------ FP8 head

def test_e4m3_rounding_against_torch(orc):
    """round_e4m3 against torch's float8_e4m3fn conversion (round to nearest,
    ties to even) on values spread over every binade and on the grid's midpoints."""
    rng = np.random.default_rng(20)
    mags = np.exp2(rng.uniform(-12, np.log2(448.0), 20000)).astype(np.float32)
    x = (mags * rng.choice([-1, 1], mags.size)).astype(np.float32)
    grid = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    grid = np.unique(grid[torch.isfinite(grid)].numpy().astype(np.float32))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, grid, mids, -mids]).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy()
    got = np.array([orc.round_e4m3(float(v)) for v in x], np.float32)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_grid_is_fixed_and_ties_go_to_even(orc):
    grid = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    grid = np.unique(grid[torch.isfinite(grid)].numpy().astype(np.float32))
    assert grid.size == 253 and grid.max() == 448.0 and grid[grid > 0].min() == 2.0 ** -9
    for v in grid:
        assert orc.round_e4m3(float(v)) == v
    codes = torch.from_numpy(grid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for a, b, ca, cb in zip(grid[:-1], grid[1:], codes[:-1], codes[1:]):
        if a < 0 or b <= 0:
            continue  # the positive half suffices (the rounding is sign-symmetric)
        even = a if int(ca) % 2 == 0 else b
        assert orc.round_e4m3(float((a + b) / 2)) == even, (a, b)
    assert orc.round_e4m3(1000.0) == 448.0 and orc.round_e4m3(-449.0) == -448.0


def _e4m3_exponent_mismatch(orc):
    rng = np.random.default_rng(21)
    for amax in np.concatenate([np.exp2(rng.uniform(-20, 20, 2000)), [448.0, 224.0, 1.0, 0.875]]):
        amax = float(np.float32(amax))
        e = orc.e4m3_scale_exponent(amax)
        if not amax * 2.0 ** e <= 448.0 < amax * 2.0 ** (e + 1):
            return True
    return orc.e4m3_scale_exponent(0.0) != 0


def test_e4m3_scale_exponent_is_the_largest_that_fits(orc):
    assert not _e4m3_exponent_mismatch(orc)


def _float8_grid(dtype):
    grid = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(dtype).float()
    return np.unique(grid[torch.isfinite(grid)].numpy().astype(np.float32))


def _fp8_rounding_mismatch(orc, n):
    """Both roundings against torch's float8 conversions (round to nearest,
    ties to even) over every binade, the grid points and their midpoints."""
    rng = np.random.default_rng(23)
    for dt, top, fn, lo in ((torch.float8_e4m3fn, 448.0, orc.round_e4m3, -12),
                            (torch.float8_e5m2, 57344.0, orc.round_e5m2, -19)):
        mags = np.exp2(rng.uniform(lo, np.log2(top), n)).astype(np.float32)
        x = (mags * rng.choice([-1, 1], mags.size)).astype(np.float32)
        grid = _float8_grid(dt)
        mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
        x = np.concatenate([x, grid, mids]).astype(np.float32)
        x = x[np.abs(x) < top]
        ref = torch.from_numpy(x).to(dt).float().numpy()
        got = np.array([fn(float(v)) for v in x], np.float32)
        if not np.array_equal(got, ref):
            return True
    return False


def test_e5m2_rounding_against_torch(orc):
    assert not _fp8_rounding_mismatch(orc, 20000)


def test_e5m2_grid_is_fixed_and_ties_go_to_even(orc):
    grid = _float8_grid(torch.float8_e5m2)
    assert grid.size == 247 and grid.max() == 57344.0 and grid[grid > 0].min() == 2.0 ** -16
    for v in grid:
        assert orc.round_e5m2(float(v)) == v
    codes = torch.from_numpy(grid).to(torch.float8_e5m2).view(torch.uint8).numpy()
    for a, b, ca, cb in zip(grid[:-1], grid[1:], codes[:-1], codes[1:]):
        if a < 0 or b <= 0:
            continue
        even = a if int(ca) % 2 == 0 else b
        assert orc.round_e5m2(float((a + b) / 2)) == even, (a, b)
    assert orc.round_e5m2(1e6) == 57344.0 and orc.round_e5m2(-60000.0) == -57344.0


def _fp8_grad_closed_form_mismatch(orc, cap_over_tau=0.0):
    """FP8 gradients at H = 0 with C = 32: every logit is 0, P = 1/32, so
    2^15 P = 1024 is on the e5m2 grid while the target entry 2^15 (1/32 - 1)
    = -31744 rounds to -32768 (spacing 4096 in that binade, not a tie):
    dH[t] = scale (sum_j W_q[cand[j]] / 32 - (33/32) W_q[y_t]) and dW = 0,
    where the exact-G gradient would have (32/32) W_q[y_t].
    With the capped head (cap = k tau), z = cap / 2 everywhere, so P is the
    same and dz/ds = k / 4: the bound k / 4 moves the exponent to 15 - log2(k/4)
    and the same e5m2 values come out, times k / 4."""
    T, V, D, C, seed, scale = 4, 64, 16, 32, 33, 0.75
    tau = 1.5
    cap = cap_over_tau * tau
    x = synth.make_inputs(T, V, D, 1.1, seed)
    H0 = np.zeros_like(x["H"])
    r = orc.loss_and_grads_fp8(H0, x["W"], x["targets"], C, seed, scale, grads=True, cap=cap,
                               tau=tau)
    Wq = synth.bf16_bits_to_f32(orc.fp8_inputs(H0, x["W"], r["cand"])[1]).astype(np.float64)
    Wc = Wq[r["cand"]]
    y = Wq[x["targets"]]
    f = cap_over_tau / 4.0 if cap_over_tau else 1.0
    expect = f * scale * (Wc.sum(0)[None, :] / 32.0 - (33.0 / 32.0) * y)
    plain = f * scale * (Wc.sum(0)[None, :] / 32.0 - y)
    bad = not np.allclose(r["dH"], expect, rtol=1e-5, atol=1e-7)
    bad |= np.allclose(r["dH"], plain, rtol=1e-5, atol=1e-7)
    bad |= bool(np.any(r["dW"] != 0))
    z0 = cap / 2.0 if cap_over_tau else 0.0
    bad |= not np.allclose(r["lse"], z0 + np.log(32.0), rtol=1e-6)
    return bad


def _g8_exponent_mismatch(orc):
    if orc.g8_exponent(0.0, 1.0) != 15 or orc.g8_exponent(30.0, 7.5) != 15:
        return True
    for cap, tau in ((4.0, 0.5), (100.0, 1.0), (1.0, 10.0), (3.0, 7.0)):
        B = cap / (4.0 * tau)
        e = orc.g8_exponent(cap, tau)
        if not B * 2.0 ** e <= 57344.0 < B * 2.0 ** (e + 1):
            return True
    return False


def test_fp8_gradient_exponent_is_the_largest_that_fits(orc):
    """2^15 for the plain head (|P - Y| <= 1); for the capped head the bound is
    cap / (4 tau), the largest dz/ds (at z = cap / 2)."""
    assert not _g8_exponent_mismatch(orc)


@pytest.mark.parametrize("k", [4.0, 8.0])
def test_capped_fp8_gradients_closed_form_at_zero_H(orc, k):
    assert not _fp8_grad_closed_form_mismatch(orc, cap_over_tau=k)


def test_fp8_gradients_closed_form_at_zero_H(orc):
    assert not _fp8_grad_closed_form_mismatch(orc)


@pytest.mark.parametrize("cap,tau", [(0.0, 1.0), (30.0, 7.5), (6.0, 0.7)])
def test_fp8_gradients_within_the_e5m2_rounding_bound(orc, cap, tau):
    """On ordinary inputs the FP8-gradient dH and dW_c differ from the
    exact-G gradients on the same rounded operands by no more than the e5m2
    rounding bound: half a unit in the last place (2^-3 relative for normals,
    2^-17 absolute below 2^-14) of every G8 entry, scaled back, times the
    operand (plus fp32 slack); and they do differ."""
    T, V, D, C, seed, scale = 24, 300, 32, 80, 34, 0.5
    x, C = _case(T, V, D, C, seed)
    a = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, seed, scale, grads=True,
                               cap=cap, tau=tau)
    b = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, seed, scale, grads=False,
                               cap=cap, tau=tau)
    cand, slot = a["cand"], a["slot"]
    Hq, Wq, _, _ = orc.fp8_inputs(x["H"], x["W"], cand)
    H64 = synth.bf16_bits_to_f32(Hq).astype(np.float64)
    Wc64 = synth.bf16_bits_to_f32(Wq[cand]).astype(np.float64)
    S = H64 @ Wc64.T
    Z = cap / (1.0 + np.exp(-S / tau)) if cap else S
    dz = Z * (cap - Z) / (cap * tau) if cap else np.ones_like(S)
    P = np.exp(Z - a["lse"].astype(np.float64)[:, None])
    G = P.copy()
    G[np.arange(T), slot] -= 1.0
    G *= dz
    e = orc.g8_exponent(cap, tau)
    err = 2.0 ** -3 * np.abs(G) + 2.0 ** -(17 + e)  # half an ulp, in units of G
    slack = 1e-4
    bH = abs(scale) * ((err + slack * np.abs(G)) @ np.abs(Wc64))
    bW = abs(scale) * ((err + slack * np.abs(G)).T @ np.abs(H64))
    assert np.all(np.abs(a["dH"] - b["dH"]) <= bH + 1e-9)
    assert np.all(np.abs(a["dWc"] - b["dWc"]) <= bW + 1e-9)
    assert not np.array_equal(a["dH"], b["dH"])
    np.testing.assert_array_equal(a["loss"], b["loss"])


def test_fp8_head_is_the_plain_loss_on_grid_inputs(orc):
    """Inputs already on the scaled e4m3 grid are left as they are, so the FP8
    head gives the plain head's results on them bit for bit; on ordinary bf16
    inputs it rounds every operand to 4 significant bits."""
    T, V, D, C = 40, 500, 32, 120
    x, C = _case(T, V, D, C, 22)
    Hq, _ = orc.quantize_e4m3(x["H"])
    cand, _, _ = orc.build_candidates(x["targets"], V, C, 22)
    Wq_rows, _ = orc.quantize_e4m3(x["W"][cand])
    W2 = x["W"].copy()
    W2[cand] = Wq_rows
    a = orc.loss_and_grads_fp8(Hq, W2, x["targets"], C, 22, 0.5)
    b = orc.loss_and_grads(Hq, W2, x["targets"], C, 22, 0.5)
    for k in ("loss", "lse", "dH", "dW"):
        np.testing.assert_array_equal(a[k], b[k])
    vals = synth.bf16_bits_to_f32(Hq) * 2.0 ** a["eH"]
    assert np.all([orc.round_e4m3(float(v)) == v for v in vals.ravel()[:500]])
    c = orc.loss_and_grads_fp8(x["H"], x["W"], x["targets"], C, 22, 0.5)
    d = orc.loss_and_grads(x["H"], x["W"], x["targets"], C, 22, 0.5)
    assert not np.array_equal(c["loss"], d["loss"])
    np.testing.assert_allclose(c["loss"], d["loss"], rtol=0.05)
