"""Seeded synthetic inputs for the sampled-softmax loss.

This module only draws numbers: hidden states H, the output-embedding matrix W,
and the batch's target token ids. It holds none of the loss's arithmetic, and it
is the one piece of code that both the CPU oracle's tests and the CUDA path's
tests/bench use, so that both sides see bit-identical inputs.

Workload shapes follow the NanoGPT speedrun setting the pages describe: a
GPT-2 sized head with model width D = 768 and a padded vocabulary of V = 50,304
("NanoGPT Training Record: Technical Optimizations & Speed", section "The
NanoGPT Benchmark and Speedrun Definition"), and candidate-set sizes taken from
the schedule given there in "Key Optimizations and Ablation Table Results"
(10,240 / 14,336 / 24,576 / 50,304). The pages use FineWeb batches; none are
available here, so token ids are drawn from a truncated Zipf law, which has the
heavy-headed frequency profile of natural-language tokens.

Value recipe (all seeded with numpy's PCG64 ``default_rng(seed)``, drawn in
this order):
  * H  ~ N(0, 1), float32 rounded to bf16 (round to nearest even), shape [T, D]
  * W  ~ N(0, 0.02^2), float32 rounded to bf16, shape [V, D]
  * targets: rank k in 1..V with p(k) proportional to k^-s, by inverse CDF of
    uniform draws; token id = k - 1 (optionally sent through a fixed seeded
    permutation of the ids so that frequent ids are not row-contiguous).
bf16 values are carried as uint16 bit patterns (numpy has no bf16 type).
"""
from __future__ import annotations

import dataclasses

import numpy as np

D_MODEL = 768
VOCAB = 50304


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    C: int
    V: int = VOCAB
    D: int = D_MODEL
    zipf_s: float = 1.1
    seed: int = 0


# The five workloads: a small latency case, the three sampled phases of the
# candidate schedule, and the final full-vocabulary phase.
WORKLOADS = {
    1: Workload("T256_C4096", T=256, C=4096, zipf_s=1.1, seed=0),
    2: Workload("T16384_C10240", T=16384, C=10240, zipf_s=1.1, seed=1),
    3: Workload("T32768_C14336", T=32768, C=14336, zipf_s=1.1, seed=2),
    4: Workload("T65536_C24576", T=65536, C=24576, zipf_s=1.0, seed=3),
    5: Workload("T65536_C50304", T=65536, C=50304, zipf_s=1.1, seed=4),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def zipf_targets(rng: np.random.Generator, T: int, V: int, s: float,
                 permute_seed: int | None = None) -> np.ndarray:
    """T token ids from a Zipf(s) law truncated to V ranks (id = rank - 1)."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    p = ranks ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    u = rng.random(T)
    ids = np.searchsorted(cdf, u, side="right")
    ids = np.minimum(ids, V - 1).astype(np.int32)
    if permute_seed is not None:
        perm = np.random.default_rng(permute_seed).permutation(V).astype(np.int32)
        ids = perm[ids]
    return ids


def make_inputs(T: int, V: int, D: int, zipf_s: float = 1.1, seed: int = 0,
                permute_seed: int | None = None, h_std: float = 1.0,
                w_std: float = 0.02) -> dict:
    """Draw (H, W, targets) for one batch. H and W are uint16 bf16 bit patterns."""
    rng = np.random.default_rng(seed)
    H = f32_to_bf16_bits(rng.standard_normal((T, D), dtype=np.float32) * np.float32(h_std))
    W = f32_to_bf16_bits(rng.standard_normal((V, D), dtype=np.float32) * np.float32(w_std))
    targets = zipf_targets(rng, T, V, zipf_s, permute_seed)
    return {"H": H, "W": W, "targets": targets}


def workload_inputs(w: Workload, T: int | None = None) -> dict:
    """Inputs for a named workload (optionally with fewer tokens, same seed)."""
    return make_inputs(T if T is not None else w.T, w.V, w.D, w.zipf_s, w.seed)


def uniform_targets(T: int, V: int, seed: int) -> np.ndarray:
    """Uniform token ids (used by edge-case tests)."""
    return np.random.default_rng(seed).integers(0, V, size=T, dtype=np.int64).astype(np.int32)
