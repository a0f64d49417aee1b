"""Shared helpers of the GPU tests: run the CUDA path through the Python binding
(which calls the C ABI) on numpy inputs drawn by ``synth``, and the tolerance
checks the tests use.

Tolerances (per token for the loss, relative Frobenius norm for the gradients):
  loss, lse : 1e-3 relative  -- the logits are fp32 sums of exact bf16 products,
              exponentials use the hardware ex2 (relative error ~2^-22), so the
              real error is ~1e-6; 1e-3 is the acceptance bound.
  dH, dW    : 2e-2 relative Frobenius -- G = scale * (P - Y) is rounded to bf16
              (relative 2^-9 per element) before the two gradient GEMMs, and dH
              is stored in bf16; the expected error is ~2e-3.
"""
from __future__ import annotations

import numpy as np
import torch

LOSS_RTOL = 1e-3
GRAD_RTOL = 2e-2


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run_gpu(ss, x: dict, C: int, seed: int, scale: float = 1.0, dW0: np.ndarray | None = None,
            accumulate: bool = False, ws: torch.Tensor | None = None, cap: float = 0.0,
            tau: float = 1.0) -> dict:
    H = to_dev_bf16(x["H"])
    W = to_dev_bf16(x["W"])
    T, D = H.shape
    V = W.shape[0]
    targets = torch.from_numpy(np.ascontiguousarray(x["targets"], np.int32)).cuda()
    if ws is None:
        ws = ss.workspace(T, V, C, D)
    cand, slot, U = ss.build_candidates(targets, V, C, seed, ws, return_U=True)
    loss, lse = ss.forward(H, W, cand, slot, ws, cap=cap, tau=tau)
    dW = (torch.from_numpy(np.ascontiguousarray(dW0, np.float32)).cuda() if dW0 is not None
          else torch.zeros(V, D, dtype=torch.float32, device="cuda"))
    dH, dW = ss.backward(H, W, cand, slot, lse, ws, scale=scale, accumulate=accumulate, dW=dW,
                         cap=cap, tau=tau)
    torch.cuda.synchronize()
    status, _ = ss.read_status(ws)
    return {"cand": cand.cpu().numpy(), "slot": slot.cpu().numpy(), "U": U,
            "loss": loss.cpu().numpy(), "lse": lse.cpu().numpy(),
            "dH": dH.float().cpu().numpy(), "dW": dW.cpu().numpy(), "status": status}


def run_gpu_step(ss, x: dict, C: int, seed: int, scale: float = 1.0,
                 dW0: np.ndarray | None = None, accumulate: bool = False,
                 ws: torch.Tensor | None = None, cap: float = 0.0, tau: float = 1.0) -> dict:
    """The same batch through the one-call entry point ss_step (with the plain
    head it keeps the forward's probabilities for the backward)."""
    H = to_dev_bf16(x["H"])
    W = to_dev_bf16(x["W"])
    T, D = H.shape
    V = W.shape[0]
    targets = torch.from_numpy(np.ascontiguousarray(x["targets"], np.int32)).cuda()
    if ws is None:
        ws = ss.workspace(T, V, C, D)
    dW = (torch.from_numpy(np.ascontiguousarray(dW0, np.float32)).cuda() if dW0 is not None
          else torch.zeros(V, D, dtype=torch.float32, device="cuda"))
    out = ss.step(H, W, targets, C, seed, ws, scale=scale, accumulate=accumulate, dW=dW, cap=cap,
                  tau=tau)
    torch.cuda.synchronize()
    status, U = ss.read_status(ws)
    return {"cand": out["cand"].cpu().numpy(), "slot": out["slot"].cpu().numpy(), "U": U,
            "loss": out["loss"].cpu().numpy(), "lse": out["lse"].cpu().numpy(),
            "dH": out["dH"].float().cpu().numpy(), "dW": out["dW"].cpu().numpy(),
            "status": status}


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def assert_loss_close(got, ref, atol=1e-5):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > LOSS_RTOL * np.abs(ref) + atol
    assert not bad.any(), f"{bad.sum()} tokens off; worst {err.max():.3e} at {int(err.argmax())}"
