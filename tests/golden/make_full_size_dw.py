"""Writes the stored oracle values for the full-size parity check of dW.

    python tests/golden/make_full_size_dw.py [workload ...]   (default: 3 4 5)

For each of the three large workloads (T32768_C14336, T65536_C24576,
T65536_C50304) this script calls only the CPU oracle (``oracle/``) on the
seeded synthetic inputs of ``synth``:

  * the candidate set, the full-batch forward (lse of every token) and the
    mean per-token loss;
  * the candidate-row gradients dW_c[j] of six candidate columns j -- both
    ends of the set, the last target (U - 1) and the first negative (U), the
    first column of the last 256-wide tile, and the middle -- with the
    backward scaled by 1 / T (the gradient of the mean loss).

The definition being evaluated: the lm_head cross-entropy restricted to the
batch's shared candidate set, in the forward and the backward ("NanoGPT
Training Record: Technical Optimizations & Speed", section "Key Optimizations
and Ablation Table Results"; the README's technique list, "sampled softmax
over a shared candidate set"). The candidate sizes are that section's
schedule (14,336, 24,576, and the full 50,304 for the final steps).

The output, ``full_size_dw_<workload>.txt``, is plain text: a header of
``# key value`` lines, then one line per column, ``j v[0] ... v[D-1]``.
The full-batch forward takes minutes on a few host cores; the file is
written once and committed.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def columns(U: int, C: int) -> list[int]:
    cols = {0, U - 1, min(U, C - 1), (C - 1) // 256 * 256, C // 2, C - 1}
    return sorted(c for c in cols if 0 <= c < C)


def path_for(name: str) -> str:
    return os.path.join(HERE, f"full_size_dw_{name}.txt")


def write(wid: int) -> str:
    w = synth.WORKLOADS[wid]
    x = synth.workload_inputs(w)
    t0 = time.time()
    cand, slot, U = oracle.build_candidates(x["targets"], w.V, w.C, w.seed)
    loss, lse = oracle.forward(x["H"], x["W"], cand, slot)
    cols = columns(U, w.C)
    scale = 1.0 / w.T
    rows = oracle.backward_dWc(x["H"], x["W"], cand, slot, lse, scale, cols=np.array(cols))
    out = path_for(w.name)
    with open(out, "w") as f:
        f.write(f"# written by: python tests/golden/make_full_size_dw.py {wid}\n")
        f.write("# values: CPU oracle (fp32), dW_c rows of the listed candidate columns, "
                "backward scale 1/T\n")
        f.write(f"# workload {w.name}\n# T {w.T}\n# V {w.V}\n# C {w.C}\n# D {w.D}\n")
        f.write(f"# seed {w.seed}\n# zipf_s {w.zipf_s}\n# U {U}\n")
        f.write(f"# mean_loss {float(np.mean(loss.astype(np.float64))):.10e}\n")
        f.write(f"# mean_lse {float(np.mean(lse.astype(np.float64))):.10e}\n")
        f.write("# columns " + " ".join(str(c) for c in cols) + "\n")
        f.write("# cand_of_columns " + " ".join(str(int(cand[c])) for c in cols) + "\n")
        for c, r in zip(cols, rows):
            f.write(f"{c} " + " ".join(f"{v:.8e}" for v in r.astype(np.float32)) + "\n")
    print(f"{w.name}: U={U} columns={cols} ({time.time() - t0:.0f} s) -> {out}")
    return out


def read(name: str) -> dict:
    """Parse a stored file: header keys, the column list and the rows [n, D]."""
    meta, cols, rows = {}, [], []
    with open(path_for(name)) as f:
        for line in f:
            if line.startswith("#"):
                parts = line[1:].split()
                if len(parts) >= 2:
                    meta[parts[0]] = parts[1:]
                continue
            vals = line.split()
            cols.append(int(vals[0]))
            rows.append(np.array([float(v) for v in vals[1:]], dtype=np.float64))
    return {"meta": meta, "cols": np.array(cols), "rows": np.stack(rows)}


if __name__ == "__main__":
    oracle.build()
    for a in (sys.argv[1:] or ["3", "4", "5"]):
        write(int(a))
