"""The candidate kernel's rarely taken branches, against the oracle.

With the default tie capacity the selected bin of the first 8-bit radix digit
is ranked directly on every workload here, so the deeper digits, the tie path
at a deeper digit and the last-digit path (equal 32-bit hashes taken in id
order) are not reached. Copies of the library built with a tie capacity of 0
(never rank: every digit down to the last, then the id-order path) and 1 (rank
only single-entry bins: deep digits) force them; cand, slot and U must match
the oracle bit for bit. Cases cover both marking schemes (all targets per CTA,
and one eighth per CTA merged over the cluster), vocabularies that are not a
multiple of 32, empty slices, C = V, and the largest supported vocabulary.
"""
import ctypes
import os

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

CASES = [  # T, V, C, seed
    (40000, 3001, 2500, 11), (70000, 100003, 30000, 12), (20000, 98304, 30000, 8),
    (100, 1000, 300, 1), (16384, 50304, 10240, 2), (7, 70, 20, 3), (5000, 524288, 200000, 4),
    (2000, 33, 33, 5), (300, 4097, 4000, 6), (65536, 50304, 24576, 7),
]


@pytest.fixture(scope="module", params=[0, 1])
def variant(request, tmp_path_factory):
    from sampled_softmax_output_gb300 import build as b
    out = str(tmp_path_factory.mktemp(f"ss_tie_cap_{request.param}"))
    lib = ctypes.CDLL(b.build_variant(out, [f"SS_TIE_CAP={request.param}"]))
    lib.ss_build_candidates.restype = ctypes.c_int
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.ss_build_candidates.argtypes = [p, i64, i64, i64, ctypes.c_uint64, p, p, p, p,
                                        ctypes.c_size_t, p]
    return lib


@pytest.mark.parametrize("T,V,C,seed", CASES)
def test_candidates_bit_exact(variant, orc, T, V, C, seed):
    tg = synth.zipf_targets(np.random.default_rng(seed), T, V, 1.1)
    U_ref = len(np.unique(tg))
    C = max(C, U_ref)
    cand_ref, slot_ref, U = orc.build_candidates(tg, V, C, seed)
    t = torch.from_numpy(tg).cuda()
    cand = torch.empty(C, dtype=torch.int32, device="cuda")
    slot = torch.empty(T, dtype=torch.int32, device="cuda")
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    Uh = ctypes.c_int32(-1)
    rc = variant.ss_build_candidates(t.data_ptr(), T, V, C, seed, cand.data_ptr(), slot.data_ptr(),
                                     ctypes.byref(Uh), ws.data_ptr(), ws.numel(), None)
    assert rc == 0
    assert Uh.value == U
    np.testing.assert_array_equal(cand.cpu().numpy(), cand_ref)
    np.testing.assert_array_equal(slot.cpu().numpy(), slot_ref)
