"""The pass criteria catch the mistakes a broken schedule would make.

Mistakes are planted in the oracle's own result on the CPU (never in the CUDA path): a
lost producer partial (one 64-deep k-iteration range of one tile missing), every split
tile losing its peers' partials, a tile copied to the wrong place, and a transposed
operand. Each must fail the checks the GPU tests apply; an honest BF16 rounding of the
result must pass.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as og
from oracle import schedule as S

from . import gpu_util as U


@pytest.fixture(scope="module")
def case():
    w = synth.Workload("t", 512, 384, 1024, "NN", "normal_sqrtk", 12)
    A_bits, B_bits = synth.make_inputs(w)
    A = og.bf16_to_f64(A_bits)
    B = og.bf16_to_f64(B_bits)
    return w, A, B, A @ B


def _fails(got, ref):
    with pytest.raises(AssertionError):
        U.assert_close(got, ref)


def test_honest_bf16_rounding_passes(case):
    _, _, _, ref = case
    got = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).double().numpy()
    U.assert_close(got, ref)


def test_lost_partial_fails(case):
    w, A, B, ref = case
    got = ref.copy()
    # tile (1, 2) loses k-iterations 3..5 (a producer's partial never added)
    r, c = 128, 256
    got[r:r + 128, c:c + 128] -= A[r:r + 128, 192:384] @ B[192:384, c:c + 128]
    _fails(got, ref)


def test_zeroed_producer_stores_fail(case):
    # Every split tile keeps only its owner's segment (the numerical control of the
    # split-K report: zero the partial store and every case must fail).
    w, A, B, ref = case
    plan = S.build_plan(w.M, w.N, w.K, 5, S.STREAMK)
    got = np.zeros_like(ref)
    for s in plan.segments():
        if s.role in (S.FULL, S.OWNER):
            r, c = (s.tile // plan.tiles_n) * 128, (s.tile % plan.tiles_n) * 128
            k0, k1 = s.k_begin * 64, s.k_end * 64
            got[r:r + 128, c:c + 128] += A[r:r + 128, k0:k1] @ B[k0:k1, c:c + 128]
    _fails(got, ref)


def test_misplaced_tile_fails(case):
    _, _, _, ref = case
    got = ref.copy()
    got[0:128, 0:128] = ref[128:256, 0:128]
    _fails(got, ref)


def test_transposed_operand_fails():
    A_bits, B_bits = synth.make_inputs(synth.Workload("t", 256, 256, 256, "NT", "normal", 2))
    ref = og.ref_gemm(A_bits, B_bits, "NT")
    _fails(og.ref_gemm(A_bits, B_bits, "NN"), ref)
