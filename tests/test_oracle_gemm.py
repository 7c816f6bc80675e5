"""Pins for the FP64 GEMM oracle and for the seeded inputs.

The oracle's GEMM is C = A . B in FP64 over BF16-rounded inputs ("Consecutive-B split-K
NAX GEMM", Contract and numerical coverage). Pins, each independent of the oracle's own
code: BF16 decoding checked on bit patterns fixed by the bfloat16 format; brute-force
correctly rounded dot products (math.fsum) on small non-square NN and NT cases, which fail
on a transposed or swapped operand; exact integer arithmetic; the zero first row and x4
last row of the small-M workloads; and the Split-K slabs covering K exactly once with the
final split clamped.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import gemm as G


def test_bf16_decode_known_patterns():
    # bfloat16 = sign, 8-bit exponent (bias 127), 7-bit fraction.
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xC000, 0x4049, 0x0001, 0x0080, 0x7F7F, 0x3E20],
                    dtype=np.uint16)
    want = [0.0, -0.0, 1.0, -2.0, 3.140625, 2.0 ** -133, 2.0 ** -126,
            (2 - 2 ** -7) * 2.0 ** 127, 0.15625]
    got = G.bf16_to_f64(bits)
    assert list(got) == want
    assert math.copysign(1.0, got[1]) == -1.0


def test_bf16_rounding_matches_torch():
    # Input rounding against a library routine: torch's float32 -> bfloat16 cast (RNE).
    x = synth.normal(synth.stream_key(11, 0), 100000).astype(np.float32) * 37.0
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 65504.0]  # ties and a big value
    mine = synth.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_generator_known_values():
    # SplitMix64 reference value: mix64 of 0x9E3779B97F4A7C15 (first output for seed 0).
    assert int(synth.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF
    u = synth.uniform01(synth.stream_key(3, 1), 0, 200000)
    assert 0.0 <= u.min() and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.01
    z = synth.normal(synth.stream_key(3, 0), 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def _fsum_gemm(A, B):
    """Correctly rounded dot products, one Python loop per output."""
    M, K = A.shape
    N = B.shape[1]
    return np.array([[math.fsum(float(A[i, k]) * float(B[k, j]) for k in range(K)) for j in range(N)]
                     for i in range(M)])


@pytest.mark.parametrize("layout", ["NN", "NT"])
def test_ref_gemm_vs_bruteforce(layout):
    M, N, K = 7, 5, 37
    w = synth.Workload("t", M, N, K, layout, "normal", 21)
    A_bits, B_bits = synth.make_inputs(w)
    A = G.bf16_to_f64(A_bits)
    Bs = G.bf16_to_f64(B_bits)
    Bkn = Bs if layout == "NN" else np.array([[Bs[j, k] for j in range(N)] for k in range(K)])
    want = _fsum_gemm(A, Bkn)
    got = G.ref_gemm(A_bits, B_bits, layout)
    assert got.shape == (M, N)
    bound = K * 2.0 ** -52 * np.abs(A) @ np.abs(Bkn)
    assert np.all(np.abs(got - want) <= bound)


def test_ref_gemm_nt_is_not_nn():
    # A square case where reading the stored [N,K] matrix as [K,N] gives a different answer.
    A_bits, B_bits = synth.small_int_inputs(4, 4, 4, "NT", 5)
    nn = G.ref_gemm(A_bits, B_bits, "NN")
    nt = G.ref_gemm(A_bits, B_bits, "NT")
    A = G.bf16_to_f64(A_bits).astype(int).tolist()
    B = G.bf16_to_f64(B_bits).astype(int).tolist()
    want = [[sum(A[i][k] * B[j][k] for k in range(4)) for j in range(4)] for i in range(4)]
    assert nt.tolist() == want
    assert not np.array_equal(nn, nt)


@pytest.mark.parametrize("layout", ["NN", "NT"])
def test_integer_exact(layout):
    M, N, K = 9, 11, 300
    A_bits, B_bits = synth.small_int_inputs(M, N, K, layout, 8)
    A = G.bf16_to_f64(A_bits).astype(np.int64)
    B = G.bf16_to_f64(B_bits).astype(np.int64)
    assert A.min() >= -4 and A.max() <= 4
    Bkn = B if layout == "NN" else B.T
    want = [[int(sum(int(A[i, k]) * int(Bkn[k, j]) for k in range(K))) for j in range(N)] for i in range(M)]
    assert G.ref_gemm(A_bits, B_bits, layout).tolist() == want


def test_zero_first_row_and_scaled_last_row():
    w = synth.Workload("t", 6, 8, 96, "NT", "normal", 2, zero_first_row=True, scale_last_row=4.0)
    A_bits, B_bits = synth.make_inputs(w)
    C = G.ref_gemm(A_bits, B_bits, "NT")
    assert np.all(C[0] == 0.0) and not np.any(np.signbit(C[0]))
    plain = synth.Workload("t", 6, 8, 96, "NT", "normal", 2)
    A2, B2 = synth.make_inputs(plain)
    assert np.array_equal(B2, B_bits)
    assert np.array_equal(C[-1], 4.0 * G.ref_gemm(A2, B2, "NT")[-1])


def test_split_ranges():
    assert G.split_ranges(2048, 8) == [(256 * j, 256 * (j + 1)) for j in range(8)]
    assert G.split_ranges(2048, 3) == [(0, 704), (704, 1408), (1408, 2048)]
    # K = 320 -> 5 iterations; s = 4 -> chunk 2 -> [0,128) [128,256) [256,320), 4th split empty.
    assert G.split_ranges(320, 4) == [(0, 128), (128, 256), (256, 320)]
    # ragged K: the final split is clamped at K.
    assert G.split_ranges(200, 2) == [(0, 128), (128, 200)]
    for K in range(1, 700, 13):
        for s in range(1, 9):
            r = G.split_ranges(K, s)
            if s > -(-K // 64):
                continue
            assert r[0][0] == 0 and r[-1][1] == K
            assert all(r[i][1] == r[i + 1][0] and r[i][0] < r[i][1] for i in range(len(r) - 1))


def test_split_partials_sum_and_slabs():
    M, N, K = 5, 6, 200
    A_bits, B_bits = synth.small_int_inputs(M, N, K, "NT", 4)
    P = G.ref_split_partials(A_bits, B_bits, "NT", 2)
    assert P.shape == (2, M, N)
    assert np.array_equal(P.sum(axis=0), G.ref_gemm(A_bits, B_bits, "NT"))
    A = G.bf16_to_f64(A_bits).astype(np.int64)
    B = G.bf16_to_f64(B_bits).astype(np.int64)
    for j, (k0, k1) in enumerate(G.split_ranges(K, 2)):
        want = [[int(sum(int(A[i, k]) * int(B[n, k]) for k in range(k0, k1))) for n in range(N)]
                for i in range(M)]
        assert P[j].tolist() == want


def test_ref_rows():
    A_bits, B_bits = synth.make_inputs(synth.Workload("t", 40, 24, 130, "NN", "normal_sqrtk", 9))
    full = G.ref_gemm(A_bits, B_bits, "NN")
    rows = [0, 7, 39]
    assert np.array_equal(G.ref_rows(A_bits, B_bits, "NN", rows), full[rows])
