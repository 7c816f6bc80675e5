"""GEMM oracle: C = A . B as FP64 dot products over the BF16-rounded inputs.

TEST INFRASTRUCTURE (see the package docstring). The method only reorders FP32
additions ("Split-K and Stream-K: The Last Wave of a GEMM", Case 3 and The trap),
so every schedule is judged against one plain definition:
    C_ref[i, j] = sum_k double(A[i, k]) * double(B[k, j])
over the inputs exactly as rounded to BF16 ("Consecutive-B split-K NAX GEMM",
Contract and numerical coverage, which compares every slab with FP64 sums taken
over the inputs after their rounding to the storage type; the Case 3 driver of the
first page also checks against an FP64 product). The FP64 matrix product of NumPy is the library primitive for the
sum; no blocking or reordering is added here.

Layouts (split-K report, Contract): A is [M, K] row-major. In NN, B is [K, N]
row-major; in NT, B is stored [N, K] row-major, so C = A . B_stored^T.
"""
from __future__ import annotations

import numpy as np

BLK_K = 64


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float64: a bfloat16 is the upper 16 bits of an
    IEEE binary32, so shifting left by 16 gives the float32 of the same value."""
    u32 = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def operand_b(B_bits: np.ndarray, layout: str) -> np.ndarray:
    """B as a [K, N] float64 matrix for either storage layout."""
    B = bf16_to_f64(B_bits)
    if layout == "NN":
        return B
    if layout == "NT":
        return B.T
    raise ValueError(layout)


def ref_gemm(A_bits: np.ndarray, B_bits: np.ndarray, layout: str = "NN") -> np.ndarray:
    """FP64 C = A . B over the BF16 inputs."""
    return bf16_to_f64(A_bits) @ operand_b(B_bits, layout)


def ref_rows(A_bits: np.ndarray, B_bits: np.ndarray, layout: str, rows) -> np.ndarray:
    """FP64 rows `rows` of C only (for spot checks of large products)."""
    rows = np.asarray(rows)
    return bf16_to_f64(A_bits[rows]) @ operand_b(B_bits, layout)


def split_ranges(K: int, splits: int):
    """K ranges of the Split-K slabs, in elements: split j covers k-iterations
    [j*chunk, min((j+1)*chunk, iters)) with chunk = ceil(iters / splits) and iters =
    ceil(K / 64) (first page, Case 2 split_k); the final split is clamped at K (split-K
    report, Contract). Empty trailing splits are dropped."""
    iters = -(-K // BLK_K)
    chunk = -(-iters // splits)
    out = []
    j = 0
    while j * chunk < iters:
        out.append((j * chunk * BLK_K, min((j + 1) * chunk * BLK_K, K)))
        j += 1
    return out


def ref_split_partials(A_bits: np.ndarray, B_bits: np.ndarray, layout: str, splits: int):
    """FP64 partial slabs P[j] = A[:, Kj] . B[Kj, :], shape [s_eff, M, N]
    (split-K report, Contract: every partial slab checked against F64 dot products)."""
    A = bf16_to_f64(A_bits)
    B = operand_b(B_bits, layout)
    return np.stack([A[:, k0:k1] @ B[k0:k1, :] for k0, k1 in split_ranges(A.shape[1], splits)])
