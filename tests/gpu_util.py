"""Helpers for the GPU parity tests: device copies of the seeded inputs, one C-ABI GEMM
call with sentinel-filled output and trailing guards, and the tolerance checks.

Numerical protocol after the split-K report ("Consecutive-B split-K NAX GEMM", Contract
and numerical coverage): outputs start at 7, 64 trailing guard elements hold 11, input
allocations have exact extents, and results are compared with FP64 dot products over
the BF16-rounded inputs.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth
from oracle import gemm as og

SENTINEL = 7.0
GUARD = 11.0
N_GUARD = 64
# Pass criteria: max |err| <= 2e-2 * max(1, |ref|) per element and relative Frobenius error
# <= 5e-3, here applied to the whole matrix and to every 128 x 128 tile.
ABS_TOL = 2e-2
FRO_TOL = 5e-3


def to_dev(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


@functools.lru_cache(maxsize=8)
def inputs(w: synth.Workload):
    return synth.make_inputs(w)


@functools.lru_cache(maxsize=4)
def reference(w: synth.Workload):
    A_bits, B_bits = inputs(w)
    return og.ref_gemm(A_bits, B_bits, w.layout)


def new_workspace(sk, M, N, K, sms, sched, red, dev):
    nbytes = sk.sk_workspace_size(M, N, K, sms, sched, red)
    return torch.zeros(nbytes, dtype=torch.uint8, device=dev), nbytes


def gemm(sk, A, B, M, N, K, layout, sched, red, sms, out, dev, ws=None, **debug):
    """Run one GEMM; return (C [M,N] as float64 numpy, guards ok, workspace, status)."""
    if ws is None:
        ws = new_workspace(sk, M, N, K, sms, sched, red, dev)
    buf, nbytes = ws
    dt = torch.float32 if out == "f32" else torch.bfloat16
    C = torch.full((M * N + N_GUARD,), SENTINEL, dtype=dt, device=dev)
    C[M * N:] = GUARD
    stream = torch.cuda.current_stream(dev)
    code = sk.SK_F32 if out == "f32" else sk.SK_BF16
    lay = sk.SK_NN if layout == "NN" else sk.SK_NT
    if debug:
        sk.sk_gemm_debug(A, B, C, code, M, N, K, lay, sched, red, sms, buf, nbytes, stream, **debug)
    else:
        sk.sk_gemm(A, B, C, code, M, N, K, lay, sched, red, sms, buf, nbytes, stream)
    status = sk.sk_status(buf, stream)
    host = C.float().cpu().numpy().astype(np.float64)
    guards_ok = bool(np.all(host[M * N:] == GUARD))
    return host[:M * N].reshape(M, N), guards_ok, ws, status


def close_report(got: np.ndarray, ref: np.ndarray):
    err = np.abs(got - ref)
    scaled = float((err / np.maximum(1.0, np.abs(ref))).max()) if got.size else 0.0
    nref = float(np.linalg.norm(ref))
    fro = float(np.linalg.norm(got - ref)) / nref if nref > 0 else float(np.linalg.norm(got))
    worst_tile = 0.0
    M, N = got.shape
    for i in range(0, M, 128):
        for j in range(0, N, 128):
            r = ref[i:i + 128, j:j + 128]
            d = got[i:i + 128, j:j + 128] - r
            nr = float(np.linalg.norm(r))
            worst_tile = max(worst_tile, float(np.linalg.norm(d)) / nr if nr > 0 else float(np.linalg.norm(d)))
    return {"max_scaled_err": scaled, "rel_fro": fro, "worst_tile_rel_fro": worst_tile}


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    rep = close_report(got, ref)
    assert rep["max_scaled_err"] <= ABS_TOL, (what, rep)
    assert rep["rel_fro"] <= FRO_TOL, (what, rep)
    assert rep["worst_tile_rel_fro"] <= FRO_TOL, (what, rep)
    return rep


def sample_rows(M: int, n: int = 48, seed: int = 0):
    rng = np.random.default_rng(seed)
    rows = set(int(x) for x in rng.choice(M, size=min(n, M), replace=False))
    rows |= {0, min(127, M - 1), min(128, M - 1), M - 1}
    return sorted(rows)
