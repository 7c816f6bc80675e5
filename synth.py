"""Seeded synthetic inputs for the work-decomposed BF16 GEMM.

This module holds only input generation: a counter-based random generator, the
value distributions the workloads use, BF16 rounding of the generated inputs,
and the list of workloads (shapes, seeds, value recipe). It holds none of the
GEMM or scheduling arithmetic. Both the CPU oracle (through the tests and the
benchmark) and the CUDA path receive the same BF16 bit patterns from here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) in counter form: value i of stream `key` is
mix64(key + (i + 1) * 0x9E3779B97F4A7C15). Uniforms take the top 53 bits.
Normals use the Box-Muller transform on pairs of uniforms.

BF16 rounding: a float32 is rounded to bfloat16 (1 sign, 8 exponent, 7
fraction bits) to nearest, ties to even, by integer arithmetic on its bits
(IEEE 754 roundTiesToEven applied to the upper 16 bits). Generated values are
finite and far from the float32 overflow threshold.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def mix64_scalar(x: int) -> int:
    """SplitMix64 finaliser on one 64-bit integer (used to derive stream keys)."""
    with np.errstate(over="ignore"):
        return int(_mix64(np.array([x & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def stream_key(seed: int, tensor: int) -> int:
    """Key of the random stream for tensor `tensor` (0 = A, 1 = B) of workload seed `seed`."""
    return mix64_scalar(seed * 4 + tensor + 1)


def splitmix64(key: int, start: int, n: int) -> np.ndarray:
    """Values start .. start+n-1 of the counter-based SplitMix64 stream `key` (uint64)."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(key) + ctr * _GAMMA
        return _mix64(z)


def uniform01(key: int, start: int, n: int) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of each stream value."""
    x = splitmix64(key, start, n) >> np.uint64(11)
    return x.astype(np.float64) * (2.0 ** -53)


def normal(key: int, n: int) -> np.ndarray:
    """n standard normals by Box-Muller: pair p uses stream values 2p and 2p+1."""
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2
    for p0 in range(0, pairs, _CHUNK):
        p1 = min(pairs, p0 + _CHUNK)
        x = splitmix64(key, 2 * p0, 2 * (p1 - p0)) >> np.uint64(11)
        u1 = (x[0::2].astype(np.float64) + 1.0) * (2.0 ** -53)   # (0, 1]
        u2 = x[1::2].astype(np.float64) * (2.0 ** -53)           # [0, 1)
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * math.pi * u2)
        z[1::2] = r * np.sin(2.0 * math.pi * u2)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo]
    return out


def normal_range(key: int, start: int, n: int) -> np.ndarray:
    """Values start .. start+n-1 of the stream `normal(key, .)` (start even), without drawing
    the ones before: pair p still uses stream values 2p and 2p+1."""
    if start % 2:
        raise ValueError("start must be even")
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2
    p_base = start // 2
    for p0 in range(0, pairs, _CHUNK):
        p1 = min(pairs, p0 + _CHUNK)
        x = splitmix64(key, 2 * (p_base + p0), 2 * (p1 - p0)) >> np.uint64(11)
        u1 = (x[0::2].astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = x[1::2].astype(np.float64) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * math.pi * u2)
        z[1::2] = r * np.sin(2.0 * math.pi * u2)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo]
    return out


def uniform(key: int, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = lo + (hi - lo) * uniform01(key, s, e - s)
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (to nearest, ties to even); return the uint16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16).reshape(f.shape)


@dataclass(frozen=True)
class Workload:
    """One GEMM input recipe: C[M,N] = A[M,K] . B, B stored [K,N] (NN) or [N,K] (NT)."""
    name: str
    M: int
    N: int
    K: int
    layout: str = "NN"          # "NN" or "NT"
    dist: str = "normal_sqrtk"  # "uniform" (U[-1,1]), "normal" (N(0,1)), "normal_sqrtk" (N(0,1)/sqrt(K))
    seed: int = 0
    zero_first_row: bool = False   # A row 0 all zeros
    scale_last_row: float = 1.0    # A last row multiplied by this before rounding
    out: str = "bf16"              # C element type: "f32" or "bf16"
    extra: dict = field(default_factory=dict, compare=False)


def make_inputs(w: Workload):
    """Return (A_bits [M,K] uint16, B_bits uint16 [K,N] for NN or [N,K] for NT)."""
    M, N, K = w.M, w.N, w.K

    def draw(tensor: int, n: int) -> np.ndarray:
        key = stream_key(w.seed, tensor)
        if w.dist == "uniform":
            return uniform(key, n, -1.0, 1.0)
        z = normal(key, n)
        if w.dist == "normal_sqrtk":
            z *= 1.0 / math.sqrt(K)
        elif w.dist != "normal":
            raise ValueError(f"unknown distribution {w.dist}")
        return z

    a = draw(0, M * K).reshape(M, K)
    if w.zero_first_row and M > 0:
        a[0, :] = 0.0
    if w.scale_last_row != 1.0 and M > 1:
        a[M - 1, :] *= w.scale_last_row
    b = draw(1, K * N)
    b = b.reshape(K, N) if w.layout == "NN" else b.reshape(N, K)
    return bf16_bits(a), bf16_bits(b)


def make_row_block(w: Workload, r0: int, r1: int):
    """Rows r0 .. r1-1 of make_inputs(w)'s A, and the whole B: the inputs of one shard of a GEMM
    whose rows are split over several devices. Bit-identical to slicing make_inputs(w)[0]."""
    M, N, K = w.M, w.N, w.K
    if not 0 <= r0 <= r1 <= M:
        raise ValueError("bad row block")
    key = stream_key(w.seed, 0)
    if w.dist == "uniform":
        a = np.empty((r1 - r0) * K, dtype=np.float64)
        for s in range(0, a.size, _CHUNK):
            e = min(a.size, s + _CHUNK)
            a[s:e] = -1.0 + 2.0 * uniform01(key, r0 * K + s, e - s)
    else:
        if (r0 * K) % 2:
            a = normal(key, r1 * K)[r0 * K:]
        else:
            a = normal_range(key, r0 * K, (r1 - r0) * K)
        if w.dist == "normal_sqrtk":
            a *= 1.0 / math.sqrt(K)
        elif w.dist != "normal":
            raise ValueError(f"unknown distribution {w.dist}")
    a = a.reshape(r1 - r0, K)
    if w.zero_first_row and r0 == 0 and r1 > 0:
        a[0, :] = 0.0
    if w.scale_last_row != 1.0 and M > 1 and r0 <= M - 1 < r1:
        a[M - 1 - r0, :] *= w.scale_last_row
    kb = stream_key(w.seed, 1)
    if w.dist == "uniform":
        b = uniform(kb, K * N, -1.0, 1.0)
    else:
        b = normal(kb, K * N)
        if w.dist == "normal_sqrtk":
            b *= 1.0 / math.sqrt(K)
    b = b.reshape(K, N) if w.layout == "NN" else b.reshape(N, K)
    return bf16_bits(a), bf16_bits(b)


def small_int_inputs(M: int, N: int, K: int, layout: str, seed: int, lo: int = -4, hi: int = 4):
    """Integer-valued BF16 inputs in [lo, hi]; every partial sum of a product stays an exact float32."""
    ka, kb = stream_key(seed, 0), stream_key(seed, 1)
    span = hi - lo + 1
    a = (np.floor(uniform01(ka, 0, M * K) * span) + lo).reshape(M, K)
    b = np.floor(uniform01(kb, 0, K * N) * span) + lo
    b = b.reshape(K, N) if layout == "NN" else b.reshape(N, K)
    return bf16_bits(a), bf16_bits(b)


# The workloads: shapes, seeds and value structure of the pages' cases (toy 4-SM Stream-K
# example, the wave-quantized shape, the small-M split-K benchmark with [N,K] weights, the
# tile-count sweep, and the large and long-K shapes).
TOY = Workload("toy_128x640x256", 128, 640, 256, "NN", "uniform", 0, out="f32")
WAVEQ = Workload("waveq_2048x2432x4096", 2048, 2432, 4096, "NN", "normal_sqrtk", 1, out="bf16")
SMALLM_96 = Workload("smallm_nt_96x512x2048", 96, 512, 2048, "NT", "normal", 2,
                     zero_first_row=True, scale_last_row=4.0, out="f32")
SMALLM_256 = Workload("smallm_nt_256x512x2048", 256, 512, 2048, "NT", "normal", 3,
                      zero_first_row=True, scale_last_row=4.0, out="f32")
LARGE = Workload("large_8192x8192x8192", 8192, 8192, 8192, "NN", "normal_sqrtk", 5, out="bf16")
SKINNY = Workload("skinny_512x512x65536", 512, 512, 65536, "NN", "normal_sqrtk", 6, out="bf16")


def sweep(m: int) -> Workload:
    """Tile-count sweep point: square M = N = m (a multiple of 128), K = 4096."""
    return Workload(f"sweep_{m}x{m}x4096", m, m, 4096, "NN", "normal_sqrtk", 4, out="bf16")


SWEEP_SIZES = tuple(range(128, 4096 + 1, 128))
