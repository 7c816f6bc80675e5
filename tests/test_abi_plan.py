"""The C ABI on the host: the library loads and exports every declared entry point, and
sk_plan's work-unit map equals the oracle's bit for bit.

The kernel walks each unit's segments with the same code that writes this map, so the map
comparison checks the device's schedule too. No GPU is used here.
"""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

from oracle import schedule as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sk():
    from gemm_work_decomposition_gb300 import build
    build.build()
    import gemm_work_decomposition_gb300 as pkg
    pkg.lib()
    return pkg


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(sk_[a-z_0-9]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(sk):
    declared = _declared()
    assert {"sk_plan", "sk_plan_size", "sk_gemm", "sk_workspace_size", "sk_status", "sk_strerror",
            "sk_reduce_splits", "sk_gemm_debug"} <= declared
    lib = ctypes.CDLL(sk.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(sk.EXPORTS) == declared


def _cmp(sk, M, N, K, sms, mode, splits=1, units=0, min_iters=0, partials=0, tile=0, raster=0, swizzle=0,
         groups=0):
    sched = sk.schedule(mode, splits, units, min_iters, partials, tile, raster, swizzle, sk_groups=groups)
    try:
        want = S.plan_map(S.build_plan(M, N, K, sms, mode, splits=splits, units=units,
                                       min_iters=min_iters or 8, split_partials=partials, tile=tile,
                                       raster=raster, swizzle=swizzle, sk_groups=groups))
    except ValueError:
        with pytest.raises(sk.SkError) as e:
            sk.sk_plan(M, N, K, sms, sched)
        assert e.value.code == sk.SK_EINVAL
        return None
    got = sk.sk_plan(M, N, K, sms, sched)
    assert got.tolist() == want, (M, N, K, sms, mode, splits, units, partials, tile, raster, swizzle, groups)
    return got


def test_plan_matches_oracle_on_workloads(sk):
    cases = [
        (128, 640, 256, 4, S.DP), (128, 640, 256, 4, S.STREAMK),            # toy, forced to 4 units
        (2048, 2432, 4096, 148, S.DP), (2048, 2432, 4096, 148, S.STREAMK),  # wave-quantized
        (2048, 2432, 4096, 148, S.HYBRID), (2048, 2432, 4096, 152, S.HYBRID),
        (96, 512, 2048, 148, S.STREAMK), (256, 512, 2048, 148, S.STREAMK),  # small-M NT
        (96, 512, 2048, 148, S.HYBRID), (256, 512, 2048, 148, S.HYBRID),
        (8192, 8192, 8192, 148, S.HYBRID), (512, 512, 65536, 148, S.HYBRID),
        (512, 512, 65536, 148, S.STREAMK),
    ]
    for M, N, K, sms, mode in cases:
        _cmp(sk, M, N, K, sms, mode)
        if mode != S.DP:
            _cmp(sk, M, N, K, sms, mode, partials=1)  # Stream-K / hybrid: separate fixup pass
    for s in (2, 4, 8, 16):
        for M in (96, 256):
            _cmp(sk, M, 512, 2048, 148, S.SPLITK, splits=s, partials=1)
            _cmp(sk, M, 512, 2048, 148, S.SPLITK, splits=s, partials=2)
            _cmp(sk, M, 512, 2048, 148, S.SPLITK, splits=s)
    _cmp(sk, 2048, 2432, 4096, 148, S.SPLITK, splits=2)
    for m in range(128, 4097, 128):
        for tile in (0, 1, 2, 3):
            for mode in (S.DP, S.STREAMK, S.HYBRID):
                _cmp(sk, m, m, 4096, 148, mode, tile=tile)
            for s in (2, 4):
                _cmp(sk, m, m, 4096, 148, S.SPLITK, splits=s, tile=tile)
    for tile in (1, 2, 3):
        for M, N, K, sms, mode in cases:
            _cmp(sk, M, N, K, sms, mode, tile=tile)


def test_plan_rasterization(sk):
    # The tile rows of the map carry each tile's grid position, so the host's tile_coords
    # (the same code the kernels run) is checked against the oracle here.
    for M, N, K in [(640, 384, 128), (2048, 2432, 4096), (8192, 8192, 8192), (129, 1000, 72), (512, 512, 65536)]:
        for tile in (0, 2):
            for raster in (0, 1):
                for sw in (0, 1, 2, 3, 4, 8, 256):
                    for mode in (S.DP, S.STREAMK, S.HYBRID):
                        _cmp(sk, M, N, K, 148, mode, tile=tile, raster=raster, swizzle=sw)
    for bad in ((2, 0), (-1, 0), (0, -1), (0, 257)):
        with pytest.raises(sk.SkError):
            sk.sk_plan(128, 128, 64, 4, sk.schedule(0, raster=bad[0], swizzle=bad[1]))


def test_split_k_slices_matches_oracle(sk):
    # The CUTLASS page's Split-K factor heuristic: the C entry point equals the oracle's on a
    # grid of shapes (ragged and below one tile) and SM counts, and rejects bad sizes.
    for sms in (1, 4, 16, 132, 148, 152):
        for m in (1, 96, 127, 128, 200, 640, 1024, 1536, 2048, 2432, 4096, 8192):
            for n in (8, 128, 512, 1000, 2432, 4096):
                assert sk.sk_split_k_slices(m, n, 4096, sms) == S.calculate_split_k(m, n, 4096, sms), (m, n, sms)
    for bad in ((0, 128, 128, 148), (128, 0, 128, 148), (128, 128, 128, 0)):
        with pytest.raises(sk.SkError) as e:
            sk.sk_split_k_slices(*bad)
        assert e.value.code == sk.SK_EINVAL


def test_overlap_is_a_launch_option(sk):
    # The overlapped launch changes how the kernels are launched, not what they compute:
    # the plan and the workspace size are the same either way.
    for M, N, K in [(2048, 2432, 4096), (512, 512, 65536), (96, 512, 2048), (300, 264, 520)]:
        for tile in (0, 2):
            for mode, splits, partials in ((S.DP, 1, 0), (S.STREAMK, 1, 0), (S.HYBRID, 1, 1), (S.SPLITK, 2, 1),
                                           (S.SPLITK, 3, 2)):
                a = sk.schedule(mode, splits, split_partials=partials, tile=tile)
                for ov in (1, 2):
                    b = sk.schedule(mode, splits, split_partials=partials, tile=tile, overlap=ov)
                    assert np.array_equal(sk.sk_plan(M, N, K, 148, a), sk.sk_plan(M, N, K, 148, b))
                    for red in (0, 1):
                        assert (sk.sk_workspace_size(M, N, K, 148, a, red) ==
                                sk.sk_workspace_size(M, N, K, 148, b, red))


def test_plan_streamk_groups(sk):
    # max_sk_groups_ grouping (first page, Case 4 knob table): the C planner's map equals
    # the oracle's for every group count on the workloads and a brute-force grid, with and
    # without the separate fixup pass.
    for M, N, K in [(128, 640, 256), (2048, 2432, 4096), (512, 512, 65536), (96, 512, 2048), (256, 512, 2048),
                    (1536, 1536, 4096), (3840, 3840, 4096), (8192, 8192, 8192)]:
        for tile in (0, 1, 2, 3):
            for g in (0, 1, 2, 3, 4, 8, 16, 64):
                for mode in (S.STREAMK, S.HYBRID):
                    _cmp(sk, M, N, K, 148, mode, tile=tile, groups=g)
                    _cmp(sk, M, N, K, 148, mode, tile=tile, groups=g, partials=1)
    for M, N, K in itertools.product((128, 300, 640), (128, 256, 640), (64, 200, 512)):
        for sms in (1, 2, 3, 5, 8, 13, 20):
            for g in (2, 3, 8):
                for mode in (S.STREAMK, S.HYBRID):
                    _cmp(sk, M, N, K, sms, mode, groups=g)
                    _cmp(sk, M, N, K, sms, mode, groups=g, tile=2)
    for bad in (-1, 65):
        with pytest.raises(sk.SkError):
            sk.sk_plan(128, 128, 64, 4, sk.schedule(2, sk_groups=bad))


def test_plan_toy_units_override(sk):
    a = _cmp(sk, 128, 640, 256, 148, S.STREAMK, units=4)
    b = _cmp(sk, 128, 640, 256, 4, S.STREAMK)
    assert np.array_equal(a, b)


def test_plan_bruteforce_small(sk):
    # M, N <= 640, K <= 512, 1..20 SMs, every mode.
    for M, N, K in itertools.product((1, 128, 129, 300, 640), (8, 128, 256, 640), (8, 64, 65, 200, 512)):
        for sms in range(1, 21):
            for tile in (0, 1, 2, 3):
                for mode in (S.DP, S.STREAMK, S.HYBRID):
                    _cmp(sk, M, N, K, sms, mode, tile=tile)
                for mode in (S.STREAMK, S.HYBRID):
                    _cmp(sk, M, N, K, sms, mode, partials=1, tile=tile)
                iters = S.cdiv(K, 64)
                for s in range(1, min(iters, 5) + 1):
                    _cmp(sk, M, N, K, sms, S.SPLITK, splits=s, tile=tile)
                    _cmp(sk, M, N, K, sms, S.SPLITK, splits=s, partials=1, tile=tile)


def test_plan_min_iters(sk):
    for mi in (1, 4, 8, 16, 64):
        for m in (1536, 1664, 3840):
            _cmp(sk, m, m, 4096, 132, S.HYBRID, min_iters=mi)


def test_workspace_size(sk):
    for (M, N, K, sms, mode, s, part), tile in itertools.product(
            [(2048, 2432, 4096, 148, S.HYBRID, 1, 0), (128, 640, 256, 4, S.STREAMK, 1, 0),
             (96, 512, 2048, 148, S.SPLITK, 8, 1), (96, 512, 2048, 148, S.SPLITK, 8, 2),
            (2048, 2432, 4096, 148, S.SPLITK, 2, 0), (2048, 2432, 4096, 148, S.HYBRID, 1, 1),
            (512, 512, 65536, 148, S.STREAMK, 1, 1),
             (2048, 2432, 4096, 148, S.DP, 1, 0)], (0, 1, 2, 3)):
        sch = sk.schedule(mode, s, 0, 0, part, tile)
        m = sk.sk_plan(M, N, K, sms, sch)
        n_slots, splits = int(m[11]), int(m[8])
        tm, tn, cg = int(m[12]), int(m[13]), int(m[14])
        if part and mode == S.SPLITK:
            want = 256 + -(-4 * splits * M * N // 256) * 256 + -(-4 * int(m[2]) * cg // 256) * 256
        else:
            want = 256 + -(-4 * n_slots * cg // 256) * 256 + n_slots * tm * tn * 4
        for r in (sk.SK_DETERMINISTIC, sk.SK_ATOMIC):
            assert sk.sk_workspace_size(M, N, K, sms, sch, r) == want


def test_errors(sk):
    bad = [
        (0, 128, 128, 4, sk.schedule(sk.SK_DP)),
        (128, 128, 128, 0, sk.schedule(sk.SK_DP)),
        (128, 128, 128, 4, sk.schedule(7)),
        (128, 128, 128, 4, sk.schedule(sk.SK_SPLITK, 3)),          # s > iters (2)
        (128, 128, 128, 4, sk.schedule(sk.SK_SPLITK, 0)),
        (128, 128, 128, 4, sk.schedule(sk.SK_STREAMK, 1, 0, 0, 2)),  # the last-arriver sum needs slabs
        (128, 128, 128, 4, sk.schedule(sk.SK_DP, 1, 0, 0, 1)),       # data-parallel tiles have no partials
        (128, 128, 128, 4, sk.schedule(sk.SK_SPLITK, 2, 0, 0, 3)),   # unknown slab reduction
        (128, 128, 128, 4, sk.schedule(sk.SK_DP, 1, -1)),
        (128, 128, 128, 1, sk.schedule(sk.SK_DP, 1, 0, 0, 0, 1)),      # a pair needs 2 SMs
        (128, 128, 128, 4, sk.schedule(sk.SK_DP, 1, 0, 0, 0, 4)),      # unknown tile shape
        (128, 128, 128, 4, sk.schedule(sk.SK_DP, overlap=3)),          # overlap is 0, 1 or 2
        (128, 128, 128, 4, sk.schedule(sk.SK_DP, overlap=-1)),
    ]
    for M, N, K, sms, sch in bad:
        with pytest.raises(sk.SkError) as e:
            sk.sk_plan_size(M, N, K, sms, sch)
        assert e.value.code == sk.SK_EINVAL
    L = sk.lib()
    buf = (ctypes.c_int32 * 4)()
    assert L.sk_plan(128, 640, 256, 4, sk.schedule(sk.SK_STREAMK), buf, 4) == sk.SK_ECAPACITY
    assert sk.sk_strerror(sk.SK_ETIMEOUT).startswith("a device-side wait")
    # sk_gemm argument checks happen before any CUDA call.
    sch = sk.schedule(sk.SK_DP)
    assert L.sk_gemm(16, 16, 16, sk.SK_F32, 128, 100, 64, sk.SK_NN, sch, 0, 148, 256, 1 << 20, None) == sk.SK_EINVAL
    assert L.sk_gemm(16, 16, 16, sk.SK_F32, 128, 128, 60, sk.SK_NN, sch, 0, 148, 256, 1 << 20, None) == sk.SK_EINVAL
    assert L.sk_gemm(16, 16, 17, sk.SK_F32, 128, 128, 64, sk.SK_NN, sch, 0, 148, 256, 1 << 20, None) == sk.SK_EINVAL
    assert L.sk_gemm(16, 16, 16, sk.SK_F32, 128, 128, 64, sk.SK_NN, sch, 0, 148, 0, 1 << 20, None) == sk.SK_EWORKSPACE
    assert L.sk_gemm(16, 16, 16, sk.SK_F32, 128, 128, 64, sk.SK_NN, sch, 0, 148, 256, 8, None) == sk.SK_EWORKSPACE
    assert L.sk_gemm(0, 0, 0, sk.SK_F32, 0, 128, 64, sk.SK_NN, sch, 0, 148, 0, 0, None) == sk.SK_OK
    assert L.sk_reduce_splits(16, 16, sk.SK_F32, 0, 64, None) == sk.SK_EINVAL
    assert L.sk_reduce_splits(16, 16, sk.SK_F32, 2, 6, None) == sk.SK_EINVAL


def test_host_staging_size(sk):
    # One set holds A [M, K] and B [K, N] in BF16 and C [M, N], each part rounded up to 256
    # bytes; depth 2 holds two sets.
    up = lambda x: -(-x // 256) * 256
    for M, N, K, dt, esz in [(128, 640, 256, sk.SK_F32, 4), (96, 512, 2048, sk.SK_BF16, 2),
                             (3, 8, 8, sk.SK_BF16, 2), (0, 8, 8, sk.SK_F32, 4), (5, 24, 0, sk.SK_F32, 4)]:
        one = up(M * K * 2) + up(K * N * 2) + up(M * N * esz)
        assert sk.sk_host_staging_size(M, N, K, dt, 1) == one
        assert sk.sk_host_staging_size(M, N, K, dt, 2) == 2 * one
    for bad in [(-1, 8, 8, 0, 1), (8, 8, 8, 2, 1), (8, 8, 8, 0, 0), (8, 8, 8, 0, 3)]:
        with pytest.raises(sk.SkError) as e:
            sk.sk_host_staging_size(*bad)
        assert e.value.code == sk.SK_EINVAL


def test_gemm_host_argument_errors(sk):
    # Rejected by the checks that run before any CUDA call, so no device is needed.
    M, N, K = 128, 256, 128
    a = np.zeros(M * K, np.uint16)
    b = np.zeros(K * N, np.uint16)
    c = np.zeros(M * N, np.float32)
    pa, pb, pc = a.ctypes.data, b.ctypes.data, c.ctypes.data
    sched = sk.schedule(sk.SK_HYBRID)
    need = sk.sk_host_staging_size(M, N, K, sk.SK_F32, 2)

    def call(A=(pa,), B=(pb,), C=(pc,), depth=1, staging=256, nbytes=need, copy_in=None, copy_out=None, m=M):
        return sk.sk_gemm_host(list(A), list(B), list(C), sk.SK_F32, m, N, K, sk.SK_NN, sched, sk.SK_DETERMINISTIC,
                               148, staging, nbytes, depth, 256, 1 << 20, None, copy_in, copy_out)

    assert call(A=(), B=(), C=()) == sk.SK_OK  # no problems: nothing to do
    assert call(m=0) == sk.SK_OK
    for kw, code in [(dict(depth=0), sk.SK_EINVAL), (dict(depth=3), sk.SK_EINVAL), (dict(m=-1), sk.SK_EINVAL),
                     (dict(C=(0,)), sk.SK_EINVAL), (dict(A=(0,)), sk.SK_EINVAL), (dict(B=(0,)), sk.SK_EINVAL),
                     (dict(depth=2), sk.SK_EINVAL),  # depth 2 needs two copy streams
                     (dict(depth=2, copy_in=7, copy_out=0), sk.SK_EINVAL),
                     (dict(depth=2, copy_in=7, copy_out=7), sk.SK_EINVAL),
                     (dict(staging=0), sk.SK_EWORKSPACE), (dict(staging=128), sk.SK_EWORKSPACE),
                     (dict(depth=2, copy_in=7, copy_out=9, nbytes=need - 1), sk.SK_EWORKSPACE)]:
        with pytest.raises(sk.SkError) as e:
            call(**kw)
        assert e.value.code == code, kw
    with pytest.raises(ValueError):
        sk.sk_gemm_host([pa], [pb], [pc, pc], sk.SK_F32, M, N, K, sk.SK_NN, sched, sk.SK_DETERMINISTIC, 148, 256,
                        need, 1, 256, 1 << 20)


def test_header_is_plain_c():
    # The boundary is a C ABI: include/sk.h must compile as C99 (and as C++) on its own.
    import shutil
    import subprocess
    hdr = os.path.join(ROOT, "include", "sk.h")
    for cc, lang, std in (("gcc", "c", "-std=c99"), ("g++", "c++", "-std=c++17")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not found")
        p = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", lang, hdr],
                           capture_output=True, text=True)
        assert p.returncode == 0, p.stderr


C_CONSUMER = r"""
#include <stdio.h>
#include <stdlib.h>
#include "sk.h"
int main(void) {
    sk_schedule s = {0};
    s.mode = SK_STREAMK;
    s.units = 4;
    int64_t n = sk_plan_size(128, 640, 256, 4, s);
    if (n < 0) return 2;
    int32_t* map = (int32_t*)malloc((size_t)n * sizeof(int32_t));
    if (!map || sk_plan(128, 640, 256, 4, s, map, n) != SK_OK) return 3;
    for (int64_t i = 0; i < n; ++i) printf("%d\n", map[i]);
    free(map);
    return sk_plan(128, 640, 256, 4, s, NULL, 0) == SK_ECAPACITY ? 0 : 4;
}
"""


def test_plain_c_consumer(sk, tmp_path):
    # A C program, compiled and linked against libsk.so with no Python or torch in between,
    # plans the toy Stream-K case (4 units, 5 tiles x 4 k-iterations) and gets the oracle's map.
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    src, exe = tmp_path / "consumer.c", tmp_path / "consumer"
    src.write_text(C_CONSUMER)
    libdir = os.path.dirname(sk.LIB_PATH)
    p = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", libdir, "-lsk", f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert p.returncode == 0, p.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    got = np.array([int(x) for x in r.stdout.split()], dtype=np.int32)
    want = S.plan_map(S.build_plan(128, 640, 256, 4, S.STREAMK, units=4))
    assert np.array_equal(got, np.asarray(want, dtype=np.int32))
