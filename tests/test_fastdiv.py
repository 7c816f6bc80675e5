"""The schedule walk's invariant-divisor division (sk_schedule.h FastDiv) against plain integer
division, compiled for the host with g++ from the same header the kernels include."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = r'''
#include <cstdio>
#include <cstdint>
#include "sk_schedule.h"
int main() {
    uint64_t bad = 0, n_checked = 0;
    const int32_t ns[] = {0, 1, 2, 3, 7, 63, 64, 65, 127, 128, 1000, 4095, 4096, 65535, 65536, 1 << 20,
                          (1 << 30) - 1, 1 << 30, 2147483646, 2147483647};
    for (uint32_t d = 1; d <= 20000; ++d) {
        const sk::FastDiv f = sk::make_fastdiv(d);
        for (int32_t n : ns) { bad += sk::fdiv(f, n) != n / static_cast<int32_t>(d); ++n_checked; }
        for (int32_t k = 0; k < 64; ++k) {  // around multiples of d
            const int64_t base = static_cast<int64_t>(d) * (k * 977 + 1);
            for (int64_t n = base - 2; n <= base + 2; ++n)
                if (n >= 0 && n <= 2147483647) { bad += sk::fdiv(f, (int32_t)n) != (int32_t)(n / d); ++n_checked; }
        }
    }
    const uint32_t big[] = {65537u, 1000003u, 2147483647u, 1u << 31};
    for (uint32_t d : big) {
        const sk::FastDiv f = sk::make_fastdiv(d);
        for (int32_t n : ns) { bad += (uint32_t)sk::fdiv(f, n) != (uint32_t)n / d; ++n_checked; }
    }
    std::printf("%llu %llu\n", (unsigned long long)bad, (unsigned long long)n_checked);
    return bad != 0;
}
'''


def test_fastdiv_matches_integer_division(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    src = tmp_path / "fd.cpp"
    src.write_text(SRC)
    exe = tmp_path / "fd"
    inc = os.path.join(ROOT, "gemm_work_decomposition_gb300", "csrc")
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", inc, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    bad, checked = map(int, out.stdout.split())
    assert out.returncode == 0 and bad == 0 and checked > 1_000_000
