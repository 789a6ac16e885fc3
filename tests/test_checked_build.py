"""The checked build on the host (no GPU): it builds, loads, exports the whole
ABI and says it is checked; and the two range predicates its kernels test every
ordinary global access with agree with their definition on every small case.

The checked build (``libgemm_checked.so``, the sources compiled with
DG_CHECKED=1) stands in for a memory checker: each load and store first tests
the range it touches -- ``span_inside(r, c, n, rows, cols)``: elements
[c, c + n) of row r inside a rows x cols rectangle; ``bytes_inside(a, n, lo,
hi)``: bytes [a, a + n) inside [lo, hi) -- and is skipped when the test fails.
The predicates are compiled for the host from the kernels' own header and run
over every case of a small grid, including negative and overflowing operands,
against a direct enumeration of the elements or bytes.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import dense_gemm_05_gb300 as g
from test_abi import declared_functions

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_05_gb300", "csrc")


@pytest.fixture(scope="module")
def checked_lib():
    g.build(checked=True)
    return ctypes.CDLL(g.CHECKED_LIB_PATH)


def test_checked_library_exports_the_abi_and_says_so(checked_lib):
    for name in declared_functions():
        assert hasattr(checked_lib, name), name
    checked_lib.gemm_build_checked.restype = ctypes.c_int32
    assert checked_lib.gemm_build_checked() == 1
    g.build(checked=False)
    normal = ctypes.CDLL(g.LIB_PATH)
    normal.gemm_build_checked.restype = ctypes.c_int32
    assert normal.gemm_build_checked() == 0


def test_device_status_needs_a_plan(checked_lib):
    assert g.lib().gemm_plan_device_status(None, None) == g.GEMM_ERR_INVALID_ARG


HARNESS = r"""
#include <cstdio>
#include <cstdint>
#include "common.cuh"
int main() {
    using dg::span_inside;
    using dg::bytes_inside;
    for (long r = -2; r < 5; ++r)
        for (long c = -3; c < 8; ++c)
            for (long n = 0; n < 6; ++n)
                for (long rows = 0; rows < 4; ++rows)
                    for (long cols = 0; cols < 7; ++cols)
                        std::printf("S %ld %ld %ld %ld %ld %d\n", r, c, n, rows, cols,
                                    int(span_inside(r, c, n, rows, cols)));
    // near the top of int64: c + n would overflow
    const int64_t big = INT64_MAX;
    std::printf("X %d %d %d\n", int(span_inside(0, big - 1, 5, 1, big)),
                int(span_inside(0, big - 5, 5, 1, big)), int(span_inside(0, big - 4, 5, 1, big)));
    for (unsigned a = 0; a < 20; ++a)
        for (unsigned n = 0; n < 8; ++n)
            for (unsigned lo = 0; lo < 10; ++lo)
                for (unsigned hi = lo; hi < 16; ++hi)
                    std::printf("B %u %u %u %u %d\n", a, n, lo, hi,
                                int(bytes_inside(a, n, lo, hi)));
    // near the top of the address space: a + n would wrap
    const uintptr_t top = UINTPTR_MAX;
    std::printf("W %d %d %d\n", int(bytes_inside(top - 3, 16, 0, top)),
                int(bytes_inside(top - 16, 16, 0, top)), int(bytes_inside(top - 15, 16, 0, top)));
    return 0;
}
"""


def test_range_predicates_match_their_definition(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "predicates.cu"
    src.write_text(HARNESS)
    exe = tmp_path / "predicates"
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    spans = bytes_ = 0
    for line in out:
        f = line.split()
        if not f:
            continue
        if f[0] == "S":
            r, c, n, rows, cols, got = map(int, f[1:])
            want = n >= 1 and all(0 <= r < rows and 0 <= c + i < cols for i in range(n))
            assert bool(got) == want, line
            spans += 1
        elif f[0] == "B":
            a, n, lo, hi, got = map(int, f[1:])
            # n = 0 touches nothing: inside when a lies in [lo, hi]
            want = (lo <= a <= hi) if n == 0 else all(lo <= a + i < hi for i in range(n))
            assert bool(got) == want, line
            bytes_ += 1
        elif f[0] == "X":
            assert list(map(int, f[1:])) == [0, 1, 0], line
        elif f[0] == "W":
            assert list(map(int, f[1:])) == [0, 1, 0], line
    assert spans == 7 * 11 * 6 * 4 * 7 and bytes_ > 5000
