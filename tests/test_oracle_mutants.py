"""The oracle's pins must reject a broken oracle (CPU only).

Each case compiles a copy of oracle/gemm_oracle.c with one plausible mistake
planted in it -- a dropped term, a flipped sign, a transposed or mis-strided
index, a wrong exponent bias, a reversed summation order -- loads it in place
of the real oracle, and checks that at least one of the pins of
tests/test_oracle.py fails on it.  The real oracle passes all of them.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads

SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")

MUTANTS = {
    "drops_last_k_term": ("for (int64_t k = 0; k < K; ++k) {\n            double a = t[A[i * lda + k]];",
                          "for (int64_t k = 0; k + 1 < K; ++k) {\n            double a = t[A[i * lda + k]];"),
    "subtracts_products": ("for (int64_t j = 0; j < N; ++j) c[j] += a * t[b[j]];",
                           "for (int64_t j = 0; j < N; ++j) c[j] -= a * t[b[j]];"),
    "row_stride_is_K": ("double a = t[A[i * lda + k]];", "double a = t[A[i * K + k]];"),
    "b_row_stride_is_N": ("const uint16_t *b = B + k * ldb;", "const uint16_t *b = B + k * N;"),
    "f16_bias_off_by_one": ("v = ldexp((double)(1024 + f), e - 25);",
                            "v = ldexp((double)(1024 + f), e - 24);"),
    "bf16_hidden_bit_missing": ("v = ldexp((double)(128 + f), e - 134);",
                                "v = ldexp((double)(f), e - 134);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "k_descending": ("for (int64_t k = 0; k < K; ++k) {\n            double a = t[A[i * lda + k]];",
                     "for (int64_t k = K - 1; k >= 0; --k) {\n            double a = t[A[i * lda + k]];"),
}


def f16(rows):
    return torch.tensor(rows, dtype=torch.float32).to(torch.float16)


def bf16(rows):
    return torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)


def pins_pass() -> bool:
    """A compact run of the oracle's pins; True only if every one holds."""
    from conftest import read_golden
    checks = []
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    got16 = np.array([oracle.decode(int(b), oracle.F16) for b in bits])
    fin = np.isfinite(ref16)
    checks.append(np.array_equal(got16[fin], ref16[fin]))
    refb = torch.from_numpy(bits.astype(np.int32)).to(torch.int16).view(torch.bfloat16)
    refb = refb.to(torch.float64).numpy()
    gotb = np.array([oracle.decode(int(b), oracle.BF16) for b in bits])
    finb = np.isfinite(refb)
    checks.append(np.array_equal(gotb[finb], refb[finb]))
    g = read_golden("matmul_4x4.txt")
    checks.append(np.array_equal(oracle.gemm(f16(g["A"]), f16(g["B"])), np.array(g["C"], float)))
    gen = torch.Generator().manual_seed(5)
    Ai = torch.randint(-4, 5, (17, 33), generator=gen)
    Bi = torch.randint(-4, 5, (33, 9), generator=gen)
    exact = (Ai.numpy().astype(np.int64) @ Bi.numpy().astype(np.int64)).astype(float)
    checks.append(np.array_equal(oracle.gemm(Ai.to(torch.bfloat16), Bi.to(torch.bfloat16)), exact))
    A, B = workloads.custom(45, 37, 29, "f16", seed=9)
    Ap, Bp = workloads.custom(45, 37, 29, "f16", seed=9, lda=48, ldb=40)
    checks.append(np.array_equal(oracle.gemm(A, B), oracle.gemm(Ap, Bp, K=37, N=29)))
    order = oracle.gemm(bf16([[1.0, 2.0 ** 60, -(2.0 ** 60)]]), bf16([[1.0], [1.0], [1.0]]))
    checks.append(order[0, 0] == 0.0)
    return all(bool(c) for c in checks)


def test_real_oracle_passes_the_pins():
    assert pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_oracle_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(c_path), "-o", str(so_path), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(str(so_path))))
    assert not pins_pass(), f"the pins did not catch the '{name}' mutant"
