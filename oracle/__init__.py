"""CPU oracle for C[M,N] = A[M,K] @ B[K,N] -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
nothing here imports the product package: the two share no code.

Contents
  * ``gemm`` / ``absbound`` / ``gemm_entries`` / ``gemm_blockwise``: ctypes
    wrappers of the plain-C binary64 loops in ``gemm_oracle.c`` (naive loop of
    Step 1 and blockwise loop of Step 2 of "I Wrote a GPU Matmul Kernel From
    Scratch in Triton"; the element definition of section 3.1 of "Writing GPU
    kernels in Triton: Vector Add, Softmax, MatMul").
  * ``schedule``: the tile-grid, mask and program-order arithmetic that the
    pages print (pure Python).
  * ``softmax``: row-wise softmax in binary64 (numpy), the five steps of
    section 2.3 of "Writing GPU kernels in Triton: Vector Add, Softmax, MatMul";
    pinned by ``tests/test_softmax_oracle.py``.
  * ``attention``: attention forward O = softmax(Q K^T / sqrt(d) [+ causal
    mask]) V in binary64 (numpy), the result the Flash Attention section of
    "How to hand-write Triton kernels for matmul and Flash Attention" reaches;
    pinned by ``tests/test_attention_oracle.py``.

Pinned by ``tests/test_oracle.py`` against the pages' worked examples, closed
forms (identity, zero, small-integer products), bit-pattern decoding by numpy
and torch, and brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F16 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into oracle/_build/liboracle.so with the host gcc.

    -ffp-contract=off keeps every multiply and add separately rounded on both
    x86_64 and aarch64 hosts.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded oracle library (also used by the
    mutation tests, which load deliberately broken builds of the same source)."""
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.oracle_gemm.argtypes = [i32, u16p, i64, u16p, i64, f64p, i64, i64, i64, i64, i32]
    lib.oracle_gemm.restype = i32
    lib.oracle_absbound.argtypes = [i32, u16p, i64, u16p, i64, f64p, i64, i64, i64, i64, i32]
    lib.oracle_absbound.restype = i32
    lib.oracle_gemm_entries.argtypes = [i32, u16p, i64, u16p, i64, i64, i64, i64,
                                        i64p, i64p, i64, f64p, f64p, i32]
    lib.oracle_gemm_entries.restype = i32
    lib.oracle_gemm_blockwise.argtypes = [i32, u16p, i64, u16p, i64, f64p, i64, i64, i64,
                                          i64, i64]
    lib.oracle_gemm_blockwise.restype = i32
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            build()
        _lib = bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _bits(x) -> tuple[np.ndarray, int]:
    """Return (uint16 bit patterns as a 2-D C-contiguous array, dtype code).

    Accepts a torch tensor of dtype float16/bfloat16 (CPU) or a numpy float16
    array.  The bits are passed as they are: the oracle decodes them itself.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.float16:
                code = F16
            elif x.dtype == torch.bfloat16:
                code = BF16
            else:
                raise TypeError(f"oracle inputs must be fp16 or bf16, got {x.dtype}")
            b = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
            return np.ascontiguousarray(b), code
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    a = np.asarray(x)
    if a.dtype == np.float16:
        return np.ascontiguousarray(a.view(np.uint16)), F16
    raise TypeError(f"unsupported oracle input type {type(x)} / {getattr(a, 'dtype', None)}")


def _u16p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _f64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _shape(A, B, K):
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("A and B must be 2-D")
    M, lda = A.shape
    Kb, ldb = B.shape
    if K is None:
        K = lda
    if Kb < K or lda < K:
        raise ValueError(f"K={K} exceeds the stored operands ({A.shape}, {B.shape})")
    return M, lda, ldb, K


def gemm(A, B, *, K: int | None = None, N: int | None = None, nthreads: int = 0) -> np.ndarray:
    """Exact-input binary64 product of the stored operands.

    A is stored as (M, lda) and B as (>=K, ldb); the product uses the first K
    columns of A, the first K rows of B and the first N (default ldb) columns
    of B -- row-major with leading dimensions lda and ldb, as in section 4.1 of
    "Writing GPU kernels in Triton".  Returns C as an (M, N) float64 array.
    """
    a, code = _bits(A)
    b, code_b = _bits(B)
    if code != code_b:
        raise TypeError("A and B must have the same dtype")
    M, lda, ldb, K = _shape(a, b, K)
    if N is None:
        N = ldb
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm(code, _u16p(a), lda, _u16p(b), ldb, _f64p(C), N, M, N, K, nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return C


def absbound(A, B, *, K: int | None = None, N: int | None = None, nthreads: int = 0) -> np.ndarray:
    """bound[i, j] = sum_k |A[i, k]| |B[k, j]| in binary64 (the tolerance scale)."""
    a, code = _bits(A)
    b, _ = _bits(B)
    M, lda, ldb, K = _shape(a, b, K)
    if N is None:
        N = ldb
    out = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_absbound(code, _u16p(a), lda, _u16p(b), ldb, _f64p(out), N, M, N, K,
                                 nthreads)
    if rc != 0:
        raise ValueError("oracle_absbound rejected its arguments")
    return out


def gemm_entries(A, B, rows, cols, *, K: int | None = None, N: int | None = None,
                 nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """(value, bound) of the product at the listed (row, col) entries only."""
    a, code = _bits(A)
    b, _ = _bits(B)
    M, lda, ldb, K = _shape(a, b, K)
    if N is None:
        N = ldb
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    val = np.empty(r.shape[0], dtype=np.float64)
    bnd = np.empty(r.shape[0], dtype=np.float64)
    rc = _load().oracle_gemm_entries(code, _u16p(a), lda, _u16p(b), ldb, M, N, K, _i64p(r),
                                     _i64p(c), r.shape[0], _f64p(val), _f64p(bnd), nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return val, bnd


def gemm_blockwise(A, B, block: int, *, K: int | None = None, N: int | None = None) -> np.ndarray:
    """The six-loop blockwise product of Step 2 (tiles of size ``block``)."""
    a, code = _bits(A)
    b, _ = _bits(B)
    M, lda, ldb, K = _shape(a, b, K)
    if N is None:
        N = ldb
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_blockwise(code, _u16p(a), lda, _u16p(b), ldb, _f64p(C), N, M, N, K,
                                       block)
    if rc != 0:
        raise ValueError("oracle_gemm_blockwise rejected its arguments")
    return C


def decode(bits: int, code: int) -> float:
    """Exact value of one 16-bit pattern (F16 or BF16) as the oracle decodes it."""
    lib = _load()
    return lib.oracle_f16_to_f64(bits) if code == F16 else lib.oracle_bf16_to_f64(bits)


def max_threads() -> int:
    """Threads the oracle's parallel loops use by default (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_max_threads())


def within_tolerance(c_gpu, c_ref, bound, rel: float = 1e-3, abs_: float = 1e-5) -> np.ndarray:
    """Element-wise pass mask |c_gpu - c_ref| <= rel * bound + abs_."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    return np.abs(c_gpu - np.asarray(c_ref)) <= rel * np.asarray(bound) + abs_
