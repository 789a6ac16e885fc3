"""The GPU parity suites run again on the checked build (GPU).

The checked build (``libgemm_checked.so``) tests every ordinary global load and
store of the kernels against the matrix or buffer it belongs to and skips any
that falls outside, recording it in the plan's status word; with debug-sync on,
gemm_run (and softmax_rows, attention_fwd) then return GEMM_ERR_BOUNDS, which
the binding raises.  The GEMM parity suites -- every kernel, layout, staged and
in-place operand, ragged edge, output type, partition slice and sampled
full-size case -- the softmax and attention suites, the waits made to run out
(the abort and drain paths) and two plans used at once are run in a child
process with DG_GEMM_CHECKED=1 and GEMM_DEBUG_SYNC=1: they must pass there
unchanged, i.e. no access of any of their launches leaves its range and the
results still match the oracle.
"""
import os
import subprocess
import sys

import pytest
import torch

import dense_gemm_05_gb300 as g

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gemm_gpu.py", "tests/test_layouts_gpu.py", "tests/test_partition_gpu.py",
          "tests/test_large_gpu.py", "tests/test_fuzz_gpu.py", "tests/test_softmax_gpu.py",
          "tests/test_attention_gpu.py", "tests/test_timeouts_gpu.py",
          "tests/test_concurrency_gpu.py"]


def test_the_checked_library_is_the_one_loaded():
    """Inside the child run: the binding loaded the checked build."""
    if not g.checked_requested():
        pytest.skip("runs inside the checked child process")
    assert g.gemm_build_checked() == 1
    p = g.Plan(0)
    try:
        assert p.device_status() == 0
    finally:
        p.close()


def test_parity_suites_pass_on_the_checked_build():
    if g.checked_requested():
        pytest.skip("this is the checked child process")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.build(checked=True)
    env = dict(os.environ, DG_GEMM_CHECKED="1", GEMM_DEBUG_SYNC="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-rs", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_checked_gpu.py", *SUITES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout[-4000:] + "\n" + r.stderr[-2000:]).strip()
    assert r.returncode == 0, tail
    # the child loaded the checked build (its first test ran rather than skipped)
    assert " passed" in r.stdout and "runs inside the checked child" not in r.stdout, tail
