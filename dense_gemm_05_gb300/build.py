"""Build the CUDA library ``_build/libgemm.so`` in-tree with nvcc (sm_103a only).

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked into
one shared library with the CUDA runtime linked statically, so the library
loads (and exports its C ABI) on a host without a GPU driver; the driver is
only needed when a plan is created.

The checked build, ``_build/libgemm_checked.so``, is the same sources compiled
with ``DG_CHECKED=1``: every ordinary global load and store of the kernels is
first tested against the matrix or buffer it belongs to (see ``include/gemm.h``,
"Checked builds").  ``build(checked=True)`` makes it; ``build_all()`` makes both
libraries in one parallel compile.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libgemm.so")
CHECKED_LIB_PATH = os.path.join(BUILD_DIR, "libgemm_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgemm.so")
    return cand


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _variant(checked: bool) -> tuple[str, str, list[str]]:
    """(library path, object directory, extra nvcc flags) of one build variant."""
    if checked:
        return CHECKED_LIB_PATH, os.path.join(BUILD_DIR, "checked"), ["-DDG_CHECKED=1"]
    return LIB_PATH, BUILD_DIR, []


def up_to_date(checked: bool = False) -> bool:
    lib = _variant(checked)[0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _build_variants(variants: list[bool], verbose: bool, ptxas_info: bool) -> None:
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for checked in variants:
        _, obj_dir, flags = _variant(checked)
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(src, obj_dir, flags) for src in _sources()]

    def compile_one(job: tuple[str, str, list[str]]) -> tuple[str, str]:
        src, obj_dir, flags = job
        obj = os.path.join(obj_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *flags, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src} {' '.join(flags)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log)
    for checked in variants:
        lib, obj_dir, _ = _variant(checked)
        objs = [o for o, _ in results if os.path.dirname(o) == obj_dir]
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
               "-lpthread", "-ldl", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool = False) -> str:
    """Compile and link libgemm.so (or, checked=True, libgemm_checked.so); returns
    its path.  Raises on any compiler error."""
    if force or not up_to_date(checked):
        _build_variants([checked], verbose, ptxas_info)
    return _variant(checked)[0]


def build_all(force: bool = False) -> list[str]:
    """Both libraries, their translation units compiled in one parallel pool."""
    todo = [c for c in (False, True) if force or not up_to_date(c)]
    if todo:
        _build_variants(todo, False, False)
    return [LIB_PATH, CHECKED_LIB_PATH]


if __name__ == "__main__":
    import sys
    if "--all" in sys.argv:
        print(build_all(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                    checked="--checked" in sys.argv))
