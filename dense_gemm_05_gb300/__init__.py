"""Python binding of the GB300 GEMM C ABI (``include/gemm.h``).

Argument marshalling only: every step of ``C = A @ B`` runs in the CUDA
kernels of ``_build/libgemm.so``.  PyTorch supplies device memory and streams.
There is no fallback: if the library has not been built, importing the
binding functions raises.  With ``DG_GEMM_CHECKED=1`` in the environment the
binding loads (and ``build()`` makes) the checked build
``_build/libgemm_checked.so`` instead: the same ABI, with every ordinary
global access of the kernels tested against its matrix (``include/gemm.h``).

    plan = gemm_plan_create(0)
    gemm_run(plan, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc, M, N, K,
             GEMM_BF16, torch.cuda.current_stream().cuda_stream)
    gemm_plan_destroy(plan)

``matmul(a, b)`` wraps the same calls for 2-D torch tensors; ``softmax(x)``
wraps the row-wise softmax of ``include/softmax.h``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import CHECKED_LIB_PATH, LIB_PATH, build_all  # noqa: F401  (for __graft_entry__)
from .build import build as _build_one


def checked_requested() -> bool:
    """Whether DG_GEMM_CHECKED=1 asks for the checked build."""
    v = os.environ.get("DG_GEMM_CHECKED", "")
    return v not in ("", "0")


def lib_path() -> str:
    return CHECKED_LIB_PATH if checked_requested() else LIB_PATH


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool | None = None) -> str:
    """Build the library the binding loads (the checked one under DG_GEMM_CHECKED=1)."""
    return _build_one(force, verbose, ptxas_info,
                      checked_requested() if checked is None else checked)

GEMM_F16 = 0
GEMM_BF16 = 1

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_CUDA = 3
GEMM_ERR_OOM = 4
GEMM_ERR_TIMEOUT = 5
GEMM_ERR_BOUNDS = 6

GEMM_OP_N = 0
GEMM_OP_T = 1

GEMM_OUT_F32 = 0
GEMM_OUT_F16 = 1
GEMM_OUT_BF16 = 2

GEMM_KERNEL_NONE = 0
GEMM_KERNEL_ZERO_FILL = 1
GEMM_KERNEL_TMA = 2
GEMM_KERNEL_GENERIC = 3
GEMM_KERNEL_SKINNY = 4
GEMM_KERNEL_PAIR = 5
GEMM_KERNEL_SPLIT_PAIR = 6

KERNEL_NAMES = {0: "none", 1: "zero_fill", 2: "tma", 3: "generic", 4: "skinny", 5: "pair",
                6: "split_pair"}

#: Every function the header declares (checked by the tests against the library's exports).
ABI_FUNCTIONS = ("gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_status_string",
                 "gemm_query", "gemm_plan_set_group", "gemm_plan_force", "gemm_tile_coord",
                 "gemm_wait_selftest", "gemm_run_noalloc", "gemm_run_ex", "gemm_query_ex",
                 "softmax_rows", "softmax_rows_query", "attention_fwd", "attention_fwd_query",
                 "gemm_plan_create_model", "gemm_noop_launch", "gemm_plan_set_staging",
                 "gemm_plan_set_debug", "gemm_partition", "gemm_run_slice",
                 "gemm_build_checked", "gemm_plan_device_status", "attention_set_debug")

GEMM_SPLIT_AUTO = -1
GEMM_SPLIT_M = 0
GEMM_SPLIT_N = 1

SOFTMAX_PATH_NONE = 0
SOFTMAX_PATH_WARP = 1
SOFTMAX_PATH_CTA = 2
SOFTMAX_PATH_STREAM = 3
SOFTMAX_PATH_NAMES = {0: "none", 1: "warp", 2: "cta", 3: "stream"}

#: Limits of gemm_run_noalloc (mirrors of the header's macros).
GEMM_NOALLOC_MAX_M = 64
GEMM_NOALLOC_MAX_N = 131072
GEMM_NOALLOC_SCRATCH_BYTES = 8392960


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


class GemmConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kernel", "block_m", "block_n", "block_k", "stages", "split_k", "grid",
                 "cluster", "group", "tiles", "shares", "staged")]

    def as_dict(self) -> dict:
        d = {n: int(getattr(self, n)) for n, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(d["kernel"], "?")
        return d


class GemmSlice(ctypes.Structure):
    _fields_ = [("axis", ctypes.c_int32), ("rank", ctypes.c_int32), ("world", ctypes.c_int32),
                ("row0", ctypes.c_int64), ("rows", ctypes.c_int64),
                ("col0", ctypes.c_int64), ("cols", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class SoftmaxConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("path", "threads_per_row", "elems_per_thread", "vec", "rows_per_cta", "block",
                 "grid", "staged", "slots")]

    def as_dict(self) -> dict:
        d = {n: int(getattr(self, n)) for n, _ in self._fields_}
        d["path_name"] = SOFTMAX_PATH_NAMES.get(d["path"], "?")
        return d


class AttentionConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("block_q", "block_kv", "head_dim", "stages", "grid_x", "grid_y", "causal")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libgemm.so (built by ``build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: run dense_gemm_05_gb300.build() (or "
                "__graft_entry__.build()) first; there is no fallback implementation")
        L = ctypes.CDLL(path)
        vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
        L.gemm_plan_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int]
        L.gemm_plan_create.restype = i32
        L.gemm_plan_create_model.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32]
        L.gemm_plan_create_model.restype = i32
        L.gemm_run.argtypes = [vp, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32, vp]
        L.gemm_run.restype = i32
        L.gemm_plan_destroy.argtypes = [vp]
        L.gemm_plan_destroy.restype = i32
        L.gemm_status_string.argtypes = [i32]
        L.gemm_status_string.restype = ctypes.c_char_p
        L.gemm_query.argtypes = [vp, vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                 ctypes.POINTER(GemmConfig)]
        L.gemm_query.restype = i32
        L.gemm_plan_set_group.argtypes = [vp, i32]
        L.gemm_plan_set_group.restype = i32
        L.gemm_plan_force.argtypes = [vp, i32, i32, i32]
        L.gemm_plan_force.restype = i32
        L.gemm_plan_set_staging.argtypes = [vp, i32]
        L.gemm_plan_set_staging.restype = i32
        L.gemm_plan_set_debug.argtypes = [vp, i32, ctypes.c_uint64]
        L.gemm_plan_set_debug.restype = i32
        L.attention_set_debug.argtypes = [i32, ctypes.c_uint64]
        L.attention_set_debug.restype = i32
        L.gemm_build_checked.argtypes = []
        L.gemm_build_checked.restype = i32
        L.gemm_plan_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        L.gemm_plan_device_status.restype = i32
        L.gemm_partition.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(GemmSlice)]
        L.gemm_partition.restype = i32
        L.gemm_run_slice.argtypes = [vp, ctypes.POINTER(GemmSlice), vp, i64, vp, i64, vp, i64,
                                     i64, i64, i64, i32, vp]
        L.gemm_run_slice.restype = i32
        L.gemm_tile_coord.argtypes = [i64, i64, i64, i32, ctypes.POINTER(i64),
                                      ctypes.POINTER(i64)]
        L.gemm_tile_coord.restype = i32
        L.gemm_wait_selftest.argtypes = [u32, vp]
        L.gemm_wait_selftest.restype = i32
        L.gemm_noop_launch.argtypes = [i32, i32, vp]
        L.gemm_noop_launch.restype = i32
        L.gemm_run_noalloc.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, i32, vp]
        L.gemm_run_noalloc.restype = i32
        L.gemm_run_ex.argtypes = [vp, i32, i32, vp, i64, vp, i64, vp, i64, i32, i64, i64, i64,
                                  i32, vp]
        L.gemm_run_ex.restype = i32
        L.gemm_query_ex.argtypes = [vp, i32, i32, vp, i64, vp, i64, vp, i64, i32, i64, i64, i64,
                                    i32, ctypes.POINTER(GemmConfig)]
        L.gemm_query_ex.restype = i32
        L.softmax_rows.argtypes = [vp, i64, vp, i64, i64, i64, vp]
        L.softmax_rows.restype = i32
        L.softmax_rows_query.argtypes = [vp, i64, vp, i64, i64, i64, ctypes.POINTER(SoftmaxConfig)]
        L.softmax_rows_query.restype = i32
        L.attention_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i32, i32,
                                    i32, vp]
        L.attention_fwd.restype = i32
        L.attention_fwd_query.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i32,
                                          i32, i32, ctypes.POINTER(AttentionConfig)]
        L.attention_fwd_query.restype = i32
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().gemm_status_string(int(status)).decode()


# ------------------------------------------------------------------ C-ABI mirrors

def gemm_plan_create(device: int = 0) -> int:
    """Create a plan on `device`; returns the opaque handle (an int)."""
    h = ctypes.c_void_p()
    st = lib().gemm_plan_create(ctypes.byref(h), int(device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_create")
    return h.value


def gemm_plan_create_model(num_sms: int = 152, pair_clusters_128: int = 76,
                           pair_clusters_256: int = 76, splitpair_clusters: int = 76) -> int:
    """A plan for a modelled device (no GPU needed), for gemm_query/gemm_query_ex only;
    the defaults are what a GB300 reports."""
    h = ctypes.c_void_p()
    st = lib().gemm_plan_create_model(ctypes.byref(h), int(num_sms), int(pair_clusters_128),
                                      int(pair_clusters_256), int(splitpair_clusters))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_create_model")
    return h.value


def gemm_run(plan: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int, M: int, N: int,
             K: int, dtype: int, stream: int = 0) -> int:
    """C = A @ B on `stream` (raw pointers as ints); returns the gemm_status_t code."""
    return int(lib().gemm_run(plan, A, lda, B, ldb, C, ldc, M, N, K, dtype, stream))


def gemm_run_ex(plan: int, op_a: int, op_b: int, A: int, lda: int, B: int, ldb: int, C: int,
                ldc: int, c_type: int, M: int, N: int, K: int, dtype: int, stream: int = 0) -> int:
    """C = A @ B with A/B stored as op_a/op_b describe and C of type c_type."""
    return int(lib().gemm_run_ex(plan, op_a, op_b, A, lda, B, ldb, C, ldc, c_type, M, N, K,
                                 dtype, stream))


def gemm_query_ex(plan: int, op_a: int, op_b: int, A: int, lda: int, B: int, ldb: int, C: int,
                  ldc: int, c_type: int, M: int, N: int, K: int, dtype: int) -> dict:
    cfg = GemmConfig()
    st = lib().gemm_query_ex(plan, op_a, op_b, A, lda, B, ldb, C, ldc, c_type, M, N, K, dtype,
                             ctypes.byref(cfg))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_query_ex")
    return cfg.as_dict()


def gemm_plan_destroy(plan: int | None) -> int:
    return int(lib().gemm_plan_destroy(plan))


def gemm_query(plan: int, A: int, lda: int, B: int, ldb: int, C: int, ldc: int, M: int, N: int,
               K: int, dtype: int) -> dict:
    cfg = GemmConfig()
    st = lib().gemm_query(plan, A, lda, B, ldb, C, ldc, M, N, K, dtype, ctypes.byref(cfg))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_query")
    return cfg.as_dict()


def gemm_plan_set_group(plan: int, group: int) -> int:
    return int(lib().gemm_plan_set_group(plan, group))


def gemm_plan_force(plan: int, kernel: int = 0, split_k: int = 0, block_n: int = 0) -> int:
    return int(lib().gemm_plan_force(plan, kernel, split_k, block_n))


def gemm_plan_set_debug(plan: int, sync: int, timeout_ns: int = 0) -> int:
    """Debug-sync mode (gemm_run waits and reports device-side give-ups) and the
    limit of every bounded device wait (0 = the default)."""
    return int(lib().gemm_plan_set_debug(plan, int(sync), int(timeout_ns)))


def attention_set_debug(sync: int, timeout_ns: int = 0) -> int:
    """Process-wide debug settings of attention_fwd: sync 1 / 0 / -1 (= as
    GEMM_DEBUG_SYNC says) and the limit of every bounded device wait (0 = default)."""
    return int(lib().attention_set_debug(int(sync), int(timeout_ns)))


def gemm_build_checked() -> int:
    """1 when the loaded library is the checked build."""
    return int(lib().gemm_build_checked())


def gemm_plan_device_status(plan: int) -> int:
    """The device status word the plan's last debug-sync gemm_run read."""
    w = ctypes.c_int32(0)
    st = int(lib().gemm_plan_device_status(plan, ctypes.byref(w)))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan_device_status")
    return int(w.value)


def gemm_partition(M: int, N: int, K: int, world: int, rank: int,
                   axis: int = GEMM_SPLIT_AUTO) -> dict:
    """The slice of C = A @ B (rows or columns) that `rank` of `world` computes."""
    sl = GemmSlice()
    st = lib().gemm_partition(M, N, K, world, rank, axis, ctypes.byref(sl))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_partition")
    return sl.as_dict()


def gemm_run_slice(plan: int, sl: dict, A: int, lda: int, B: int, ldb: int, C: int, ldc: int,
                   M: int, N: int, K: int, dtype: int, stream: int = 0) -> int:
    """One slice of C = A @ B on the whole matrices' layouts (raw pointers); returns the status."""
    s = GemmSlice(**sl)
    return int(lib().gemm_run_slice(plan, ctypes.byref(s), A, lda, B, ldb, C, ldc, M, N, K,
                                    dtype, stream))


def gemm_plan_set_staging(plan: int, enabled: bool) -> int:
    return int(lib().gemm_plan_set_staging(plan, int(enabled)))


def gemm_tile_coord(t: int, tiles_m: int, tiles_n: int, group: int) -> tuple[int, int]:
    tm, tn = ctypes.c_int64(), ctypes.c_int64()
    st = lib().gemm_tile_coord(t, tiles_m, tiles_n, group, ctypes.byref(tm), ctypes.byref(tn))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_tile_coord")
    return tm.value, tn.value


def gemm_wait_selftest(timeout_us: int, stream: int = 0) -> int:
    return int(lib().gemm_wait_selftest(timeout_us, stream))


def gemm_noop_launch(grid: int, cluster: int = 1, stream: int = 0) -> int:
    """Enqueue one kernel with no work, launched like the GEMM kernels (the launch floor)."""
    return int(lib().gemm_noop_launch(grid, cluster, stream))


def gemm_run_noalloc(A: int, lda: int, B: int, ldb: int, C: int, ldc: int, M: int, N: int,
                     K: int, dtype: int, stream: int = 0) -> int:
    """Small-M C = A @ B on the current device with no plan and no allocation (for
    callers that cannot allocate device memory); returns the gemm_status_t code."""
    return int(lib().gemm_run_noalloc(A, lda, B, ldb, C, ldc, M, N, K, dtype, stream))


def softmax_rows(X: int, ldx: int, Y: int, ldy: int, M: int, N: int, stream: int = 0) -> int:
    """Y = row-wise softmax of X (fp32, raw pointers as ints) on `stream`; returns the status."""
    return int(lib().softmax_rows(X, ldx, Y, ldy, M, N, stream))


def softmax_rows_query(X: int, ldx: int, Y: int, ldy: int, M: int, N: int) -> dict:
    cfg = SoftmaxConfig()
    st = lib().softmax_rows_query(X, ldx, Y, ldy, M, N, ctypes.byref(cfg))
    if st != GEMM_OK:
        raise GemmError(st, "softmax_rows_query")
    return cfg.as_dict()


def attention_fwd(Q: int, K: int, V: int, O: int, BH: int, seq: int, d: int, ld: int, hs: int,
                  ldo: int, hso: int, causal: int, dtype: int, out_type: int,
                  stream: int = 0) -> int:
    """O = softmax(Q K^T / sqrt(d) [causal]) V per head (raw pointers); returns the status."""
    return int(lib().attention_fwd(Q, K, V, O, BH, seq, d, ld, hs, ldo, hso, causal, dtype,
                                   out_type, stream))


def attention_fwd_query(Q: int, K: int, V: int, O: int, BH: int, seq: int, d: int, ld: int,
                        hs: int, ldo: int, hso: int, causal: int, dtype: int,
                        out_type: int) -> dict:
    cfg = AttentionConfig()
    st = lib().attention_fwd_query(Q, K, V, O, BH, seq, d, ld, hs, ldo, hso, causal, dtype,
                                   out_type, ctypes.byref(cfg))
    if st != GEMM_OK:
        raise GemmError(st, "attention_fwd_query")
    return cfg.as_dict()


# ------------------------------------------------------------------ torch convenience

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return GEMM_F16
    if t.dtype == torch.bfloat16:
        return GEMM_BF16
    raise TypeError(f"A and B must be float16 or bfloat16, got {t.dtype}")


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("matrices must be 2-D with unit inner stride (row-major)")
    return t.stride(0) if t.size(0) > 1 else max(t.stride(0), t.size(1))


def _operand(t) -> tuple[int, int]:
    """(op, ld) of a 2-D logical operand view: row-major storage is GEMM_OP_N; a
    transposed view of row-major storage (unit stride along dim 0) is GEMM_OP_T."""
    if t.dim() != 2:
        raise ValueError("matrices must be 2-D")
    if t.stride(1) == 1 and (t.size(0) <= 1 or t.stride(0) >= t.size(1)):
        return GEMM_OP_N, max(t.stride(0), t.size(1))
    if t.stride(0) == 1 and (t.size(1) <= 1 or t.stride(1) >= t.size(0)):
        return GEMM_OP_T, max(t.stride(1), t.size(0))
    raise ValueError("each operand must be row-major or a transposed view of row-major storage")


def _out_code(t) -> int:
    import torch
    codes = {torch.float32: GEMM_OUT_F32, torch.float16: GEMM_OUT_F16,
             torch.bfloat16: GEMM_OUT_BF16}
    if t.dtype not in codes:
        raise TypeError(f"C must be float32, float16 or bfloat16, got {t.dtype}")
    return codes[t.dtype]


class Plan:
    """Owns one C-ABI plan; ``run``/``matmul`` marshal torch tensors into gemm_run."""

    def __init__(self, device: int = 0):
        self.device = device
        self.handle = gemm_plan_create(device)

    def close(self):
        if self.handle:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_group(self, group: int):
        st = gemm_plan_set_group(self.handle, group)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_plan_set_group")

    def set_debug(self, sync: bool, timeout_ns: int = 0):
        st = gemm_plan_set_debug(self.handle, int(bool(sync)), timeout_ns)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_plan_set_debug")

    def device_status(self) -> int:
        return gemm_plan_device_status(self.handle)

    def set_staging(self, enabled: bool):
        st = gemm_plan_set_staging(self.handle, enabled)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_plan_set_staging")

    def force(self, kernel: int = 0, split_k: int = 0, block_n: int = 0):
        st = gemm_plan_force(self.handle, kernel, split_k, block_n)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_plan_force")

    def query(self, a, b, c, M=None, N=None, K=None) -> dict:
        M = a.size(0) if M is None else M
        K = a.size(1) if K is None else K
        N = b.size(1) if N is None else N
        return gemm_query(self.handle, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(),
                          _ld(c), M, N, K, _dtype_code(a))

    def run(self, a, b, c, M=None, N=None, K=None, stream=None) -> None:
        """c[:M, :N] = a[:M, :K] @ b[:K, :N] (fp32 c); raises GemmError on failure."""
        import torch
        if a.dtype != b.dtype:
            raise TypeError("A and B must have the same dtype")
        if c.dtype != torch.float32:
            raise TypeError("C must be float32")
        M = a.size(0) if M is None else M
        K = a.size(1) if K is None else K
        N = b.size(1) if N is None else N
        s = (torch.cuda.current_stream(a.device) if stream is None else stream).cuda_stream
        st = gemm_run(self.handle, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), c.data_ptr(),
                      _ld(c), M, N, K, _dtype_code(a), s)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_run")

    def run_ex(self, a, b, c, stream=None) -> None:
        """c = a @ b for logical views a (M x K), b (K x N), c (M x N): each of a, b
        row-major or a transposed view of row-major storage; c row-major fp32/fp16/bf16."""
        import torch
        if a.dtype != b.dtype:
            raise TypeError("A and B must have the same dtype")
        M, K = a.shape
        K2, N = b.shape
        if K != K2 or tuple(c.shape) != (M, N):
            raise ValueError(f"shapes {tuple(a.shape)} @ {tuple(b.shape)} -> {tuple(c.shape)}")
        op_a, lda = _operand(a)
        op_b, ldb = _operand(b)
        s = (torch.cuda.current_stream(a.device) if stream is None else stream).cuda_stream
        st = gemm_run_ex(self.handle, op_a, op_b, a.data_ptr(), lda, b.data_ptr(), ldb,
                         c.data_ptr(), _ld(c), _out_code(c), M, N, K, _dtype_code(a), s)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_run_ex")

    def query_ex(self, a, b, c) -> dict:
        M, K = a.shape
        N = b.shape[1]
        op_a, lda = _operand(a)
        op_b, ldb = _operand(b)
        return gemm_query_ex(self.handle, op_a, op_b, a.data_ptr(), lda, b.data_ptr(), ldb,
                             c.data_ptr(), _ld(c), _out_code(c), M, N, K, _dtype_code(a))

    def run_slice(self, a, b, c, sl: dict, stream=None) -> None:
        """The slice `sl` (from gemm_partition) of c = a @ b, all three the whole
        matrices (row-major fp16/bf16 a, b; fp32 c); raises GemmError on failure."""
        import torch
        if a.dtype != b.dtype:
            raise TypeError("A and B must have the same dtype")
        M, K = a.shape
        N = b.shape[1]
        s = (torch.cuda.current_stream(a.device) if stream is None else stream).cuda_stream
        st = gemm_run_slice(self.handle, sl, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                            c.data_ptr(), _ld(c), M, N, K, _dtype_code(a), s)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_run_slice")

    def matmul(self, a, b, out_dtype=None):
        """C = a @ b (fp32 by default); a and b may be transposed views."""
        import torch
        if a.size(1) != b.size(0):
            raise ValueError(f"inner dimensions differ: {tuple(a.shape)} @ {tuple(b.shape)}")
        c = torch.empty((a.size(0), b.size(1)), dtype=out_dtype or torch.float32,
                        device=a.device)
        self.run_ex(a, b, c)
        return c


_default_plans: dict = {}


def matmul(a, b, out_dtype=None):
    """C = A @ B for 2-D fp16/bf16 CUDA tensors (either may be a transposed view),
    fp32 accumulation, C in fp32 or `out_dtype`, through a per-device default plan."""
    dev = a.device.index or 0
    if dev not in _default_plans:
        _default_plans[dev] = Plan(dev)
    return _default_plans[dev].matmul(a, b, out_dtype)


def _rows_view(t, what):
    import torch
    if t.dtype != torch.float32:
        raise TypeError(f"{what} must be float32, got {t.dtype}")
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError(f"{what} must be 2-D with unit inner stride (row-major)")
    return max(t.stride(0), t.size(1)) if t.size(0) > 1 else max(t.size(1), 1)


def softmax(x, out=None, stream=None):
    """Row-wise softmax of a 2-D float32 CUDA tensor (each row on its own); `out`
    may be `x` itself (in place).  Raises GemmError on failure."""
    import torch
    ldx = _rows_view(x, "x")
    if out is None:
        out = torch.empty_like(x, memory_format=torch.contiguous_format)
    if tuple(out.shape) != tuple(x.shape):
        raise ValueError(f"out has shape {tuple(out.shape)}, x {tuple(x.shape)}")
    ldy = _rows_view(out, "out")
    s = (torch.cuda.current_stream(x.device) if stream is None else stream).cuda_stream
    st = softmax_rows(x.data_ptr(), ldx, out.data_ptr(), ldy, x.size(0), x.size(1), s)
    if st != GEMM_OK:
        raise GemmError(st, "softmax_rows")
    return out


def _heads_view(t, what):
    """(ld, head_stride) of a [BH, seq, d] view with unit stride along d."""
    if t.dim() != 3 or (t.size(2) > 1 and t.stride(2) != 1):
        raise ValueError(f"{what} must be [BH, seq, d] with unit stride along d")
    return t.stride(1), t.stride(0)


def attention(q, k, v, causal: bool = False, out=None, out_dtype=None, stream=None):
    """O = softmax(q k^T / sqrt(d)) v for [BH, seq, d] fp16/bf16 CUDA tensors (q, k, v
    with the same strides); with `causal`, key j counts for query i only if j <= i.
    O is fp32 unless `out_dtype` (or `out`) says otherwise."""
    import torch
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must have the same dtype")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"shapes differ: {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    lds = {_heads_view(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"))}
    if len(lds) != 1:
        raise ValueError("q, k and v must share one layout (strides)")
    ld, hs = lds.pop()
    BH, seq, d = q.shape
    if out is None:
        out = torch.empty((BH, seq, d), dtype=out_dtype or torch.float32, device=q.device)
    ldo, hso = _heads_view(out, "out")
    s = (torch.cuda.current_stream(q.device) if stream is None else stream).cuda_stream
    st = attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), BH, seq, d, ld,
                       hs, ldo, hso, int(bool(causal)), _dtype_code(q), _out_code(out), s)
    if st != GEMM_OK:
        raise GemmError(st, "attention_fwd")
    return out


def gather_c(c_local, M: int, N: int, K: int, axis: int = GEMM_SPLIT_AUTO, group=None):
    """All of C on every rank, from each rank's slice `c_local` (rows x cols of
    its gemm_partition slice, any device torch.distributed's backend handles):
    the slices are padded to the largest one, all-gathered, and placed.  This is
    the one collective of the partitioned GEMM, and only for callers that need
    all of C on every device; the slices themselves need no exchange."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    slices = [gemm_partition(M, N, K, world, r, axis) for r in range(world)]
    rows = max(sl["rows"] for sl in slices)
    cols = max(sl["cols"] for sl in slices)
    padded = torch.zeros(rows, cols, dtype=c_local.dtype, device=c_local.device)
    padded[:c_local.shape[0], :c_local.shape[1]] = c_local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    out = torch.empty(M, N, dtype=c_local.dtype, device=c_local.device)
    for sl, part in zip(slices, parts):
        out[sl["row0"]:sl["row0"] + sl["rows"], sl["col0"]:sl["col0"] + sl["cols"]] = \
            part[:sl["rows"], :sl["cols"]]
    return out
