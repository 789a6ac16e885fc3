"""C-ABI library checks that need no GPU: it loads, exports every function the
header declares, and its host-side logic (status strings, argument checks that
precede any CUDA call, the scheduler's tile order) behaves as documented."""
import ctypes
import os
import re

import pytest

import dense_gemm_05_gb300 as g
from oracle import schedule

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    g.build()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += [n for n in re.findall(r"GEMM_API\s+[\w\s\*]*?\b(\w+)\s*\(", text)
                      if not n.startswith("__")]
    return names


def test_header_declares_the_binding_functions():
    assert sorted(declared_functions()) == sorted(g.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(g.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    assert g.status_string(0) == "GEMM_OK"
    assert g.status_string(1) == "GEMM_ERR_INVALID_ARG"
    assert g.status_string(5) == "GEMM_ERR_TIMEOUT"
    assert g.status_string(6) == "GEMM_ERR_BOUNDS"
    assert g.status_string(99) == "GEMM_ERR_UNKNOWN"


def test_null_plan_is_rejected_before_any_cuda_call():
    assert g.gemm_run(None, 0, 1, 0, 1, 0, 1, 1, 1, 1, g.GEMM_F16, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan_destroy(None) == g.GEMM_OK
    assert g.gemm_plan_set_group(None, 8) == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_plan_force(None, 0, 0, 0) == g.GEMM_ERR_INVALID_ARG
    assert g.lib().gemm_plan_create(None, 0) == g.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("tm,tn,grp", [(4, 4, 2), (5, 3, 2), (64, 32, 8), (7, 11, 3), (13, 1, 8),
                                       (1, 9, 4), (32, 32, 16), (9, 5, 1), (6, 6, 0), (3, 17, 0)])
def test_tile_order_matches_the_oracle(tm, tn, grp):
    for t in range(tm * tn):
        want = (schedule.row_major_tile(t, tn) if grp == 0
                else schedule.group_major_tile(t, tm, tn, grp))
        assert g.gemm_tile_coord(t, tm, tn, grp) == want


def test_tile_order_rejects_bad_arguments():
    with pytest.raises(g.GemmError):
        g.gemm_tile_coord(16, 4, 4, 2)
    with pytest.raises(g.GemmError):
        g.gemm_tile_coord(-1, 4, 4, 2)
    with pytest.raises(g.GemmError):
        g.gemm_tile_coord(0, 0, 4, 2)


def test_plan_create_without_a_usable_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = g.lib().gemm_plan_create(ctypes.byref(h), 0)
    assert st in (g.GEMM_ERR_CUDA, g.GEMM_ERR_INVALID_ARG) and not h.value


def test_softmax_argument_checks_need_no_gpu():
    """Argument errors and empty shapes are decided before any CUDA call."""
    sr = g.softmax_rows
    assert sr(0, 1, 0, 1, -1, 4) == g.GEMM_ERR_INVALID_ARG          # negative M
    assert sr(0, 1, 0, 1, 4, -1) == g.GEMM_ERR_INVALID_ARG          # negative N
    assert sr(0, 8, 0, 8, 0, 8) == g.GEMM_OK                        # M == 0: no-op
    assert sr(0, 8, 0, 8, 8, 0) == g.GEMM_OK                        # N == 0: no-op
    assert sr(0, 8, 4096, 8, 2, 8) == g.GEMM_ERR_INVALID_ARG        # null X
    assert sr(4096, 7, 65536, 8, 2, 8) == g.GEMM_ERR_INVALID_ARG    # ldx < N
    assert sr(4096, 8, 65536, 7, 2, 8) == g.GEMM_ERR_INVALID_ARG    # ldy < N
    assert sr(4098, 8, 65536, 8, 2, 8) == g.GEMM_ERR_INVALID_ARG    # X not 4-byte aligned
    assert sr(4096, 8, 4096 + 16, 8, 2, 8) == g.GEMM_ERR_INVALID_ARG  # partial overlap
    assert sr(4096, 8, 4096, 16, 2, 8) == g.GEMM_ERR_INVALID_ARG    # same start, other pitch
    assert sr(4096, 1 << 31, 1 << 40, 1 << 31, 2, 1 << 31) == g.GEMM_ERR_UNSUPPORTED  # N > 2^31-1
    with pytest.raises(g.GemmError):
        g.softmax_rows_query(0, 1, 0, 1, -1, 1)
    assert g.softmax_rows_query(0, 1, 0, 1, 0, 5)["path_name"] == "none"


def test_attention_argument_checks_need_no_gpu():
    """Argument errors and empty shapes are decided before any CUDA call."""
    af = g.attention_fwd
    a, b, c, o = 1 << 20, 2 << 20, 3 << 20, 4 << 20            # distinct, aligned, unused
    F16, BF16 = g.GEMM_F16, g.GEMM_BF16
    F32 = g.GEMM_OUT_F32
    assert af(a, b, c, o, 0, 128, 64, 64, 8192, 64, 8192, 1, BF16, F32, 0) == g.GEMM_OK       # BH 0
    assert af(a, b, c, o, 2, 0, 64, 64, 8192, 64, 8192, 1, BF16, F32, 0) == g.GEMM_OK        # seq 0
    assert af(a, b, c, o, -1, 8, 64, 64, 512, 64, 512, 0, BF16, F32, 0) == g.GEMM_ERR_INVALID_ARG
    assert af(0, b, c, o, 2, 8, 64, 64, 512, 64, 512, 0, BF16, F32, 0) == g.GEMM_ERR_INVALID_ARG
    assert af(a, b, c, o, 2, 8, 64, 32, 512, 64, 512, 0, BF16, F32, 0) == g.GEMM_ERR_INVALID_ARG  # ld < d
    assert af(a + 8, b, c, o, 2, 8, 64, 64, 512, 64, 512, 0, F16, F32, 0) == g.GEMM_ERR_INVALID_ARG  # align
    assert af(a, b, c, o, 2, 8, 96, 96, 768, 96, 768, 0, F16, F32, 0) == g.GEMM_ERR_UNSUPPORTED    # d
    assert af(a, b, c, o, 2, 8, 64, 68, 544, 64, 512, 0, F16, F32, 0) == g.GEMM_ERR_UNSUPPORTED   # ld % 8
    assert af(a, b, c, o, 2, 8, 64, 64, 512, 64, 512, 0, 7, F32, 0) == g.GEMM_ERR_UNSUPPORTED     # dtype
    assert af(a, b, c, o, 2, 8, 64, 64, 512, 64, 512, 0, F16, 9, 0) == g.GEMM_ERR_UNSUPPORTED     # out
    assert af(a, b, c, b + 256, 2, 8, 64, 64, 512, 64, 512, 0, F16, F32, 0) == g.GEMM_ERR_INVALID_ARG  # O on K
    with pytest.raises(g.GemmError):
        g.attention_fwd_query(a, b, c, o, -1, 8, 64, 64, 512, 64, 512, 0, F16, F32)
    cfg = g.attention_fwd_query(a, b, c, o, 3, 1000, 64, 64, 64000, 64, 64000, 1, BF16, F32)
    # 8 query blocks of 128 per head, two per CTA (d = 64) or one (d = 128)
    assert cfg["grid_x"] == 4 and cfg["grid_y"] == 3 and cfg["block_q"] == 128 and cfg["causal"] == 1
    cfg = g.attention_fwd_query(a, b, c, o, 3, 1000, 128, 128, 128000, 128, 128000, 0, BF16, F32)
    assert cfg["grid_x"] == 8 and cfg["head_dim"] == 128
    # The longest sequence whose row and key indices stay inside int32 (one
    # head, rows 8 elements apart, the four tensors far apart), and one longer.
    longest = (1 << 31) - 256
    far = [(1 << 44) * i for i in (1, 2, 3, 4)]
    cfg = g.attention_fwd_query(*far, 1, longest, 64, 64, 0, 64, 0, 0, BF16, F32)
    assert cfg["grid_x"] == (longest + 255) // 256
    assert af(*far, 1, longest + 1, 64, 64, 0, 64, 0, 0, BF16, F32, 0) == g.GEMM_ERR_UNSUPPORTED
