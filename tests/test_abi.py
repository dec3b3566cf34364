"""The C ABI without a GPU: the library loads, exports every call that
include/mxfp8norm.h declares, and rejects bad arguments before any launch.
Only argument-checking paths are exercised here; nothing reaches the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp8norm.h")


@pytest.fixture(scope="module")
def mx():
    from mxfp8_block_scaled_rmsnorm_gb300 import build
    build.build()
    import mxfp8_block_scaled_rmsnorm_gb300 as mx
    mx.library()
    return mx


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_calls():
    assert declared_functions() == sorted(
        ["rmsnorm_quant_mxfp8", "quant_mxfp8", "rmsnorm_quant_mxfp8_ex", "quant_mxfp8_ex",
         "add_rmsnorm_quant_mxfp8", "mxfp8_update_planes", "mm_mxfp8",
         "mm_mxfp8_workspace_size", "mm_mxfp8_static", "mm_mxfp8_quantized",
         "mxfp8_last_error",
         "mxfp8_abi_version", "mxfp8_rmsnorm_quant", "mxfp8_quant", "mxfp8_set_test_hook",
         "mxfp8_device_status"])


def test_library_exports_every_declared_symbol(mx):
    L = mx.library()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.mxfp8_abi_version() == 7


def test_desc_struct_layout_matches_header(mx):
    # 7 pointers, two int64, two float32: 80 bytes with no padding
    assert ctypes.sizeof(mx.MXFP8Desc) == 80
    assert mx.MXFP8Desc.rows.offset == 56 and mx.MXFP8Desc.eps.offset == 72


def _desc(mx, rows=32, cols=64, base=0x10000, **over):
    d = mx.MXFP8Desc()
    for i, f in enumerate(("x", "gamma", "normed", "q_row", "s_row", "q_col", "s_col")):
        setattr(d, f, base + 0x100000 * (i + 1))
    d.rows, d.cols, d.eps, d.weight_offset = rows, cols, 1e-6, 0.0
    for k, v in over.items():
        setattr(d, k, v)
    return d


def _call(mx, fn, descs, n=None, rowwise=1, columnwise=1):
    L = mx.library()
    arr = (mx.MXFP8Desc * max(1, len(descs)))(*descs)
    rc = getattr(L, fn)(arr, len(descs) if n is None else n, rowwise, columnwise, None)
    return rc, L.mxfp8_last_error().decode()


@pytest.mark.parametrize("fn", ["rmsnorm_quant_mxfp8", "quant_mxfp8"])
def test_argument_errors(mx, fn):
    L = mx.library()
    assert getattr(L, fn)(None, 1, 1, 1, None) == -4
    rc, msg = _call(mx, fn, [_desc(mx)], n=0)
    assert rc == -4 and "outside" in msg
    rc, _ = _call(mx, fn, [_desc(mx)], n=257)
    assert rc == -4
    rc, msg = _call(mx, fn, [_desc(mx)], rowwise=0, columnwise=0)
    assert rc == -3 and "neither" in msg
    rc, msg = _call(mx, fn, [_desc(mx, cols=48)])
    assert rc == -2 and "multiple of 32" in msg
    rc, msg = _call(mx, fn, [_desc(mx, rows=33)])
    assert rc == -2 and "columnwise" in msg
    rc, _ = _call(mx, fn, [_desc(mx, rows=-1)])
    assert rc == -2
    rc, msg = _call(mx, fn, [_desc(mx, x=None)])
    assert rc == -1 and "x is NULL" in msg
    rc, msg = _call(mx, fn, [_desc(mx, q_row=0x10008)])
    assert rc == -1 and "q_row is not 16-byte aligned" in msg
    rc, msg = _call(mx, fn, [_desc(mx), _desc(mx, s_col=None)])
    assert rc == -1 and "entry 1: s_col" in msg
    rc, _ = _call(mx, fn, [_desc(mx, rows=1 << 40)])
    assert rc == -2


def test_fused_needs_gamma_and_normed_but_quant_does_not(mx):
    rc, msg = _call(mx, "rmsnorm_quant_mxfp8", [_desc(mx, gamma=None)])
    assert rc == -1 and "gamma" in msg
    rc, msg = _call(mx, "rmsnorm_quant_mxfp8", [_desc(mx, normed=0x10004)])
    assert rc == -1 and "normed" in msg
    # quant ignores gamma/normed: the first failing check must be elsewhere
    rc, msg = _call(mx, "quant_mxfp8", [_desc(mx, gamma=None, normed=None, x=None)])
    assert rc == -1 and "x is NULL" in msg


def test_disabled_plane_pointers_are_ignored(mx):
    # rows % 32 != 0 is fine without the columnwise plane, whose pointers may be NULL;
    # an odd-shaped entry later in the list must still be caught
    rc, msg = _call(mx, "quant_mxfp8", [_desc(mx, rows=33, q_col=None, s_col=None),
                                        _desc(mx, cols=40)], columnwise=0)
    assert rc == -2 and "entry 1" in msg


def test_empty_entries_launch_nothing(mx):
    rc, msg = _call(mx, "rmsnorm_quant_mxfp8", [_desc(mx, rows=0, x=None), _desc(mx, cols=0)])
    assert rc == 0 and msg == ""


def test_unknown_scale_layout_is_rejected(mx):
    L = mx.library()
    arr = (mx.MXFP8Desc * 1)(_desc(mx))
    for fn in ("rmsnorm_quant_mxfp8_ex", "quant_mxfp8_ex"):
        assert getattr(L, fn)(arr, 1, 1, 1, 7, None) == -3
        assert "scale layout" in L.mxfp8_last_error().decode()


def test_residual_call_checks_its_pointers(mx):
    L = mx.library()
    arr = (mx.MXFP8Desc * 1)(_desc(mx))
    assert L.add_rmsnorm_quant_mxfp8(arr, None, 1, 1, 1, 0, None) == -1
    res = (mx.MXFP8Residual * 1)()
    res[0].residual = 0x10008
    assert L.add_rmsnorm_quant_mxfp8(arr, res, 1, 1, 1, 0, None) == -1
    assert "residual is not 16-byte aligned" in L.mxfp8_last_error().decode()
    res[0].residual, res[0].residual_out = None, 0x20004
    assert L.add_rmsnorm_quant_mxfp8(arr, res, 1, 1, 1, 0, None) == -1
    assert "residual_out" in L.mxfp8_last_error().decode()


@pytest.mark.parametrize("fn", ["mxfp8_rmsnorm_quant", "mxfp8_quant"])
def test_alias_names_check_like_the_main_calls(mx, fn):
    L = mx.library()
    getattr(L, fn).argtypes = [ctypes.POINTER(mx.MXFP8Desc), ctypes.c_int, ctypes.c_int,
                               ctypes.c_int, ctypes.c_void_p]
    assert getattr(L, fn)(None, 1, 1, 1, None) == -4
    rc, msg = _call(mx, fn, [_desc(mx, cols=48)])
    assert rc == -2 and "multiple of 32" in msg


HOOK_FAIL_LAUNCH, HOOK_MAX_CLUSTER = 1, 2


@pytest.fixture
def fail_launches(mx):
    """Every launch reports a CUDA error (injected on the host: nothing reaches
    a device, so this runs without a GPU)."""
    L = mx.library()
    L.mxfp8_set_test_hook.argtypes = [ctypes.c_int, ctypes.c_int]
    L.mxfp8_set_test_hook.restype = ctypes.c_int
    prev = L.mxfp8_set_test_hook(HOOK_FAIL_LAUNCH, 1)
    yield L
    L.mxfp8_set_test_hook(HOOK_FAIL_LAUNCH, prev)


def test_test_hook_arguments(mx):
    L = mx.library()
    L.mxfp8_set_test_hook.argtypes = [ctypes.c_int, ctypes.c_int]
    assert L.mxfp8_set_test_hook(99, 1) == -3
    assert "unknown test hook" in L.mxfp8_last_error().decode()
    assert L.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, -1) == -3
    assert L.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, 4) == 0
    assert L.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, 0) == 4
    # the GEMM hooks: form 0-2, split 0-3; out-of-range values change nothing
    HOOK_GEMM_FORM, HOOK_GEMM_SPLITS = 3, 4
    assert L.mxfp8_set_test_hook(HOOK_GEMM_FORM, 3) == -3
    assert L.mxfp8_set_test_hook(HOOK_GEMM_FORM, 2) == 0
    assert L.mxfp8_set_test_hook(HOOK_GEMM_FORM, 0) == 2
    assert L.mxfp8_set_test_hook(HOOK_GEMM_SPLITS, 4) == -3
    assert L.mxfp8_set_test_hook(HOOK_GEMM_SPLITS, 3) == 0
    assert L.mxfp8_set_test_hook(HOOK_GEMM_SPLITS, 0) == 3


@pytest.mark.parametrize("fn", ["rmsnorm_quant_mxfp8", "quant_mxfp8", "mxfp8_rmsnorm_quant",
                                "mxfp8_quant"])
def test_launch_error_is_reported_as_err_cuda(mx, fail_launches, fn):
    getattr(fail_launches, fn).argtypes = [ctypes.POINTER(mx.MXFP8Desc), ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    for n in (1, 9):  # the small and the large launch table
        rc, msg = _call(mx, fn, [_desc(mx, base=0x10000 * (i + 1)) for i in range(n)])
        assert rc == -5 and msg.startswith("kernel launch failed") and "invalid argument" in msg
    # argument errors still come first
    rc, _ = _call(mx, fn, [_desc(mx, cols=48)])
    assert rc == -2


def test_launch_error_in_the_other_calls(mx, fail_launches):
    L = fail_launches
    arr = (mx.MXFP8Desc * 1)(_desc(mx))
    for fn in ("rmsnorm_quant_mxfp8_ex", "quant_mxfp8_ex"):
        for layout in (0, 1, 2):
            assert getattr(L, fn)(arr, 1, 1, 1, layout, None) == -5
            assert "invalid argument" in L.mxfp8_last_error().decode()
    res = (mx.MXFP8Residual * 1)()
    res[0].residual, res[0].residual_out = 0x900000, 0xA00000
    assert L.add_rmsnorm_quant_mxfp8(arr, res, 1, 1, 1, 0, None) == -5
    src = (mx.MXFP8Planes * 1)()
    dst = (mx.MXFP8Planes * 1)()
    for i, o in enumerate((src[0], dst[0])):
        o.q_row, o.s_row, o.q_col, o.s_col = (0x100000 * (4 * i + k + 1) for k in range(4))
        o.rows, o.cols = 64, 64
    assert L.mxfp8_update_planes(src, dst, 1, 1, 1, 2, None) == -5
    assert "invalid argument" in L.mxfp8_last_error().decode()
    # the matrix multiply reports MXFP8_ERR_CUDA before it launches anything:
    # at its first launch, or earlier where no driver can make its TMA tensor
    # maps (this container has no GPU driver)
    rc = L.mm_mxfp8(0x100000, 256, 256, 0x200000, 0x300000, 256, 0x400000, 0x500000,
                    1 << 22, None)
    msg = L.mxfp8_last_error().decode()
    assert rc == -5 and ("invalid argument" in msg or "tensor map" in msg), msg
    rc = L.mm_mxfp8_quantized(0x100000, 0x600000, 256, 256, 0x200000, 0x300000, 256,
                              0x400000, None)
    msg = L.mxfp8_last_error().decode()
    assert rc == -5 and ("invalid argument" in msg or "tensor map" in msg), msg


def test_mm_quantized_rejects_before_launch(mx):
    """Shape and pointer checks of the GEMM-only entry (no GPU needed: each
    returns before any CUDA call)."""
    L = mx.library()
    A, S, W, WS, O = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000
    for M, K, N in [(0, 256, 256), (256, 0, 256), (256, 48, 256), (256, 256, 24),
                    (-1, 256, 256), (256, 256, 1 << 31)]:
        assert L.mm_mxfp8_quantized(A, S, M, K, W, WS, N, O, None) == -2, (M, K, N)
        assert "mm_mxfp8 needs" in L.mxfp8_last_error().decode()
    for bad in range(5):
        ptrs = [A, S, W, WS, O]
        ptrs[bad] = 0 if bad % 2 == 0 else ptrs[bad] + 16
        assert L.mm_mxfp8_quantized(ptrs[0], ptrs[1], 256, 256, ptrs[2], ptrs[3], 256,
                                    ptrs[4], None) == -1, bad
        assert "256-byte aligned" in L.mxfp8_last_error().decode()


def test_bounds_checking_build_is_made_and_exports_the_same_calls(mx):
    from mxfp8_block_scaled_rmsnorm_gb300 import build
    import subprocess
    assert os.path.exists(build.BOUNDS_LIB_PATH)
    B = ctypes.CDLL(build.BOUNDS_LIB_PATH)
    for name in declared_functions():
        assert hasattr(B, name), name
    # the bounds build holds the device status word of its checks; the normal
    # build does not (its checks compile to nothing)
    sym = lambda path: subprocess.run(["nm", "-C", path], capture_output=True,
                                      text=True).stdout
    assert "mx::g_bounds_status" in sym(build.BOUNDS_LIB_PATH)
    assert "mx::g_bounds_status" not in sym(build.LIB_PATH)
