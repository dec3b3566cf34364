"""GPU: paths that the library takes only under conditions a healthy GB300 does
not produce, forced through the testing hooks of include/mxfp8norm.h.

- The one-CTA path of the fused kernel (no thread-block cluster: the row sums
  of a 32-row stripe stay in one CTA, which walks the whole row in 512-column
  passes) is what a device that co-schedules no cluster gets. Capped at one
  CTA per stripe, the fused call must meet the same parity bar as everywhere
  else: planes equal to the oracle's quantize of the GPU's own normed, normed
  within one bf16 step of the oracle's float32 RMSNorm.
- A launch that the CUDA runtime rejects: every call reports MXFP8_ERR_CUDA
  with the runtime's text, and once the injection stops the same buffers work
  (the rejection is not sticky).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import bf16_bits, to_dev, u8
from parity import assert_quant_exact, check_fused, sync

pytestmark = pytest.mark.gpu

HOOK_FAIL_LAUNCH, HOOK_MAX_CLUSTER = 1, 2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = mx.library()
    L.mxfp8_set_test_hook.argtypes = [ctypes.c_int, ctypes.c_int]
    L.mxfp8_set_test_hook.restype = ctypes.c_int
    return L


@pytest.fixture
def one_cta(lib):
    prev = lib.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, 1)
    yield
    lib.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, prev)


@pytest.mark.parametrize("C", [4096, 20480])
def test_fused_one_cta_per_stripe(one_cta, C):
    wl = W.random_fused(96, C, seed=C + 5, scale=3.0, eps=1e-5, offset=0.25)
    _, stats = check_fused(wl)
    assert stats[0] < 1e-2, stats


def test_fused_one_cta_residual_and_tiled_scales(one_cta):
    R, C = 64, 8192
    wl = W.random_fused(R, C, seed=77, scale=2.0)
    t = wl.tensors[0]
    r_bits = W.random_weights([(R, C)], seed=78, scale=1.0).tensors[0].x
    h, o = mx.add_rmsnorm_quant_mxfp8(to_dev(t.x), to_dev(r_bits), to_dev(t.gamma), t.eps,
                                      t.offset, scale_layout="mma")
    sync()
    h_ref = oracle.residual_add(t.x, r_bits)
    assert np.array_equal(bf16_bits(h), h_ref)
    q_row, s_row, q_col, s_col = oracle.quant_mxfp8(bf16_bits(o.normed))
    assert np.array_equal(u8(o.q_row), q_row) and np.array_equal(u8(o.q_col), q_col)
    assert np.array_equal(u8(o.s_row).ravel(), oracle.scales_to_mma(s_row))
    assert np.array_equal(u8(o.s_col).ravel(), oracle.scales_to_mma(s_col, columnwise=True))


def test_rejected_launch_reports_err_cuda_and_is_not_sticky(lib):
    wl = W.random_fused(64, 1024, seed=3)
    t = wl.tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)
    out = mx.make_outputs(x, True, True, True)
    wout = mx.make_outputs(x, False, True, True)
    prev = lib.mxfp8_set_test_hook(HOOK_FAIL_LAUNCH, 1)
    try:
        calls = [
            lambda: mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset, out=[out]),
            lambda: mx.quant_mxfp8(x, out=[wout]),
            lambda: mx.add_rmsnorm_quant_mxfp8(x, x, g, t.eps, t.offset, out=[out]),
            lambda: mx.update_planes(wout, mx.make_outputs(x, False, True, True, "padded")),
        ]
        for call in calls:
            with pytest.raises(mx.MXFP8Error) as e:
                call()
            assert e.value.code == -5 and "invalid argument" in str(e.value)
    finally:
        lib.mxfp8_set_test_hook(HOOK_FAIL_LAUNCH, prev)
    mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset, out=[out])
    sync()
    want = oracle.quant_mxfp8(bf16_bits(out.normed))
    assert_quant_exact(tuple(u8(v) for v in out[1:]), want, "after the rejected launches")
