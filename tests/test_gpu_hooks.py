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
- The matrix multiply in a form or K split the planner would not choose for
  the shape: the 256 x 256-tile form for decode-sized M, the swapped-operand
  form over several waves of tiles, and K splits whose clusters each walk
  several output blocks (the hand-over of partial sums across tiles). Each
  must meet the GEMM's bound against the oracle.
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

HOOK_FAIL_LAUNCH, HOOK_MAX_CLUSTER, HOOK_GEMM_FORM, HOOK_GEMM_SPLITS = 1, 2, 3, 4


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


@pytest.mark.parametrize("M,N,K,form,splits", [
    (16, 2064, 4000, 1, 0),    # decode-sized M in the 256 x 256-tile form
    (300, 20480, 1056, 2, 0),  # swapped form, 3 activation blocks x 80 weight blocks: 4 waves
    (16, 28672, 1056, 0, 3),   # three pairs per K range, 112 blocks: several per cluster
    (200, 20480, 1056, 2, 2),  # two pairs, 2 activation blocks x 80 weight blocks
    (64, 272, 96, 0, 3),       # one K step: the split falls back to one pair
])
def test_gemm_forced_form_and_split(lib, M, N, K, form, splits):
    x = W.random_fused(M, K, seed=M + N, scale=2.0).tensors[0].x
    w = W.random_weights([(N, K)], seed=N + K).tensors[0].x
    wq = mx.quantize_weight_for_mm(to_dev(w))
    prev_form = lib.mxfp8_set_test_hook(HOOK_GEMM_FORM, form)
    prev_splits = lib.mxfp8_set_test_hook(HOOK_GEMM_SPLITS, splits)
    try:
        out = mx.mm_mxfp8(to_dev(x), wq.q_row, wq.s_row)
        sync()
    finally:
        lib.mxfp8_set_test_hook(HOOK_GEMM_FORM, prev_form)
        lib.mxfp8_set_test_hook(HOOK_GEMM_SPLITS, prev_splits)
    assert mx.device_status() == 0
    qx, sx, _, _ = oracle.quant_mxfp8(x, True, False)
    qw, sw, _, _ = oracle.quant_mxfp8(w, True, False)
    A, B = oracle.dequantize_rowwise(qx, sx), oracle.dequantize_rowwise(qw, sw)
    ref = A @ B.T
    got = out.double().cpu().numpy()
    bound = 2.0**-8 * np.abs(ref) + 2.0**-16 * (np.abs(A) @ np.abs(B).T) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
