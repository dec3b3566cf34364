"""GPU parity of the fused residual add + RMSNorm + MXFP8 call.

h = bf16(x + residual) must equal the oracle bit for bit (one rounding of the
exact sum on both sides); normed must be within 1 bf16 step of the oracle's
float32 RMSNorm of h; the planes must equal a standalone quantize of the GPU's
normed output byte for byte (whose own parity with the oracle is covered in
test_gpu_parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import bf16_bits, to_dev, ulp_dist_bf16
from parity import NORMED_ULP_TOL, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()


def _residual(shape, seed, scale=1.0):
    return W.random_weights([shape], seed=seed, scale=scale).tensors[0].x


def _check(t, r_bits, h_dev, o, rowwise=True, columnwise=True):
    h_ref = t.x if r_bits is None else oracle.residual_add(t.x, r_bits)
    if h_dev is not None:
        assert np.array_equal(bf16_bits(h_dev), h_ref), "residual_out differs from the oracle"
    ref = oracle.rmsnorm_f32(h_ref, t.gamma, t.eps, t.offset, threads=None)
    assert ulp_dist_bf16(bf16_bits(o.normed), ref).max() <= NORMED_ULP_TOL
    s = mx.quant_mxfp8(o.normed, rowwise, columnwise)
    sync()
    for name in ("q_row", "s_row", "q_col", "s_col"):
        a, b = getattr(o, name), getattr(s, name)
        assert (a is None) == (b is None)
        if a is not None:
            assert torch.equal(a, b), name


# Small launches take one pass per CTA in clusters of up to 16 (64 x 20480:
# 16 CTAs of 1280 columns, three passes each through the residual staging
# buffer); 24576 x 1056 is more stripes than the device holds CTAs at once,
# so two CTAs of 544 columns take two passes each, the second partial.
@pytest.mark.parametrize("R,C", [(32, 32), (64, 1024), (96, 2080), (32, 8192), (64, 9216),
                                 (256, 4096), (64, 20480), (24576, 1056)])
def test_residual_add_shapes(R, C):
    t = W.random_fused(R, C, seed=R + 5 * C, eps=1e-5, offset=0.25).tensors[0]
    r = _residual((R, C), seed=R * C + 1, scale=0.5)
    h, o = mx.add_rmsnorm_quant_mxfp8(to_dev(t.x), to_dev(r), to_dev(t.gamma), t.eps, t.offset)
    sync()
    _check(t, r, h, o)


@pytest.mark.parametrize("R", [1, 50])
def test_residual_rowwise_ragged_rows(R):
    t = W.random_fused(R, 1024, seed=R).tensors[0]
    r = _residual((R, 1024), seed=R + 100)
    h, o = mx.add_rmsnorm_quant_mxfp8(to_dev(t.x), to_dev(r), to_dev(t.gamma), t.eps, t.offset,
                                      True, False)
    sync()
    _check(t, r, h, o, True, False)


def test_residual_list_with_and_without_residual_and_output():
    shapes = [(64, 4096), (32, 1024), (96, 2048)]
    ts = [W.random_fused(R, C, seed=R + C).tensors[0] for R, C in shapes]
    rs = [_residual(shapes[0], 7), None, _residual(shapes[2], 9)]
    houts = [torch.empty(shapes[0], dtype=torch.bfloat16, device="cuda"),
             torch.empty(shapes[1], dtype=torch.bfloat16, device="cuda"), None]
    pairs = mx.add_rmsnorm_quant_mxfp8([to_dev(t.x) for t in ts],
                                       [None if r is None else to_dev(r) for r in rs],
                                       [to_dev(t.gamma) for t in ts], [t.eps for t in ts],
                                       [t.offset for t in ts], residual_out=houts)
    sync()
    for t, r, (h, o) in zip(ts, rs, pairs):
        _check(t, r, h, o)


def test_residual_matches_two_step_path():
    # one launch of add+norm+quant against the fused call applied to the GPU's
    # h: both run the same tile geometry and cluster split, so the float32
    # row sums are taken in the same order and every output is identical
    t = W.stress(256, 8192, seed=12).tensors[0]
    r = _residual((256, 8192), seed=13, scale=1e-3)
    x, g = to_dev(t.x), to_dev(t.gamma)
    h, o = mx.add_rmsnorm_quant_mxfp8(x, to_dev(r), g, t.eps, t.offset)
    o2 = mx.rmsnorm_quant_mxfp8(h, g, t.eps, t.offset)
    sync()
    for name in ("normed", "q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(getattr(o, name), getattr(o2, name)), name
    _check(t, r, h, o)
