"""GPU: scales in the tiled layout of a block-scaled GEMM operand.

1. Bit-exact against the oracle's compact scales scattered by the oracle's
   layout function, for both kernels, with padded row and column tiles.
2. Pinned to a library consumer: the planes and tiled scales go straight into
   PyTorch's block-scaled matrix multiply (torch._scaled_mm with
   float8_e8m0fnu scales, which runs cuBLASLt's 1x32-block-scaled GEMM), and
   the product must match a float64 product of the dequantized values. A wrong
   layout would scale elements by the wrong powers of two.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import bf16_bits, to_dev, u8
from parity import sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()


SHAPES = [(32, 32), (96, 160), (160, 1056), (256, 4096), (128, 8192 + 1024)]


@pytest.mark.parametrize("R,C", SHAPES)
def test_quant_mma_scales_match_oracle(R, C):
    t = W.random_weights([(R, C)], seed=R + C, scale=1.0).tensors[0]
    got = mx.quant_mxfp8(to_dev(t.x), scale_layout="mma")
    sync()
    q_row, s_row, q_col, s_col = oracle.quant_mxfp8(t.x)
    assert np.array_equal(u8(got.q_row), q_row) and np.array_equal(u8(got.q_col), q_col)
    assert np.array_equal(u8(got.s_row).ravel(), oracle.scales_to_mma(s_row))
    assert np.array_equal(u8(got.s_col).ravel(), oracle.scales_to_mma(s_col, columnwise=True))


# 24576 x 1056: more stripes than the device holds CTAs at once, so the
# two-pass slices (two CTAs of 544 columns) rather than one pass per CTA
@pytest.mark.parametrize("R,C", SHAPES + [(24576, 1056)])
def test_fused_mma_scales_match_compact_call(R, C):
    wl = W.random_fused(R, C, seed=3 * R + C, eps=1e-5, offset=0.5)
    t = wl.tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)
    a = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset)
    b = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset, scale_layout="mma")
    sync()
    assert torch.equal(a.normed, b.normed)
    assert torch.equal(a.q_row, b.q_row) and torch.equal(a.q_col, b.q_col)
    assert np.array_equal(u8(b.s_row).ravel(), oracle.scales_to_mma(u8(a.s_row)))
    assert np.array_equal(u8(b.s_col).ravel(), oracle.scales_to_mma(u8(a.s_col), columnwise=True))


def test_rowwise_only_ragged_rows_mma():
    t = W.random_weights([(45, 256)], seed=5, scale=2.0).tensors[0]
    got = mx.quant_mxfp8(to_dev(t.x), True, False, scale_layout="mma")
    sync()
    q_row, s_row, _, _ = oracle.quant_mxfp8(t.x, True, False)
    assert got.s_row.shape == (128, 8)
    assert np.array_equal(u8(got.s_row).ravel(), oracle.scales_to_mma(s_row))
    assert np.array_equal(u8(got.q_row), q_row)


# ---------------------------------------------------------------- GEMM pin ---

def _dequant(q: torch.Tensor, s_compact: torch.Tensor, along_rows: bool) -> torch.Tensor:
    """float64 values of codes q [R, C] with compact scales (rowwise [R, C/32]
    or columnwise [R/32, C])."""
    v = q.view(torch.float8_e4m3fn).double()
    e = s_compact.double() - 127.0
    scale = torch.exp2(e.repeat_interleave(32, dim=0 if along_rows else 1))
    return v * scale


def _scaled_mm(a, b, sa, sb):
    e8 = torch.float8_e8m0fnu
    try:
        return torch._scaled_mm(a.view(torch.float8_e4m3fn), b.view(torch.float8_e4m3fn),
                                sa.view(e8), sb.view(e8), out_dtype=torch.float32)
    except (RuntimeError, TypeError, NotImplementedError) as err:
        pytest.skip(f"no block-scaled _scaled_mm here: {str(err).splitlines()[0][:200]}")


def _check_close(out, ref, abs_ref):
    """Elementwise |out - ref| <= 1e-3 * (|A| |B|^T): loose enough for any
    float32 accumulation order, far too tight for a scale off by a factor 2."""
    err = (out.double() - ref).abs()
    assert bool((err <= 1e-3 * abs_ref + 1e-30).all()), (err / (abs_ref + 1e-30)).max().item()


@pytest.mark.parametrize("M,N,K", [(256, 384, 1024), (200, 128, 512)])
def test_rowwise_planes_feed_block_scaled_gemm(M, N, K):
    xs = W.random_fused(M, K, seed=M + K, scale=3.0).tensors[0]
    w = W.random_weights([(N, K)], seed=N + K).tensors[0]
    x, g = to_dev(xs.x), to_dev(xs.gamma)
    wd = to_dev(w.x)
    a = mx.rmsnorm_quant_mxfp8(x, g, xs.eps, xs.offset, True, False, scale_layout="mma")
    b = mx.quant_mxfp8(wd, True, False, scale_layout="mma")
    ac = mx.rmsnorm_quant_mxfp8(x, g, xs.eps, xs.offset, True, False)
    bc = mx.quant_mxfp8(wd, True, False)
    sync()
    out = _scaled_mm(a.q_row, b.q_row.t(), a.s_row, b.s_row)
    A, B = _dequant(ac.q_row, ac.s_row, False), _dequant(bc.q_row, bc.s_row, False)
    _check_close(out, A @ B.t(), A.abs() @ B.abs().t())


def test_columnwise_planes_feed_block_scaled_gemm():
    # X^T Y with the reduction over the 32-row blocks: the columnwise planes,
    # transposed to K-major for the library, with the tiled s_col as is
    R, Cx, Cy = 512, 256, 128
    X = to_dev(W.random_weights([(R, Cx)], seed=1, scale=1.0).tensors[0].x)
    Y = to_dev(W.random_weights([(R, Cy)], seed=2, scale=1.0).tensors[0].x)
    xq = mx.quant_mxfp8(X, False, True, scale_layout="mma")
    yq = mx.quant_mxfp8(Y, False, True, scale_layout="mma")
    xc = mx.quant_mxfp8(X, False, True)
    yc = mx.quant_mxfp8(Y, False, True)
    sync()
    a = xq.q_col.t().contiguous()                  # [Cx, R], K-major
    b = yq.q_col.t().contiguous().t()              # [R, Cy], column-major
    out = _scaled_mm(a, b, xq.s_col, yq.s_col)
    A, B = _dequant(xc.q_col, xc.s_col, True), _dequant(yc.q_col, yc.s_col, True)
    _check_close(out, A.t() @ B, A.abs().t() @ B.abs())


# ------------------------------------------------------ padded row-major ---

@pytest.mark.parametrize("R,C", SHAPES)
def test_padded_layout_matches_oracle_both_kernels(R, C):
    wl = W.random_fused(R, C, seed=5 * R + C, eps=1e-6, offset=0.0)
    t = wl.tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)
    a = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset)
    b = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset, scale_layout="padded")
    q = mx.quant_mxfp8(to_dev(t.x), scale_layout="padded")
    sync()
    assert torch.equal(a.q_row, b.q_row) and torch.equal(a.q_col, b.q_col)
    assert np.array_equal(u8(b.s_row), oracle.scales_to_padded(u8(a.s_row), R, C, False))
    assert np.array_equal(u8(b.s_col), oracle.scales_to_padded(u8(a.s_col), R, C, True))
    _, s_row, _, s_col = oracle.quant_mxfp8(t.x)
    assert np.array_equal(u8(q.s_row), oracle.scales_to_padded(s_row, R, C, False))
    assert np.array_equal(u8(q.s_col), oracle.scales_to_padded(s_col, R, C, True))
