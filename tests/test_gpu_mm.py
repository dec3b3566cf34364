"""GPU: the MXFP8 matrix multiply consumer (x quantized on the fly, weight
pre-quantized, this library's tcgen05 block-scaled GEMM) against the oracle's
float64 value of the same quantized product. After every product the
library's device status must read 0 (no wait of the GEMM's pipeline gave up).

Tolerance, elementwise: |out - ref| <= 2^-8 |ref| + 2^-16 (|A| |B|^T): one bf16
rounding of the output plus float32 accumulation. A different activation
quantization (a step off in a code or a scale) moves terms by >= 2^-4
relative, far outside it.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import to_dev
from parity import sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()


def _abs_bound(x, w):
    qx, sx, _, _ = oracle.quant_mxfp8(x, True, False)
    qw, sw, _, _ = oracle.quant_mxfp8(w, True, False)
    return np.abs(oracle.dequantize_rowwise(qx, sx)) @ np.abs(oracle.dequantize_rowwise(qw, sw)).T


@pytest.mark.parametrize("M,N,K", [(256, 384, 1024), (200, 128, 512), (1, 16, 32),
                                   (33, 256, 7168), (1024, 4096, 4096),
                                   # ragged in all three: partial 256-row and
                                   # 256-column tiles, K % 128 == 32; the
                                   # general form (M past the swapped form's
                                   # limit, or its row blocks over more than
                                   # one wave) and the swapped form with
                                   # several 128-row activation blocks
                                   (2100, 272, 1056), (2000, 2064, 4000), (2100, 16, 32),
                                   (1000, 2064, 4000), (200, 272, 1056),
                                   # M <= 128 (the swapped-operand form): MMA
                                   # widths 32, 64 and 128, K split over two or
                                   # three pairs (few output blocks) or not,
                                   # partial last K steps, and the first M of
                                   # the general form
                                   (16, 4096, 4096), (48, 2048, 14336), (64, 1040, 896),
                                   (5, 16, 32), (17, 272, 1056), (32, 14336, 640),
                                   (64, 512, 640), (65, 512, 1024), (128, 4096, 14336),
                                   (100, 2064, 4000), (96, 16, 32), (128, 14336, 640),
                                   (127, 1040, 896), (129, 512, 1024),
                                   # K split with a partial last K step, MMA
                                   # widths 128 and 32
                                   (100, 2064, 14016), (17, 272, 14048), (33, 512, 4000),
                                   # two 128-row activation blocks and a K split
                                   (256, 1040, 14016)])
def test_mm_matches_oracle(M, N, K):
    x = W.random_fused(M, K, seed=M + K, scale=2.0).tensors[0].x
    w = W.random_weights([(N, K)], seed=N + K).tensors[0].x
    wq = mx.quantize_weight_for_mm(to_dev(w))
    out = mx.mm_mxfp8(to_dev(x), wq.q_row, wq.s_row)
    sync()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.mm_mxfp8(x, w)
    bound = 2.0**-8 * np.abs(ref) + 2.0**-16 * _abs_bound(x, w) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    assert mx.device_status() == 0


@pytest.mark.slow
def test_mm_full_size_sampled_rows():
    """8192 x 14336 x 4096, the shape bench.py --mm times, in the same launch
    configuration (one persistent grid of CTA pairs walking 1792 tiles): up to
    128 sampled rows (the first and last rows of the first and last 256-row
    tiles, and random ones) of the whole output against the oracle."""
    M, N, K = 8192, 14336, 4096
    rng = np.random.default_rng(7)
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = W.to_bf16_bits(0.02 * rng.standard_normal((N, K), dtype=np.float32))
    wq = mx.quantize_weight_for_mm(to_dev(w))
    out = mx.mm_mxfp8(to_dev(x), wq.q_row, wq.s_row)
    sync()
    assert mx.device_status() == 0
    rows = np.unique(np.concatenate([[0, 127, 128, 255, M - 256, M - 129, M - 128, M - 1],
                                     rng.choice(M, 120, replace=False)]))
    got = out[torch.from_numpy(rows).to(out.device)].double().cpu().numpy()
    qx, sx, _, _ = oracle.quant_mxfp8(np.ascontiguousarray(x[rows]), True, False, threads=None)
    qw, sw, _, _ = oracle.quant_mxfp8(w, True, False, threads=None)
    A, B = oracle.dequantize_rowwise(qx, sx), oracle.dequantize_rowwise(qw, sw)
    ref = A @ B.T
    bound = 2.0**-8 * np.abs(ref) + 2.0**-16 * (np.abs(A) @ np.abs(B).T) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def test_mm_reuses_weight_and_workspace_and_matches_scaled_mm():
    M, N, K = 128, 256, 2048
    x1 = to_dev(W.random_fused(M, K, seed=1).tensors[0].x)
    x2 = to_dev(W.random_fused(M, K, seed=2).tensors[0].x)
    w = to_dev(W.random_weights([(N, K)], seed=3).tensors[0].x)
    wq = mx.quantize_weight_for_mm(w)
    ws = torch.empty(mx.mm_mxfp8_workspace_size(M, K), dtype=torch.uint8, device="cuda")
    o1 = mx.mm_mxfp8(x1, wq.q_row, wq.s_row, workspace=ws)
    o2 = mx.mm_mxfp8(x2, wq.q_row, wq.s_row, workspace=ws)
    o1b = mx.mm_mxfp8(x1, wq.q_row, wq.s_row, workspace=ws)
    sync()
    assert torch.equal(o1, o1b) and not torch.equal(o1, o2)


def test_mm_argument_errors():
    x = torch.zeros((16, 48), dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros((16, 48), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((4096,), dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXFP8Error) as e:
        mx.mm_mxfp8(x, wq, ws)
    assert e.value.code == -2
    x = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros((24, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXFP8Error) as e:
        mx.mm_mxfp8(x, wq, ws)
    assert e.value.code == -2
    wq = torch.zeros((16, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXFP8Error) as e:
        mx.mm_mxfp8(x, wq, ws, workspace=torch.zeros((64,), dtype=torch.uint8, device="cuda"))
    assert e.value.code == -2


@pytest.mark.parametrize("M,N,K", [(256, 512, 4096), (200, 272, 1056), (33, 16, 32),
                                   (16, 4096, 4096), (64, 2064, 14016)])
def test_norm_quant_feeds_gemm(M, N, K):
    """rmsnorm_quant_mxfp8 with tiled scales, then mm_mxfp8_quantized on its
    rowwise plane: the activation codes match the oracle's quantize of the
    normed bf16 byte for byte, the product is within the bound against the
    oracle's float64 product of the two quantized operands, and it equals
    (byte for byte) mm_mxfp8 of the normed bf16, which quantizes it again."""
    t = W.random_fused(M, K, seed=M + 3 * K, scale=2.0).tensors[0]
    w = W.random_weights([(N, K)], seed=N + 5 * K).tensors[0].x
    wq = mx.quantize_weight_for_mm(to_dev(w))
    nq = mx.rmsnorm_quant_mxfp8(to_dev(t.x), to_dev(t.gamma), t.eps, t.offset, True, False,
                                scale_layout="mma")
    out = mx.mm_mxfp8_quantized(nq.q_row, nq.s_row, wq.q_row, wq.s_row)
    again = mx.mm_mxfp8(nq.normed, wq.q_row, wq.s_row)
    sync()
    assert mx.device_status() == 0
    normed = nq.normed.view(torch.int16).cpu().numpy().view(np.uint16)
    qx, sx, _, _ = oracle.quant_mxfp8(normed, True, False)
    assert np.array_equal(nq.q_row.cpu().numpy(), qx)
    qw, sw, _, _ = oracle.quant_mxfp8(w, True, False)
    A, B = oracle.dequantize_rowwise(qx, sx), oracle.dequantize_rowwise(qw, sw)
    ref = A @ B.T
    got = out.double().cpu().numpy()
    bound = 2.0**-8 * np.abs(ref) + 2.0**-16 * (np.abs(A) @ np.abs(B).T) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_mm_quantized_argument_errors():
    xq = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((24, 64), dtype=torch.uint8, device="cuda")
    s = torch.zeros((4096,), dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXFP8Error) as e:
        mx.mm_mxfp8_quantized(xq, s, wq, s)
    assert e.value.code == -2
    with pytest.raises(ValueError):
        mx.mm_mxfp8_quantized(xq, s, torch.zeros((16, 32), dtype=torch.uint8, device="cuda"), s)


@pytest.mark.parametrize("M,N,K", [(2100, 272, 1056), (1000, 2064, 4000), (16, 4096, 4096),
                                   (128, 4096, 4096), (17, 272, 14048)])
def test_mm_is_deterministic_across_calls_and_streams(M, N, K):
    """The GEMM accumulates every output in a fixed order (K steps in turn,
    four 32-element blocks each; in the swapped-operand form, four accumulators or one and
    the K split's partial sums added in pair order), so repeated calls give the same
    bytes, on the default stream and on a side stream alike."""
    x = to_dev(W.random_fused(M, K, seed=11, scale=2.0).tensors[0].x)
    wq = mx.quantize_weight_for_mm(to_dev(W.random_weights([(N, K)], seed=12).tensors[0].x))
    first = mx.mm_mxfp8(x, wq.q_row, wq.s_row)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        again = mx.mm_mxfp8(x, wq.q_row, wq.s_row, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    third = mx.mm_mxfp8(x, wq.q_row, wq.s_row)
    sync()
    assert mx.device_status() == 0
    assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    assert torch.equal(first.view(torch.int16), third.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 16, 32), (5, 272, 1056), (16, 4096, 4096), (31, 512, 640),
                                   (32, 1040, 896), (33, 2064, 4000), (48, 2048, 14336),
                                   (63, 272, 14048), (64, 14336, 640), (64, 512, 8192)])
def test_mm_equals_quantize_then_quantized_gemm(M, N, K):
    """mm_mxfp8 on bf16 x gives the bytes of quant_mxfp8 (tiled scales)
    followed by mm_mxfp8_quantized, and that quantize equals the oracle's bit
    for bit, at decode-sized M (the swapped-operand form, with and without a
    K split). Rows of x are scaled by 2^-60 .. 2^60, with zero and sub-normal
    blocks, so that scale bytes across the range, the zero-scale rule and
    saturation are all taken."""
    x_bits = W.wide_range(M, K, seed=M * 7 + K)
    x = to_dev(x_bits)
    wq = mx.quantize_weight_for_mm(to_dev(W.random_weights([(N, K)], seed=N + K).tensors[0].x))
    fused = mx.mm_mxfp8(x, wq.q_row, wq.s_row)
    xq = mx.quant_mxfp8(x, True, False, scale_layout="mma")
    two = mx.mm_mxfp8_quantized(xq.q_row, xq.s_row, wq.q_row, wq.s_row)
    sync()
    assert mx.device_status() == 0
    qx, _, _, _ = oracle.quant_mxfp8(x_bits, True, False)
    assert np.array_equal(xq.q_row.cpu().numpy(), qx)
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(16, 14336, 4096), (1, 4096, 14336), (64, 2048, 4096),
                                   (128, 4096, 4096)])
def test_mm_reads_the_weight_written_just_before(M, N, K):
    """mm_mxfp8's GEMM fetches the first ring stages of the weight before its
    dependency wait (the activation quantize before it writes only the
    scratch, and started after all earlier work). So a weight quantized into
    the same buffers by the launch right before each call, with no
    synchronization in between, must give the product of that new weight:
    each call equals the same call repeated after everything has finished."""
    x = to_dev(W.random_fused(M, K, seed=21, scale=1.0).tensors[0].x)
    ws = [to_dev(W.random_weights([(N, K)], seed=30 + i).tensors[0].x) for i in range(4)]
    wq = mx.quantize_weight_for_mm(ws[0])
    outs = []
    for i in range(8):
        mx.quant_mxfp8(ws[i % 4], True, False, out=wq, scale_layout="mma")
        outs.append(mx.mm_mxfp8(x, wq.q_row, wq.s_row))
    sync()
    assert mx.device_status() == 0
    for i in range(4):
        fresh = mx.quantize_weight_for_mm(ws[i])
        want = mx.mm_mxfp8_quantized(*_act(x), fresh.q_row, fresh.s_row)
        sync()
        for j in (i, i + 4):
            assert torch.equal(outs[j].view(torch.int16), want.view(torch.int16)), (i, j)


def _act(x):
    q = mx.quant_mxfp8(x, True, False, scale_layout="mma")
    return q.q_row, q.s_row
