"""GPU: mm_mxfp8_static, the matrix multiply for callers that cannot allocate
device memory (its scratch is a fixed array inside the library), called
through the C ABI twice in a row and compared with mm_mxfp8 (caller-provided
workspace) on the same operands.

Tolerance, as for the mm_mxfp8 parity tests: each output within
2^-8 |ref| + 2^-16 (|A| |B|^T) of the float64 value of the quantized product;
two such outputs are within twice that of each other.

This file is collected last on purpose, and passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # MXFP8_MM_STATIC_SCRATCH_BYTES in include/mxfp8norm.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = mx.library()
    L.mm_mxfp8_static.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.c_void_p, ctypes.c_void_p]
    L.mm_mxfp8_static.restype = ctypes.c_int
    return L


def _static(L, x, wq, out):
    M, K = x.shape
    N = wq.q_row.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.mm_mxfp8_static(x.data_ptr(), M, K, wq.q_row.data_ptr(), wq.s_row.data_ptr(), N,
                           out.data_ptr(), stream)
    return rc, L.mxfp8_last_error().decode()


def _bounds(x_bits, w_bits):
    qx, sx, _, _ = oracle.quant_mxfp8(x_bits, True, False)
    qw, sw, _, _ = oracle.quant_mxfp8(w_bits, True, False)
    A, B = oracle.dequantize_rowwise(qx, sx), oracle.dequantize_rowwise(qw, sw)
    ref = A @ B.T
    return ref, 2.0**-8 * np.abs(ref) + 2.0**-16 * (np.abs(A) @ np.abs(B).T) + 1e-30


@pytest.mark.parametrize("M,N,K", [(200, 256, 1024), (1024, 512, 4096)])
def test_static_matches_workspace_entry_point_twice(lib, M, N, K):
    w_bits = W.random_weights([(N, K)], seed=N + K).tensors[0].x
    wq = mx.quantize_weight_for_mm(to_dev(w_bits))
    # two calls in a row on new operands; every tensor is allocated up front, so
    # that the device's free memory can be compared across the second call
    xs_bits = [W.random_fused(M, K, seed=M + c, scale=2.0).tensors[0].x for c in (1, 2)]
    xs = [to_dev(b) for b in xs_bits]
    outs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in xs]
    torch.cuda.synchronize()
    free = []
    for call, (x, out_s) in enumerate(zip(xs, outs)):
        torch.cuda.empty_cache()
        free.append(torch.cuda.mem_get_info()[0])
        rc, msg = _static(lib, x, wq, out_s)
        assert rc == 0, msg
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    # the second call (after the first call's set-up) takes no device memory
    assert free[3] == free[2], f"free device memory changed by {free[2] - free[3]} bytes"
    for call, (x_bits, x, out_s) in enumerate(zip(xs_bits, xs, outs)):
        out_w = mx.mm_mxfp8(x, wq.q_row, wq.s_row)
        torch.cuda.synchronize()
        ref, bound = _bounds(x_bits, w_bits)
        got_s = out_s.double().cpu().numpy()
        got_w = out_w.double().cpu().numpy()
        assert np.all(np.abs(got_s - ref) <= bound), f"call {call}"
        assert np.all(np.abs(got_s - got_w) <= 2 * bound), f"call {call}"


def test_static_rejects_problems_beyond_its_scratch(lib):
    M, K, N = 8192, 4096 + 32, 16  # M * K alone exceeds 32 MiB
    assert M * K > SCRATCH_BYTES
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    wq = mx.quantize_weight_for_mm(torch.zeros((N, K), dtype=torch.bfloat16, device="cuda"))
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    rc, msg = _static(lib, x, wq, out)
    assert rc == -2 and "static scratch" in msg


def _act_bytes(M, K):
    """Scratch the static entry needs: the quantized activation (codes, then
    tiled scales), each part rounded up to 256 bytes (include/mxfp8norm.h)."""
    a256 = lambda v: (v + 255) // 256 * 256
    return a256(M * K) + a256((M + 127) // 128 * 128 * ((K // 32 + 3) // 4) * 4)


def test_static_runs_just_under_and_rejects_just_over_its_scratch(lib):
    """A problem whose activation fills the array to within 32 KB runs and
    gives the same bytes as mm_mxfp8 (the GEMM takes no scratch of its own);
    the next size up is refused with MXFP8_ERR_SHAPE, not a CUDA error."""
    K, N = 4096, 16
    assert _act_bytes(7936, K) <= SCRATCH_BYTES < _act_bytes(8000, K)
    assert SCRATCH_BYTES - _act_bytes(7936, K) <= 32 << 10
    w_bits = W.random_weights([(N, K)], seed=5).tensors[0].x
    wq = mx.quantize_weight_for_mm(to_dev(w_bits))
    x = to_dev(W.random_fused(7936, K, seed=6, scale=2.0).tensors[0].x)
    out_s = torch.full((7936, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc, msg = _static(lib, x, wq, out_s)
    assert rc == 0, msg
    out_w = mx.mm_mxfp8(x, wq.q_row, wq.s_row)
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), out_w.view(torch.int16))
    x = torch.zeros((8000, K), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((8000, N), dtype=torch.bfloat16, device="cuda")
    rc, msg = _static(lib, x, wq, out)
    assert rc == -2 and "static scratch" in msg, msg
