"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

The bar (written in each check):
 - quantize outputs (E4M3 codes, E8M0 scale bytes) are bit-exact;
 - normed bf16 is within 1 bf16 step of the oracle's float32 result;
 - the fused quantize equals a standalone quantize of the fused normed output,
   byte for byte, and the standalone quantize equals the oracle on any bf16
   input (fed here with the oracle's own normed output), so the fused planes
   equal the oracle applied to the GPU's normed output; wherever the GPU normed
   block equals the oracle's, the fused planes equal the oracle's planes too.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import bf16_bits, to_dev, ulp_dist_bf16
from parity import NORMED_ULP_TOL, assert_quant_exact, check_fused, quant_dev, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()


# ------------------------------------------------------------ quantize ---

def test_quant_list_random_shapes_one_launch():
    shapes = [(32, 256), (64, 4128), (96, 160), (32, 32), (128, 1120), (32, 7168)]
    wl = W.random_weights(shapes, seed=21, scale=1.0)
    got = quant_dev([t.x for t in wl.tensors])
    for t, g in zip(wl.tensors, got):
        assert_quant_exact(g, oracle.quant_mxfp8(t.x), str(t.shape))


@pytest.mark.parametrize("rowwise,columnwise", [(True, False), (False, True)])
def test_quant_single_plane(rowwise, columnwise):
    wl = W.random_weights([(64, 384)], seed=22, scale=3.0)
    got = quant_dev([wl.tensors[0].x], rowwise, columnwise)[0]
    assert_quant_exact(got, oracle.quant_mxfp8(wl.tensors[0].x, rowwise, columnwise))


def test_quant_rowwise_ragged_rows():
    wl = W.random_weights([(1, 64), (45, 256), (33, 1024)], seed=23, scale=0.5)
    got = quant_dev([t.x for t in wl.tensors], True, False)
    for t, g in zip(wl.tensors, got):
        assert_quant_exact(g, oracle.quant_mxfp8(t.x, True, False), str(t.shape))


def _reachable_blocks():
    """Every finite bf16 value against every block exponent it can meet, laid
    out as 32-element blocks led by the largest bf16 of that exponent."""
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    fin = allb[((allb >> 7) & 0xFF) != 0xFF]
    mag = np.abs(oracle.bf16_value(fin))
    rows = []
    for e in range(-127, 120):
        lim = -118 if e == -127 else e + 9
        vals = fin[mag < 2.0**lim]
        carrier = np.uint16(((lim + 127) << 7) - 1)
        n = -(-vals.size // 31) * 31
        vals = np.concatenate([vals, np.zeros(n - vals.size, np.uint16)]).reshape(-1, 31)
        rows.append(np.concatenate([np.full((vals.shape[0], 1), carrier, np.uint16), vals], 1))
    blocks = np.concatenate(rows)
    return blocks[: blocks.shape[0] - blocks.shape[0] % 32]


def test_quant_exhaustive_bf16_values_and_exponents():
    """The kernel's element encoder against the oracle over all ~8.4M
    (value, exponent) pairs, through the rowwise and the columnwise plane."""
    blocks = _reachable_blocks()
    want_r = oracle.quant_mxfp8(blocks, True, False, threads=None)
    got_r = quant_dev([blocks], True, False)[0]
    assert_quant_exact(got_r, want_r, "rowwise")
    t = np.ascontiguousarray(blocks.T)
    want_c = oracle.quant_mxfp8(t, False, True, threads=None)
    got_c = quant_dev([t], False, True)[0]
    assert_quant_exact(got_c, want_c, "columnwise")


def test_quant_special_blocks():
    R, C = 64, 128
    x = np.zeros((R, C), np.uint16)
    x[0, 32:64] = 0x8000                                   # negative zeros
    x[1, 64:96] = np.arange(1, 33, dtype=np.uint16)        # sub-normals only
    x[2, 96:128] = 0x7F7F                                  # largest finite bf16
    x[3, 0:32] = oracle.bf16_round(np.ldexp(1.0, np.arange(-16, 16)))
    x[4:36, 5] = 0x3FFF                                    # column block of 1.9921875
    got = quant_dev([x])[0]
    assert_quant_exact(got, oracle.quant_mxfp8(x))
    assert got[0][0, 32:64].tolist() == [0x80] * 32
    assert got[1][2, 3] == 246


# ------------------------------------------------------------- fused ---

@pytest.mark.parametrize("R,C", [(32, 32), (64, 1024), (96, 2080), (32, 8192),
                                 (64, 9216), (32, 19968), (160, 3072)])
def test_fused_both_planes_shapes(R, C):
    # wide rows take several passes per CTA (each re-reads its earlier passes from L2)
    wl = W.random_fused(R, C, seed=R * 7 + C, eps=1e-5, offset=0.25)
    check_fused(wl)


@pytest.mark.parametrize("R,C", [(24576, 1056), (12288, 2080)])
def test_fused_two_pass_slices_ragged_columns(R, C):
    """Launches of more stripes than the device holds CTAs at once keep two
    512-column passes per CTA (smaller ones take one pass per CTA in larger
    clusters, which the shapes above cover); here with slices that end in a
    partial pass (C = 1056: two CTAs of 544 columns; 2080: three of 704).
    Checked on whole 32-row stripes at the start, middle and end."""
    wl = W.random_fused(R, C, seed=R + C, eps=1e-6, offset=0.5)
    mid = R // 2 - (R // 2) % 32
    rows = np.concatenate([np.arange(0, 64), np.arange(mid, mid + 64), np.arange(R - 64, R)])
    check_fused(wl, rows_sample=rows)


@pytest.mark.parametrize("rowwise,columnwise", [(True, False), (False, True)])
def test_fused_single_plane(rowwise, columnwise):
    wl = W.random_fused(64, 2048, seed=5, scale=4.0)
    outs, _ = check_fused(wl, rowwise, columnwise)
    o = outs[0]
    assert (o.q_row is None) != rowwise and (o.q_col is None) != columnwise


@pytest.mark.parametrize("R", [1, 17, 50])
def test_fused_rowwise_ragged_rows(R):
    wl = W.random_fused(R, 1024, seed=R, scale=0.1)
    check_fused(wl, True, False)


def test_fused_list_mixed_widths_one_launch():
    wls = [W.random_fused(32, c, seed=c) for c in (256, 4096, 1024, 8192)]
    wl = W.Workload("mix", True, True, True, [w.tensors[0] for w in wls])
    check_fused(wl)


def test_fused_stress_recipe_small():
    check_fused(W.stress(256, 4096, seed=31))


def test_fused_degenerate_rows():
    C = 1024
    x = np.zeros((64, C), np.uint16)
    x[1] = 0x3F80                                          # all ones
    x[2, ::2] = 0x0001                                     # sub-normal row
    x[3] = oracle.bf16_round(np.full(C, 3e38))             # x^2 overflows float32
    x[4, 7] = 0x4000                                       # a single 2.0
    g = oracle.bf16_round(np.where(np.arange(C) % 3 == 0, -1.0, 0.5))
    wl = W.Workload("degenerate", True, True, True, [W.Tensor2D(x, g, 1e-6, 0.0)])
    check_fused(wl)


def test_fused_outputs_respect_guard_bands():
    """Outputs sit inside larger buffers filled with a canary; no byte outside
    the logical extent may change (stands in for a memory checker)."""
    R, C = 96, 2080
    wl = W.random_fused(R, C, seed=77)
    t = wl.tensors[0]
    pad = 4096
    dev = "cuda"

    def carve(nbytes):
        buf = torch.full((nbytes + 2 * pad,), 0xA5, dtype=torch.uint8, device=dev)
        return buf, buf[pad:pad + nbytes]

    sizes = {"normed": R * C * 2, "q_row": R * C, "s_row": R * C // 32,
             "q_col": R * C, "s_col": R * C // 32}
    bufs = {k: carve(v) for k, v in sizes.items()}
    out = mx.NormQuantOut(
        bufs["normed"][1].view(torch.bfloat16).view(R, C),
        bufs["q_row"][1].view(R, C), bufs["s_row"][1].view(R, C // 32),
        bufs["q_col"][1].view(R, C), bufs["s_col"][1].view(R // 32, C))
    mx.rmsnorm_quant_mxfp8(to_dev(t.x), to_dev(t.gamma), t.eps, t.offset, out=[out])
    sync()
    for k, (buf, _) in bufs.items():
        b = buf.cpu().numpy()
        assert np.all(b[:pad] == 0xA5) and np.all(b[-pad:] == 0xA5), k
    ref = oracle.rmsnorm_f32(t.x, t.gamma, t.eps, t.offset)
    assert ulp_dist_bf16(bf16_bits(out.normed), ref).max() <= NORMED_ULP_TOL


def test_repeat_calls_are_deterministic():
    wl = W.random_fused(128, 8192, seed=9)
    t = wl.tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)
    a = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset)
    b = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset)
    sync()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_launch_on_a_side_stream():
    wl = W.random_fused(64, 4096, seed=10)
    t = wl.tensors[0]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        x, g = to_dev(t.x), to_dev(t.gamma)
        o = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset)
    s.synchronize()
    ref = oracle.rmsnorm_f32(t.x, t.gamma, t.eps, t.offset)
    assert ulp_dist_bf16(bf16_bits(o.normed), ref).max() <= NORMED_ULP_TOL


def test_error_codes_on_device():
    x = torch.zeros((32, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MXFP8Error) as e:
        mx.quant_mxfp8(x)
    assert e.value.code == -2
    x = torch.zeros((33, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mx.MXFP8Error) as e:
        mx.quant_mxfp8(x, True, True)
    assert e.value.code == -2
    o = mx.quant_mxfp8(x, True, False)          # rowwise only: 33 rows are fine
    sync()
    assert o.q_col is None and o.q_row.shape == (33, 64)
    with pytest.raises(mx.MXFP8Error) as e:
        mx.quant_mxfp8(torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda"), False, False)
    assert e.value.code == -3


def test_max_list_length_one_launch():
    shapes = [(32, 32 * (1 + i % 9)) for i in range(256)]
    wl = W.random_weights(shapes, seed=12, scale=1.0)
    got = quant_dev([t.x for t in wl.tensors])
    for t, g in zip(wl.tensors, got):
        assert_quant_exact(g, oracle.quant_mxfp8(t.x), str(t.shape))


def test_cuda_graph_capture_and_replay():
    """Caller-owned outputs and a by-value descriptor table make the call
    capturable: replaying the graph on new input contents gives the eager result."""
    wl1 = W.random_fused(64, 4096, seed=41)
    wl2 = W.random_fused(64, 4096, seed=42)
    t1, t2 = wl1.tensors[0], wl2.tensors[0]
    x, g = to_dev(t1.x), to_dev(t1.gamma)
    out = mx.make_outputs(x, True, True, True)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mx.rmsnorm_quant_mxfp8(x, g, t1.eps, t1.offset, out=[out])
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mx.rmsnorm_quant_mxfp8(x, g, t1.eps, t1.offset, out=[out])
    x.copy_(to_dev(t2.x))
    graph.replay()
    sync()
    eager = mx.rmsnorm_quant_mxfp8(to_dev(t2.x), g, t1.eps, t1.offset)
    sync()
    for a, b in zip(out, eager):
        assert torch.equal(a, b)


def test_row_chunked_calls_equal_one_call():
    """Rows are independent in 32-row blocks: calling on row ranges (as a
    pipelined host path does) gives the same bytes as one call."""
    t = W.stress(512, 4096, seed=17).tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)
    whole = mx.rmsnorm_quant_mxfp8(x, g, t.eps, t.offset)
    parts = mx.make_outputs(x, True, True, True)
    for r0, r1 in ((0, 96), (96, 352), (352, 512)):
        view = mx.NormQuantOut(parts.normed[r0:r1], parts.q_row[r0:r1], parts.s_row[r0:r1],
                               parts.q_col[r0:r1], parts.s_col[r0 // 32:r1 // 32])
        mx.rmsnorm_quant_mxfp8(x[r0:r1], g, t.eps, t.offset, out=[view])
    sync()
    for a, b in zip(whole, parts):
        assert torch.equal(a, b)
