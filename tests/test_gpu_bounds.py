"""GPU: the bounds-checking build of the library (libmxfp8norm_bounds.so, the
quantize kernels compiled with -DMXFP8_DEBUG_BOUNDS) on the parity suite's
small shapes. In that build every global access of the fused and quantize
kernels is checked against the extent that include/mxfp8norm.h states for its
buffer (given the entry's shape and scale layout); an access outside it is
skipped and recorded in the device status word instead of faulting.

Each case runs through both libraries on identical inputs: the bounds build
must record nothing (mxfp8_device_status == 0) and write the same bytes as the
normal build. This stands in for a memory checker (compute-sanitizer is closed
on this pool): it shows that no index of these launch geometries leaves the
buffers the contract defines.
"""
import contextlib
import os

import numpy as np
import pytest
import torch

import mxfp8_block_scaled_rmsnorm_gb300 as mx
from mxfp8_block_scaled_rmsnorm_gb300 import build as B
from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
from helpers import to_dev

pytestmark = pytest.mark.gpu

HOOK_MAX_CLUSTER = 2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    assert os.path.exists(B.BOUNDS_LIB_PATH), "build() makes the bounds-checking library too"


@contextlib.contextmanager
def bounds_library():
    """Route the binding's calls to the bounds-checking build."""
    saved = (mx._lib, mx.LIB_PATH)
    mx._lib, mx.LIB_PATH = None, B.BOUNDS_LIB_PATH
    try:
        L = mx.library()
        assert mx.device_status(clear=True) == 0
        yield L
    finally:
        mx._lib, mx.LIB_PATH = saved


def _fill(t: torch.Tensor, byte: int):
    t.view(torch.uint8).fill_(byte)


def _outs_like(xs, fused, rowwise, columnwise, layout):
    outs = [mx.make_outputs(x, fused, rowwise, columnwise, layout) for x in xs]
    for o in outs:  # the same known contents in both runs (padding is left untouched)
        for v in o:
            if v is not None:
                _fill(v, 0x5A)
    return outs


def _same(a, b, tag):
    for name, u, v in zip(a._fields, a, b):
        if u is None:
            assert v is None
            continue
        assert torch.equal(u.view(torch.uint8), v.view(torch.uint8)), f"{tag}: {name} differs"


def _both(run, tag):
    """run() -> list of output tuples; run it on both builds and compare."""
    want = run()
    torch.cuda.synchronize()
    with bounds_library():
        got = run()
        status = mx.device_status(clear=True)
    assert status == 0, f"{tag}: bounds-checking build recorded {status:#x}"
    for i, (a, b) in enumerate(zip(want, got)):
        _same(a, b, f"{tag} entry {i}")


SHAPES = [(32, 32), (64, 4128), (96, 160), (128, 1120), (32, 7168)]


@pytest.mark.parametrize("layout", ["compact", "mma", "padded"])
@pytest.mark.parametrize("planes", [(True, True), (True, False), (False, True)])
def test_fused_list(layout, planes):
    xs = [to_dev(W.random_weights([s], seed=i, scale=2.0).tensors[0].x)
          for i, s in enumerate(SHAPES)]
    gs = [to_dev(W.random_fused(1, s[1], seed=i).tensors[0].gamma) for i, s in enumerate(SHAPES)]

    def run():
        outs = _outs_like(xs, True, *planes, layout)
        return mx.rmsnorm_quant_mxfp8(xs, gs, 1e-5, 0.5, *planes, out=outs, scale_layout=layout)
    _both(run, f"fused {layout} {planes}")


@pytest.mark.parametrize("layout", ["compact", "mma", "padded"])
def test_fused_rowwise_ragged_rows(layout):
    shapes = [(1, 64), (45, 256), (33, 1024)]
    xs = [to_dev(W.random_weights([s], seed=10 + i).tensors[0].x) for i, s in enumerate(shapes)]
    gs = [to_dev(W.random_fused(1, s[1], seed=i).tensors[0].gamma) for i, s in enumerate(shapes)]

    def run():
        outs = _outs_like(xs, True, True, False, layout)
        return mx.rmsnorm_quant_mxfp8(xs, gs, 1e-6, 0.0, True, False, out=outs,
                                      scale_layout=layout)
    _both(run, f"fused ragged {layout}")


@pytest.mark.parametrize("C", [20480, 32800])
def test_fused_wide_rows(C):
    t = W.random_fused(64, C, seed=C).tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)

    def run():
        return mx.rmsnorm_quant_mxfp8([x], [g], t.eps, t.offset,
                                      out=_outs_like([x], True, True, True, "compact"))
    _both(run, f"fused wide {C}")


@pytest.mark.parametrize("layout", ["compact", "mma"])
@pytest.mark.parametrize("write_h", [True, False])
def test_residual(layout, write_h):
    t = W.random_fused(96, 8192, seed=5).tensors[0]
    r = W.random_weights([(96, 8192)], seed=6, scale=1.0).tensors[0].x
    x, g, rd = to_dev(t.x), to_dev(t.gamma), to_dev(r)

    def run():
        h = torch.empty_like(x) if write_h else None
        if h is not None:
            _fill(h, 0x5A)
        outs = _outs_like([x], True, True, True, layout)
        mx.add_rmsnorm_quant_mxfp8([x], [rd], [g], t.eps, t.offset, out=outs,
                                   residual_out=[h] if write_h else None, scale_layout=layout)
        hs = mx.QuantOut(h, None, None, None)
        return [outs[0], hs]
    _both(run, f"residual {layout} h={write_h}")


def test_fused_one_cta_path():
    t = W.random_fused(64, 4096, seed=8).tensors[0]
    x, g = to_dev(t.x), to_dev(t.gamma)

    def run():
        L = mx.library()
        prev = L.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, 1)
        try:
            return [mx.rmsnorm_quant_mxfp8([x], [g], t.eps, t.offset,
                                           out=_outs_like([x], True, True, True, "mma"),
                                           scale_layout="mma")[0]]
        finally:
            L.mxfp8_set_test_hook(HOOK_MAX_CLUSTER, prev)
    _both(run, "fused one CTA per stripe")


@pytest.mark.parametrize("layout", ["compact", "mma", "padded"])
def test_quant_list(layout):
    shapes = [(32, 256), (64, 4128), (96, 160), (32, 32), (128, 1120), (32, 7168)]
    xs = [to_dev(W.random_weights([s], seed=20 + i).tensors[0].x) for i, s in enumerate(shapes)]

    def run():
        outs = _outs_like(xs, False, True, True, layout)
        return mx.quant_mxfp8(xs, True, True, out=outs, scale_layout=layout)
    _both(run, f"quant {layout}")


def test_quant_rowwise_ragged_and_many_entries():
    rng = np.random.default_rng(3)
    shapes = [(int(32 * rng.integers(1, 5)) - int(rng.integers(0, 2)) * 7,
               int(32 * rng.integers(1, 40))) for _ in range(64)]
    xs = [to_dev(W.random_weights([s], seed=40 + i).tensors[0].x) for i, s in enumerate(shapes)]

    def run():
        outs = _outs_like(xs, False, True, False, "compact")
        return mx.quant_mxfp8(xs, True, False, out=outs)
    _both(run, "quant 64 ragged entries")
