"""Parity checks shared by the GPU tests (CUDA path against the CPU oracle).

``check_fused`` checks one fused call four ways: (0) its planes equal the
oracle's quantize of the GPU's own normed output, byte for byte; (1) they equal
the GPU's standalone quantize of that normed; (2) normed is within one bf16
step of the oracle's float32 RMSNorm; (3) the GPU's standalone quantize of the
oracle's normed equals the oracle's planes; (4) the fused planes equal the
oracle's planes wherever the normed block matches the oracle's.
"""
import numpy as np
import torch

import oracle
import mxfp8_block_scaled_rmsnorm_gb300 as mx
from helpers import (block_equal_colwise, block_equal_rowwise, bf16_bits, to_dev, u8,
                     ulp_dist_bf16)

NORMED_ULP_TOL = 1


def sync():
    torch.cuda.synchronize()


def quant_dev(bits_list, rowwise=True, columnwise=True):
    outs = mx.quant_mxfp8([to_dev(b) for b in bits_list], rowwise, columnwise)
    sync()
    return [tuple(u8(t) for t in o) for o in outs]


def assert_quant_exact(got, want, tag=""):
    for g, w, name in zip(got, want, ("q_row", "s_row", "q_col", "s_col")):
        if w is None:
            assert g is None
            continue
        bad = np.flatnonzero(g != w)
        assert bad.size == 0, f"{tag} {name}: {bad.size} bytes differ, first at {bad[:5]}"


def check_fused(wl, rowwise=True, columnwise=True, threads=None, rows_sample=None):
    """Run the fused call on every tensor of ``wl`` and check it (see module doc)."""
    xs = [to_dev(t.x) for t in wl.tensors]
    gs = [to_dev(t.gamma) for t in wl.tensors]
    outs = mx.rmsnorm_quant_mxfp8(xs, gs, [t.eps for t in wl.tensors],
                                  [t.offset for t in wl.tensors], rowwise, columnwise)
    sync()
    stats = []
    for t, o, xd in zip(wl.tensors, outs, xs):
        # (1) fused planes == standalone quantize of the fused normed (GPU only)
        s = mx.quant_mxfp8(o.normed, rowwise, columnwise)
        sync()
        for name in ("q_row", "s_row", "q_col", "s_col"):
            a, b = getattr(o, name), getattr(s, name)
            assert (a is None) == (b is None)
            if a is not None:
                assert torch.equal(a, b), f"fused {name} != standalone quantize of normed"
        normed = bf16_bits(o.normed)
        R = t.x.shape[0]
        rows = np.arange(R) if rows_sample is None else rows_sample
        x_s = np.ascontiguousarray(t.x[rows])
        # (0) fused planes == the oracle's quantize of the GPU's own bf16 normed,
        # byte for byte on every checked row (the Mojo page's description: the
        # quantize reads the bf16 that lands in outputs_normed). The oracle is a
        # checker here: its input is the GPU's output, its answer its own.
        R_q = rows.size - (rows.size % 32 if columnwise else 0)
        sel_q = rows[:R_q]
        want = oracle.quant_mxfp8(np.ascontiguousarray(normed[sel_q]), rowwise, columnwise,
                                  threads=threads)
        got = (u8(o.q_row)[sel_q] if rowwise else None,
               u8(o.s_row)[sel_q] if rowwise else None,
               u8(o.q_col)[sel_q] if columnwise else None,
               u8(o.s_col)[sel_q.reshape(-1, 32)[:, 0] // 32] if columnwise else None)
        assert_quant_exact(got, want, "fused planes vs oracle quantize of the GPU normed")
        # (2) normed within 1 bf16 step of the oracle's float32 RMSNorm
        ref = oracle.rmsnorm_f32(x_s, t.gamma, t.eps, t.offset, threads=threads)
        d = ulp_dist_bf16(normed[rows], ref)
        assert d.max() <= NORMED_ULP_TOL, f"normed off by {d.max()} ulp"
        # (3) standalone GPU quantize of the oracle's normed == oracle quantize
        R_s = ref.shape[0] - (ref.shape[0] % 32 if columnwise else 0)
        ref_q = oracle.quant_mxfp8(ref[:R_s], rowwise, columnwise, threads=threads)
        got_q = quant_dev([ref[:R_s]], rowwise, columnwise)[0]
        assert_quant_exact(got_q, ref_q, "standalone on oracle normed")
        # (4) fused planes == oracle planes wherever the normed block matches
        sel = rows[:R_s]
        if rowwise:
            eq = block_equal_rowwise(normed[sel], ref[:R_s])
            qr, sr = u8(o.q_row)[sel], u8(o.s_row)[sel]
            assert np.array_equal(sr[eq], ref_q[1][eq])
            m = np.repeat(eq, 32, axis=1)
            assert np.array_equal(qr[m], ref_q[0][m])
        if columnwise:
            eq = block_equal_colwise(normed[sel], ref[:R_s])
            stripes = sel.reshape(-1, 32)[:, 0] // 32
            sc = u8(o.s_col)[stripes]
            assert np.array_equal(sc[eq], ref_q[3][eq])
            m = np.repeat(eq, 32, axis=0)
            assert np.array_equal(u8(o.q_col)[sel][m], ref_q[2][m])
        stats.append(float((d > 0).mean()))
    return outs, stats
