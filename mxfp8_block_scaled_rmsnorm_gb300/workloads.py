"""Seeded synthetic inputs for the five benchmark workloads and for tests.

This module only draws random numbers and lays out bit patterns; it holds none
of the method's arithmetic. Values are drawn in float32 with NumPy's PCG64
generator and rounded to bf16 by PyTorch's float32 -> bfloat16 cast (a library
routine, round-to-nearest-even). Sub-normal bf16 inputs are written directly as
bit patterns.

Workload ``k`` (1..5) uses seed ``k - 1``. The recipes:

1. fused, rowwise only: x [256, 1024] ~ N(0, 1); gamma = 1 + 0.1 N(0, 1);
   eps 1e-6; offset 0.
2. fused, both planes: x [8192, 4096] ~ N(0, 1); exactly round(0.001 R C)
   positions, drawn without replacement, are multiplied by 100 in float32 before
   rounding; gamma = 0.1 N(0, 1); offset 1.0; eps 1e-5.
3. weight-only, both planes, one launch over four Llama-3-8B-like layer shapes
   [4096, 4096], [1024, 4096], [14336, 4096], [4096, 14336], each ~ N(0, 0.02).
4. fused, both planes, stress: x [32768, 8192]; row r is N(0, 1) * 2^k_r with
   k_r uniform in the integers [-20, 20]; 1% of the 32-element row blocks
   (floor(0.01 * R * C / 32), drawn without replacement) are set to +0 and a
   disjoint 1% hold random-sign bf16 sub-normals with fraction uniform in
   1..127 (magnitude below 2^-126); gamma = 1 + 0.1 N(0, 1); eps 1e-6; offset 0.
5. weight-only, both planes, one launch over 128 tensors ~ N(0, 0.02) with
   rows = 32 * U{1..128} and cols = 32 * U{8..224}.
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

BLOCK = 32


@dataclasses.dataclass
class Tensor2D:
    """One list entry: bf16 bits of x [R, C] and, for the fused map, gamma [C]."""
    x: np.ndarray
    gamma: np.ndarray | None = None
    eps: float = 1e-6
    offset: float = 0.0

    @property
    def shape(self):
        return self.x.shape


@dataclasses.dataclass
class Workload:
    name: str
    fused: bool
    rowwise: bool
    columnwise: bool
    tensors: list

    @property
    def elements(self) -> int:
        return int(sum(t.x.size for t in self.tensors))

    def algorithmic_bytes(self) -> int:
        return sum(algorithmic_bytes(t.shape[0], t.shape[1], self.fused,
                                     self.rowwise, self.columnwise)
                   for t in self.tensors)

    def sha256(self) -> str:
        h = hashlib.sha256()
        for t in self.tensors:
            h.update(np.ascontiguousarray(t.x).tobytes())
            if t.gamma is not None:
                h.update(np.ascontiguousarray(t.gamma).tobytes())
        return h.hexdigest()


def algorithmic_bytes(rows: int, cols: int, fused: bool, rowwise: bool,
                      columnwise: bool) -> int:
    """Bytes one pass must move at minimum: read x (2 B/elem) and gamma (2 B/col)
    once; write normed (2 B/elem, fused only), each enabled data plane (1 B/elem)
    and its scales (1 B per 32 elements)."""
    n = rows * cols
    b = 2 * n
    if fused:
        b += 2 * n + 2 * cols
    if rowwise:
        b += n + n // BLOCK
    if columnwise:
        b += n + n // BLOCK
    return b


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns through PyTorch's round-to-nearest-even cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _normal(rng, shape, scale=1.0, loc=0.0):
    a = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    if loc != 0.0:
        a += np.float32(loc)
    return a


def config(k: int) -> Workload:
    """The seeded workload ``k`` (1..5) at full size."""
    rng = np.random.default_rng(k - 1)
    if k == 1:
        x = _normal(rng, (256, 1024))
        g = _normal(rng, (1024,), 0.1, 1.0)
        return Workload("fused-rowwise-256x1024", True, True, False,
                        [Tensor2D(to_bf16_bits(x), to_bf16_bits(g), 1e-6, 0.0)])
    if k == 2:
        R, C = 8192, 4096
        x = _normal(rng, (R, C))
        n_out = int(round(0.001 * R * C))
        pos = rng.choice(R * C, size=n_out, replace=False)
        x.reshape(-1)[pos] *= np.float32(100.0)
        g = _normal(rng, (C,), 0.1)
        return Workload("fused-both-8192x4096", True, True, True,
                        [Tensor2D(to_bf16_bits(x), to_bf16_bits(g), 1e-5, 1.0)])
    if k == 3:
        shapes = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
        ts = [Tensor2D(to_bf16_bits(_normal(rng, s, 0.02))) for s in shapes]
        return Workload("quant-both-llama3-8b-layer", False, True, True, ts)
    if k == 4:
        return stress(32768, 8192, rng)
    if k == 5:
        rows = BLOCK * rng.integers(1, 129, size=128)
        cols = BLOCK * rng.integers(8, 225, size=128)
        ts = [Tensor2D(to_bf16_bits(_normal(rng, (int(r), int(c)), 0.02)))
              for r, c in zip(rows, cols)]
        return Workload("quant-both-grouped-128", False, True, True, ts)
    raise ValueError(f"no workload {k}")


def stress(R: int, C: int, rng=None, seed: int = 3) -> Workload:
    """Workload 4's recipe at any size (R, C multiples of 32)."""
    if rng is None:
        rng = np.random.default_rng(seed)
    x = _normal(rng, (R, C))
    k = rng.integers(-20, 21, size=R)
    x *= np.ldexp(np.float32(1.0), k.astype(np.int32)).astype(np.float32)[:, None]
    bits = to_bf16_bits(x)
    del x
    nblocks = R * C // BLOCK
    nsel = int(0.01 * nblocks)
    sel = rng.choice(nblocks, size=2 * nsel, replace=False)
    blk = bits.reshape(nblocks, BLOCK)
    blk[sel[:nsel]] = 0
    sub_frac = rng.integers(1, 128, size=(nsel, BLOCK)).astype(np.uint16)
    sub_sign = rng.integers(0, 2, size=(nsel, BLOCK)).astype(np.uint16) << 15
    blk[sel[nsel:]] = sub_sign | sub_frac
    g = _normal(rng, (C,), 0.1, 1.0)
    return Workload(f"fused-both-stress-{R}x{C}", True, True, True,
                    [Tensor2D(bits, to_bf16_bits(g), 1e-6, 0.0)])


def wide_range(R: int, C: int, seed: int) -> np.ndarray:
    """bf16 bits [R, C] (C a multiple of 32, any R): N(0, 1) rows scaled by
    2^k, k uniform in [-60, 60] per row, with 2 % of the 32-element blocks
    zero and 2 % sub-normal (random signs and fractions)."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (R, C))
    k = rng.integers(-60, 61, size=R)
    x *= np.ldexp(np.float32(1.0), k.astype(np.int32)).astype(np.float32)[:, None]
    bits = to_bf16_bits(x)
    nblocks = R * C // BLOCK
    nsel = max(1, int(0.02 * nblocks)) if nblocks >= 4 else 0
    if nsel:
        sel = rng.choice(nblocks, size=2 * nsel, replace=False)
        blk = bits.reshape(nblocks, BLOCK)
        blk[sel[:nsel]] = 0
        sub_frac = rng.integers(1, 128, size=(nsel, BLOCK)).astype(np.uint16)
        sub_sign = rng.integers(0, 2, size=(nsel, BLOCK)).astype(np.uint16) << 15
        blk[sel[nsel:]] = sub_sign | sub_frac
    return bits


def random_fused(R: int, C: int, seed: int, scale: float = 1.0, eps: float = 1e-6,
                 offset: float = 0.0, rowwise=True, columnwise=True) -> Workload:
    rng = np.random.default_rng(seed)
    x = _normal(rng, (R, C), scale)
    g = _normal(rng, (C,), 0.1, 1.0)
    return Workload(f"fused-{R}x{C}", True, rowwise, columnwise,
                    [Tensor2D(to_bf16_bits(x), to_bf16_bits(g), eps, offset)])


def random_bits_fused(R: int, C: int, seed: int, rows_per_draw: int = 4096) -> Workload:
    """Fused input for very large tensors, drawn directly as bf16 bit patterns
    (no float32 pass): uniform sign, biased exponent uniform in 113..140
    (magnitudes 2^-14 .. 2^14), uniform 7-bit fraction; gamma = 1 + 0.1 N(0, 1);
    eps 1e-6; offset 0. Drawn in blocks of rows to bound host memory."""
    rng = np.random.default_rng(seed)
    bits = np.empty((R, C), dtype=np.uint16)
    for r0 in range(0, R, rows_per_draw):
        r1 = min(R, r0 + rows_per_draw)
        u = rng.integers(0, 1 << 16, size=(r1 - r0, C), dtype=np.uint16)
        e = rng.integers(113, 141, size=(r1 - r0, C), dtype=np.uint16)
        bits[r0:r1] = (u & np.uint16(0x807F)) | (e << np.uint16(7))
    g = _normal(rng, (C,), 0.1, 1.0)
    return Workload(f"fused-bits-{R}x{C}", True, True, True,
                    [Tensor2D(bits, to_bf16_bits(g), 1e-6, 0.0)])


def random_weights(shapes, seed: int, scale: float = 0.02, rowwise=True,
                   columnwise=True) -> Workload:
    rng = np.random.default_rng(seed)
    ts = [Tensor2D(to_bf16_bits(_normal(rng, s, scale))) for s in shapes]
    return Workload("quant-list", False, rowwise, columnwise, ts)
