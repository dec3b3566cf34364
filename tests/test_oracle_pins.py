"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check ties one part of the oracle to the format definitions, a closed form,
a library routine (PyTorch's float8/bfloat16 casts and ``rms_norm``), brute
force, or a hand-worked block, so that a plausible slip anywhere in it (a
dropped term, a wrong sign or index, a transposed operand, ties rounded the
wrong way) fails at least one of them. None of these tests needs a GPU.
"""
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_blocks.txt")


def ulp_dist_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable steps between bf16 bit patterns (+0 == -0)."""
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(ordered(a) - ordered(b))


def torch_bf16_bits(v) -> np.ndarray:
    t = torch.as_tensor(np.asarray(v, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_e4m3_sat(v: np.ndarray) -> np.ndarray:
    """Library E4M3 encoding with saturation: PyTorch's cast is not saturating
    (it maps past-the-range values to NaN), so clamp to +-448 first."""
    t = torch.as_tensor(np.asarray(v, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
FINITE_BF16 = ALL_BF16[((ALL_BF16 >> 7) & 0xFF) != 0xFF]


# ---------------------------------------------------------------- bf16 ---

def test_bf16_decode_all_codes_match_torch():
    mine = oracle.bf16_value(ALL_BF16)
    ref = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_bf16_round_matches_torch_cast_near_every_boundary():
    # every float32 whose low half sits at or next to a rounding boundary,
    # for every high half, plus random floats
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    rng = np.random.default_rng(7)
    bits = np.concatenate([bits, rng.integers(0, 1 << 32, 400_000, dtype=np.uint64).astype(np.uint32)])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    mine = oracle.bf16_round(f.astype(np.float64))
    ref = torch_bf16_bits(f)
    assert np.array_equal(mine, ref)


def test_bf16_round_spot_values():
    assert oracle.bf16_round(np.array([1.0 + 2**-8]))[0] == 0x3F80      # tie -> even
    assert oracle.bf16_round(np.array([1.0 + 3 * 2**-8]))[0] == 0x3F82  # tie -> even (up)
    assert oracle.bf16_round(np.array([-0.0]))[0] == 0x8000
    assert oracle.bf16_round(np.array([2.0**-134]))[0] == 0x0000        # half of min subnormal
    assert oracle.bf16_round(np.array([3 * 2.0**-134]))[0] == 0x0002    # 1.5 ulp -> even (2)
    assert oracle.bf16_round(np.array([2.0**128]))[0] == 0x7F80


# ---------------------------------------------------------------- E4M3 ---

def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0**-9 and mine[0x08] == 2.0**-6


def _reachable_block_values():
    """Every finite bf16 b against every block exponent e it can meet:
    |b| < 2^(e+9) (b can sit in a block whose amax has floor(log2) = e + 8), or
    e = -127 with |b| < 2^-118 (the clamped exponent). Returns (b, e)."""
    mag = oracle.bf16_value(FINITE_BF16)
    bs, es = [], []
    for e in range(-127, 120):
        lim = 2.0**-118 if e == -127 else 2.0 ** (e + 9)
        sel = np.abs(mag) < lim
        bs.append(FINITE_BF16[sel])
        es.append(np.full(int(sel.sum()), e, np.int32))
    return np.concatenate(bs), np.concatenate(es)


@pytest.fixture(scope="module")
def reachable():
    return _reachable_block_values()


def test_e4m3_encoders_exhaustive_on_all_reachable_values(reachable):
    b, e = reachable
    v = oracle.bf16_value(b) * np.ldexp(1.0, -e)
    assert v.size > 8_000_000
    near = oracle.e4m3_nearest(v)
    scan = oracle.e4m3_scan(v)
    assert np.array_equal(near, scan)
    # v has at most 8 significant bits and |v| < 512, so float32 holds it
    # exactly whenever |v| >= 2^-126; below that both sides give signed zero
    ref = torch_e4m3_sat(v.astype(np.float32))
    assert np.array_equal(near, ref)


def test_e4m3_spot_values():
    vals = np.array([460.0, 2.0**-10, 1.5 * 2.0**-10, -1e-9, -0.0, 448.0, 464.0, 1e30, 2.0**-9])
    want = np.array([0x7E, 0x00, 0x01, 0x80, 0x80, 0x7E, 0x7E, 0x7E, 0x01], np.uint8)
    assert np.array_equal(oracle.e4m3_nearest(vals), want)
    assert np.array_equal(oracle.e4m3_scan(vals), want)


# ---------------------------------------------------------------- E8M0 ---

def test_e8m0_scale_all_bf16_amax_closed_form():
    pos = FINITE_BF16[FINITE_BF16 < 0x8000]              # +0 .. largest finite
    amax = oracle.bf16_value(pos)
    byte = oracle.e8m0_byte(amax)
    field = (pos.astype(np.int32) >> 7) & 0xFF
    # closed form of clamp(floor(log2 amax) - 8, -127, 127) + 127 for bf16 amax
    assert np.array_equal(byte, np.maximum(field - 8, 0).astype(np.uint8))
    # library decode of the byte: 2^(byte-127); unclamped blocks land in [256, 512)
    scale = torch.from_numpy(byte.copy()).view(torch.float8_e8m0fnu).double().numpy()
    assert np.array_equal(scale, np.ldexp(1.0, byte.astype(np.int32) - 127))
    un = byte > 0
    r = amax[un] / scale[un]
    assert np.all((r >= 256) & (r < 512))
    # clamped: amax below 2^-118 (including every sub-normal) -> byte 0
    assert np.all(amax[~un] < 2.0**-118)


def test_e8m0_special_cases():
    m = np.arange(-119, 128)
    assert np.array_equal(oracle.e8m0_byte(np.ldexp(1.0, m)), (m + 119).astype(np.uint8))
    assert oracle.e8m0_byte(np.array([1.0]))[0] == 119
    assert oracle.e8m0_byte(np.array([0.0]))[0] == 0
    assert oracle.e8m0_value(np.array([0, 127, 255]))[:2].tolist() == [2.0**-127, 1.0]
    assert math.isnan(oracle.e8m0_value(np.array([255]))[0])


# ------------------------------------------------------- block quantize ---

def _expected_blocks(b, e):
    """Blocks of 32: one carrier (the largest bf16 below 2^(e+9), or below
    2^-118 for the clamped exponent) plus 31 reachable values of that exponent."""
    rows, want_q, want_s = [], [], []
    for ee in np.unique(e):
        vals = b[e == ee]
        lim_exp = -118 if ee == -127 else ee + 9
        # bf16 code of 2^lim_exp is (lim_exp + 127) << 7; one code below it is
        # the largest bf16 under 2^lim_exp
        carrier = np.uint16(((int(lim_exp) + 127) << 7) - 1)
        assert oracle.bf16_value(np.array([carrier]))[0] < 2.0**lim_exp
        n = -(-vals.size // 31) * 31
        padded = np.concatenate([vals, np.zeros(n - vals.size, np.uint16)]).reshape(-1, 31)
        blk = np.concatenate([np.full((padded.shape[0], 1), carrier, np.uint16), padded], axis=1)
        rows.append(blk)
        v = oracle.bf16_value(blk) * 2.0 ** (-ee)
        want_q.append(torch_e4m3_sat(v.astype(np.float32)))
        want_s.append(np.full(blk.shape[0], ee + 127, np.uint8))
    return np.concatenate(rows), np.concatenate(want_q), np.concatenate(want_s)


def test_block_quantize_exhaustive_rowwise_and_columnwise(reachable):
    b, e = reachable
    blocks, want_q, want_s = _expected_blocks(b, e)
    nb = blocks.shape[0] - blocks.shape[0] % 32            # whole 32-row groups
    blocks, want_q, want_s = blocks[:nb], want_q[:nb], want_s[:nb]
    q_row, s_row, _, _ = oracle.quant_mxfp8(blocks, True, False)
    assert np.array_equal(s_row[:, 0], want_s)
    assert np.array_equal(q_row, want_q)
    # the same blocks laid down columns of a [32, nb] matrix
    t = np.ascontiguousarray(blocks.T)
    _, _, q_col, s_col = oracle.quant_mxfp8(t, False, True)
    assert np.array_equal(s_col[0], want_s)
    assert np.array_equal(q_col, np.ascontiguousarray(want_q.T))


def _golden_blocks():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, sbyte, pairs = [p.strip() for p in line.split("|")]
        vals, codes = [], []
        for p in pairs.split():
            v, c = p.split(":")
            vals.append(float(v))
            codes.append(int(c, 16))
        out.append((name, int(sbyte), vals, codes))
    return out


@pytest.mark.parametrize("blk", _golden_blocks(), ids=lambda b: b[0])
def test_golden_hand_worked_blocks(blk):
    name, sbyte, vals, codes = blk
    bits = oracle.bf16_round(np.array(vals))
    assert np.array_equal(oracle.bf16_value(bits), np.array(vals)), "fixture values must be bf16"
    row = np.zeros((32, 32), np.uint16)                 # 32 rows so columnwise applies
    row[0, :len(vals)] = bits
    row[:, :] = row[0]                                  # every row the same block
    q_row, s_row, q_col, s_col = oracle.quant_mxfp8(row)
    want = np.zeros(32, np.uint8)
    want[:len(codes)] = codes
    assert s_row[0, 0] == sbyte
    assert np.array_equal(q_row[0], want)
    # column c holds 32 copies of element c: its scale follows |element c|
    colmax = np.abs(oracle.bf16_value(bits))
    assert np.array_equal(s_col[0, :len(vals)], oracle.e8m0_byte(colmax))


def test_structured_layout_closed_form():
    """x[r, c] = s(r, c) * 2^p(r, c) with integer exponents: every scale and
    code follows from integer arithmetic on p, for both planes, so a swapped
    index, a transposed plane or a mis-laid scale array fails here."""
    R, C = 64, 96
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    p = (r * 7 + c * 3) % 23 - 11
    sign = ((r + 2 * c) % 5 == 0)
    x = np.where(sign, -1.0, 1.0) * np.ldexp(1.0, p)
    bits = oracle.bf16_round(x)
    q_row, s_row, q_col, s_col = oracle.quant_mxfp8(bits)

    def code(t, neg):  # E4M3 code of 2^t with t <= 8
        m = np.where(t >= -6, (t + 7) << 3, np.where(t >= -9, 1 << np.clip(t + 9, 0, 3), 0))
        return (m | np.where(neg, 0x80, 0)).astype(np.uint8)

    P_row = p.reshape(R, C // 32, 32).max(axis=2)
    assert np.array_equal(s_row, (P_row - 8 + 127).astype(np.uint8))
    t_row = p - np.repeat(P_row, 32, axis=1) + 8
    assert np.array_equal(q_row, code(t_row, sign))
    P_col = p.reshape(R // 32, 32, C).max(axis=1)
    assert np.array_equal(s_col, (P_col - 8 + 127).astype(np.uint8))
    t_col = p - np.repeat(P_col, 32, axis=0) + 8
    assert np.array_equal(q_col, code(t_col, sign))


# ------------------------------------------------------------- RMSNorm ---

def _bits(v):
    return oracle.bf16_round(np.asarray(v, np.float64))


def _exact_rms_value(c: float, eps: float) -> float:
    getcontext().prec = 60
    d = Decimal(c)
    return float(d / (d * d + Decimal(eps)).sqrt())


@pytest.mark.parametrize("j", [-30, -12, -8, -3, 0, 5, 40])
@pytest.mark.parametrize("C", [32, 1024, 96])
def test_rmsnorm_constant_rows_closed_form(j, C):
    # constant row c (gamma 1, offset 0): y = c / sqrt(c^2 + eps), whatever C is
    eps = float(np.float32(1e-6))
    cval = 2.0**j
    x = _bits(np.full((2, C), cval))
    x[1] = _bits(np.full(C, -cval))
    g = _bits(np.ones(C))
    y = oracle.rmsnorm_f32(x, g, eps, 0.0)
    exact = _exact_rms_value(cval, eps)
    want = torch_bf16_bits(np.float32(exact))
    assert ulp_dist_bf16(y[0], np.full(C, want)).max() <= 1
    assert ulp_dist_bf16(y[1], np.full(C, want | 0x8000)).max() <= 1


def test_rmsnorm_unit_rows_exact():
    C = 1024
    x = _bits(np.where(np.arange(C) % 3 == 0, -1.0, 1.0)[None, :].repeat(4, 0))
    y = oracle.rmsnorm_f32(x, _bits(np.ones(C)), float(np.float32(1e-6)), 0.0)
    assert np.array_equal(y, x)


def test_rmsnorm_gamma_and_offset_per_column():
    # x = +-2^k per row and eps 0: inv is exact, so y = sign * bf16(gamma + offset)
    rng = np.random.default_rng(1)
    C = 256
    g = _bits(rng.standard_normal(C) * 0.3)
    off = 0.75
    ks = np.array([-9, 0, 3, 7])
    sg = np.array([1.0, -1.0, 1.0, -1.0])
    x = _bits((sg * np.ldexp(1.0, ks))[:, None].repeat(C, 1))
    y = oracle.rmsnorm_f32(x, g, 0.0, off)
    w32 = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).float() + torch.tensor(off, dtype=torch.float32)
    want = w32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for i in range(4):
        exp = want if sg[i] > 0 else want ^ 0x8000
        assert np.array_equal(y[i], exp), i


def test_rmsnorm_scale_invariance_eps0():
    rng = np.random.default_rng(2)
    x = _bits(rng.standard_normal((8, 512)))
    g = _bits(1 + 0.1 * rng.standard_normal(512))
    base = oracle.rmsnorm_f32(x, g, 0.0, 0.0)
    for k in (-40, -7, 9, 50):
        xs = _bits(oracle.bf16_value(x) * 2.0**k)
        assert np.array_equal(oracle.rmsnorm_f32(xs, g, 0.0, 0.0), base)


@pytest.mark.parametrize("eps,offset,scale", [(1e-6, 0.0, 1.0), (1e-5, 1.0, 3.0), (1e-6, 0.5, 1e-3)])
def test_rmsnorm_matches_torch_rms_norm_float64(eps, offset, scale):
    rng = np.random.default_rng(3)
    R, C = 16, 768
    x = _bits(rng.standard_normal((R, C)) * scale)
    g = _bits(0.1 * rng.standard_normal(C) + (0.0 if offset else 1.0))
    eps32 = float(np.float32(eps))
    xt = torch.from_numpy(oracle.bf16_value(x))
    w = torch.from_numpy(oracle.bf16_value(g)) + offset
    ref = torch.nn.functional.rms_norm(xt, (C,), weight=w, eps=eps32).numpy()
    y64 = oracle.rmsnorm_f64(x, g, eps32, offset)
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-300)
    y32 = oracle.rmsnorm_f32(x, g, eps32, offset)
    assert ulp_dist_bf16(y32, oracle.bf16_round(ref)).max() <= 1


def test_rmsnorm_zero_row_is_zero_and_signed():
    C = 64
    x = np.zeros((2, C), np.uint16)
    g = _bits(np.where(np.arange(C) % 2 == 0, 1.0, -1.0))
    y = oracle.rmsnorm_f32(x, g, float(np.float32(1e-6)), 0.0)
    assert np.array_equal(y[0], np.where(np.arange(C) % 2 == 0, 0, 0x8000).astype(np.uint16))


# ------------------------------------------------- invariants on workloads ---

def dequant_error_ok(vals, q, s_bytes_per_elem):
    """Bound for round-to-nearest E4M3 after the power-of-two scaling (|v| < 512):
    normal codes: |err| <= 2^-4 |x|; sub-normal region (|v| < 2^-6): |err| <=
    2^(e-10); saturated (|v| > 448): |err| < 64 * 2^e."""
    e = s_bytes_per_elem.astype(np.int32) - 127
    deq = oracle.e4m3_value(q) if q.size < 5000 else _e4m3_table()[q]
    deq = deq * np.ldexp(1.0, e)
    err = np.abs(deq - vals)
    v = np.abs(vals) * np.ldexp(1.0, -e)
    bound = np.where(v > 448, 64.0 * np.ldexp(1.0, e),
                     np.where(v >= 2.0**-6, 2.0**-4 * np.abs(vals), np.ldexp(1.0, e - 10)))
    return bool(np.all(err <= bound))


_TABLE = None


def _e4m3_table():
    global _TABLE
    if _TABLE is None:
        _TABLE = oracle.e4m3_value(np.arange(256, dtype=np.uint8))
    return _TABLE


def check_invariants(v_bits, q_row, s_row, q_col, s_col):
    vals = oracle.bf16_value(v_bits)
    R, C = v_bits.shape
    if q_row is not None:
        srow = np.repeat(s_row, 32, axis=1)
        assert dequant_error_ok(vals, q_row, srow)
        # the block's largest element lands in the top binade (codes 0x78..0x7E)
        blk = np.abs(vals).reshape(R, C // 32, 32)
        arg = blk.argmax(axis=2)
        qa = np.take_along_axis(q_row.reshape(R, C // 32, 32), arg[..., None], 2)[..., 0] & 0x7F
        live = s_row > 0
        assert np.all((qa[live] >= 0x78) & (qa[live] <= 0x7E))
    if q_col is not None:
        scol = np.repeat(s_col, 32, axis=0)
        assert dequant_error_ok(vals, q_col, scol)
        blk = np.abs(vals).reshape(R // 32, 32, C)
        arg = blk.argmax(axis=1)
        qa = np.take_along_axis(q_col.reshape(R // 32, 32, C), arg[:, None, :], 1)[:, 0, :] & 0x7F
        live = s_col > 0
        assert np.all((qa[live] >= 0x78) & (qa[live] <= 0x7E))
    if q_row is not None and q_col is not None:
        same = np.repeat(s_row, 32, axis=1) == np.repeat(s_col, 32, axis=0)
        assert np.array_equal(q_row[same], q_col[same])


def test_invariants_workload_shapes_small():
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
    cases = [W.config(1), W.stress(256, 1024, seed=11),
             W.random_fused(96, 320, seed=5, scale=100.0, eps=1e-5, offset=1.0)]
    for wl in cases:
        t = wl.tensors[0]
        R = t.x.shape[0] - t.x.shape[0] % 32
        normed, q_row, s_row, q_col, s_col = oracle.rmsnorm_quant_mxfp8(
            t.x[:R], t.gamma, t.eps, t.offset, True, True)
        check_invariants(normed, q_row, s_row, q_col, s_col)
        # float32 statement stays within one bf16 step of the float64 one
        y64 = oracle.rmsnorm_f64(t.x[:R], t.gamma, t.eps, t.offset)
        assert ulp_dist_bf16(normed, oracle.bf16_round(y64)).max() <= 1
    w = W.random_weights([(64, 256), (32, 1024)], seed=4)
    for t in w.tensors:
        check_invariants(t.x, *oracle.quant_mxfp8(t.x))


def test_threaded_oracle_equals_single_thread():
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
    t = W.stress(320, 512, seed=9).tensors[0]
    a = oracle.rmsnorm_quant_mxfp8(t.x, t.gamma, t.eps, t.offset, threads=1)
    b = oracle.rmsnorm_quant_mxfp8(t.x, t.gamma, t.eps, t.offset, threads=4)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ------------------------------------------------ tiled GEMM scale layout ---

def test_mma_scale_layout_hand_worked_offsets():
    # tiles of 128 rows x 4 scale columns, 512 bytes each, row tiles outer;
    # inside: (m % 32) * 16 + ((m // 32) % 4) * 4 + k % 4
    cases = [((0, 0, 4), 0), ((1, 0, 4), 16), ((31, 3, 4), 31 * 16 + 3), ((32, 0, 4), 4),
             ((127, 3, 4), 31 * 16 + 12 + 3), ((128, 0, 4), 512), ((0, 4, 8), 512),
             ((130, 5, 8), (1 * 2 + 1) * 512 + 2 * 16 + 1), ((0, 0, 5), 0), ((128, 0, 5), 1024)]
    for (m, k, Kb), want in cases:
        assert oracle.mma_scale_offset(m, k, Kb) == want, (m, k, Kb)


@pytest.mark.parametrize("M,Kb", [(128, 4), (256, 8), (96, 3), (1, 1), (300, 7)])
def test_mma_scale_layout_is_a_bijection_onto_the_unpadded_positions(M, Kb):
    s = (np.arange(M * Kb) % 251 + 1).astype(np.uint8).reshape(M, Kb)
    out = oracle.scales_to_mma(s, fill=0)
    rows, cols = oracle.mma_scale_shape(M, Kb)
    assert out.size == rows * cols
    offs = np.array([[oracle.mma_scale_offset(m, k, Kb) for k in range(Kb)] for m in range(M)])
    assert len(np.unique(offs)) == M * Kb and offs.max() < out.size
    assert np.array_equal(out[offs], s)
    pad = np.ones(out.size, bool)
    pad[offs.ravel()] = False
    assert np.all(out[pad] == 0)
    # every 128 x 4 tile is one contiguous 512-byte run; inside it, 16-byte
    # line b holds rows b, b+32, b+64, b+96 (4 scales each)
    if M % 128 == 0 and Kb % 4 == 0:
        t = out.reshape(-1, 32, 4, 4)             # [tile, line b, row group a, k]
        for tm in range(M // 128):
            for tk in range(Kb // 4):
                tile = t[tm * (Kb // 4) + tk]
                for b in range(32):
                    for a in range(4):
                        assert np.array_equal(tile[b, a], s[tm * 128 + a * 32 + b, tk * 4:tk * 4 + 4])


def test_mma_scale_layout_columnwise_reads_transposed():
    Kb, M = 3, 160                                # compact columnwise scales [R/32, C]
    s = (np.arange(Kb * M) % 253).astype(np.uint8).reshape(Kb, M)
    out = oracle.scales_to_mma(s, columnwise=True)
    for m in (0, 31, 32, 127, 128, 159):
        for k in range(Kb):
            assert out[oracle.mma_scale_offset(m, k, Kb)] == s[k, m]


# ------------------------------------------------------------ residual add ---

def test_residual_add_matches_torch_float32_sum_cast():
    # random finite pairs over the whole bf16 range, pairs far apart in
    # exponent, cancelling pairs and pairs whose sum lands on a bf16 midpoint
    rng = np.random.default_rng(11)
    x = FINITE_BF16[rng.integers(0, FINITE_BF16.size, 3_000_000)]
    r = FINITE_BF16[rng.integers(0, FINITE_BF16.size, 3_000_000)]
    one = np.uint16(0x3F80)
    ties = oracle.bf16_round(np.ldexp(1.0, -np.arange(8, 20)))      # 1 + 2^-k
    x = np.concatenate([x, np.full(ties.size, one), x[:1000], x[:1000] ^ 0x8000])
    r = np.concatenate([r, ties, x[:1000] ^ 0x8000, x[:1000] ^ 0x8000])
    h = oracle.residual_add(x, r)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    rt = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).float()
    s = (xt + rt)
    ok = torch.isfinite(s).numpy()
    want = s.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert ok.mean() > 0.99
    assert np.array_equal(h[ok], want[ok])


def test_residual_add_closed_forms():
    a = oracle.bf16_round(np.array([1.0, 1.0, 3.0, -2.0, 0.0, -0.0]))
    b = oracle.bf16_round(np.array([2.0**-8, 3 * 2.0**-8, -3.0, 2.0, -0.0, -0.0]))
    h = oracle.bf16_value(oracle.residual_add(a, b))
    # 1 + 2^-8 ties to 1; 1 + 3*2^-8 ties up to 1 + 2^-6; x + (-x) = +0; -0 + -0 = -0
    assert h[0] == 1.0 and h[1] == 1.0 + 2.0**-6 and h[2] == 0.0 and not np.signbit(h[2])
    assert h[3] == 0.0 and h[4] == 0.0 and not np.signbit(h[4]) and np.signbit(h[5])


# ------------------------------------------- padded scales, plane update ---

def test_padded_scale_shapes_and_placement():
    # TE's allocation shapes: rowwise [roundup(R,128), roundup(C/32,4)],
    # columnwise [roundup(R/32,4), roundup(C,128)]
    assert oracle.padded_scale_shape(45, 160, False) == (128, 8)
    assert oracle.padded_scale_shape(96, 160, True) == (4, 256)
    assert oracle.padded_scale_shape(256, 8192, False) == (256, 256)
    s = (np.arange(45 * 5) % 200 + 1).astype(np.uint8).reshape(45, 5)
    p = oracle.scales_to_padded(s, 45, 160, False, fill=7)
    assert p.shape == (128, 8) and np.array_equal(p[:45, :5], s)
    assert np.all(p[45:] == 7) and np.all(p[:, 5:] == 7)
    sc = (np.arange(3 * 160) % 200 + 1).astype(np.uint8).reshape(3, 160)
    pc = oracle.scales_to_padded(sc, 96, 160, True)
    assert pc.shape == (4, 256) and np.array_equal(pc[:3, :160], sc) and np.all(pc[3:] == 0)


def test_update_planes_semantics_hand_worked():
    R, C = 32, 64
    rng = np.random.default_rng(5)
    src = {"rows": R, "cols": C,
           "q_row": rng.integers(0, 256, (R, C), dtype=np.uint8),
           "s_row": rng.integers(1, 200, (R, C // 32), dtype=np.uint8),
           "q_col": None, "s_col": None}                  # columnwise plane absent
    dst = {"q_row": np.full(R * C, 9, np.uint8), "s_row": np.full(128 * 4, 9, np.uint8),
           "q_col": np.full(R * C, 9, np.uint8), "s_col": np.full(4 * 128, 9, np.uint8)}
    # only rowwise selected: rowwise installed (padding kept), columnwise kept
    out = oracle.update_planes(src, dst, True, False, "padded")
    assert np.array_equal(out["q_row"], src["q_row"].ravel())
    srow = out["s_row"].reshape(128, 4)
    assert np.array_equal(srow[:R, :2], src["s_row"]) and np.all(srow[R:] == 9) and np.all(srow[:, 2:] == 9)
    assert np.all(out["q_col"] == 9) and np.all(out["s_col"] == 9)
    # columnwise selected but absent from src: cleared, padding included
    out = oracle.update_planes(src, dst, False, True, "padded")
    assert np.all(out["q_col"] == 0) and np.all(out["s_col"] == 0)
    assert np.all(out["q_row"] == 9)
    # src untouched
    assert src["q_col"] is None and dst["q_row"][0] == 9


def test_dequantize_matches_library_decode_and_mm_closed_form():
    rng = np.random.default_rng(6)
    q = rng.integers(0, 256, (4, 64), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x10                         # no NaN codes
    s = rng.integers(100, 140, (4, 2), dtype=np.uint8)
    got = oracle.dequantize_rowwise(q, s)
    v = torch.from_numpy(q).view(torch.float8_e4m3fn).double()
    sc = torch.from_numpy(s).view(torch.float8_e8m0fnu).double().repeat_interleave(32, dim=1)
    assert np.array_equal(got, (v * sc).numpy())
    # powers of two quantize exactly: x = 2^a[m] (all K), w = 2^b[n] -> x w^T = K 2^(a+b)
    K = 64
    a = np.array([-3, 0, 5]); b = np.array([1, -2])
    x = oracle.bf16_round(np.repeat(np.ldexp(1.0, a)[:, None], K, 1))
    w = oracle.bf16_round(np.repeat(np.ldexp(1.0, b)[:, None], K, 1))
    assert np.array_equal(oracle.mm_mxfp8(x, w, threads=1), K * np.ldexp(1.0, a[:, None] + b[None, :]))


def test_mm_closed_form_with_a_scale_per_block():
    """Each 32-element block of x and w holds one power of two, different from
    block to block, so every block quantizes exactly (code 1.0 times its own
    scale) and x w^T = sum over blocks of 32 * 2^(a[m, k] + b[n, k]): a block
    paired with the wrong scale or the wrong partner block changes the sum."""
    rng = np.random.default_rng(8)
    M, N, nk = 3, 4, 5
    a = rng.integers(-20, 20, (M, nk))
    b = rng.integers(-20, 20, (N, nk))
    x = oracle.bf16_round(np.repeat(np.ldexp(1.0, a), 32, axis=1))
    w = oracle.bf16_round(np.repeat(np.ldexp(1.0, b), 32, axis=1))
    want = 32.0 * np.ldexp(1.0, a[:, None, :] + b[None, :, :]).sum(axis=2)
    assert np.array_equal(oracle.mm_mxfp8(x, w, threads=1), want)
