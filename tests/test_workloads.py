"""The seeded input generators: deterministic, and shaped as their recipes say."""
import numpy as np

from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W


def test_same_seed_same_bytes():
    a = W.random_fused(64, 256, seed=3)
    b = W.random_fused(64, 256, seed=3)
    c = W.random_fused(64, 256, seed=4)
    assert a.sha256() == b.sha256() != c.sha256()


def test_config1_shape_and_flags():
    wl = W.config(1)
    t = wl.tensors[0]
    assert t.x.shape == (256, 1024) and t.gamma.shape == (1024,)
    assert wl.fused and wl.rowwise and not wl.columnwise
    assert (t.eps, t.offset) == (1e-6, 0.0)
    assert wl.algorithmic_bytes() == 1_320_960
    assert W.config(1).sha256() == wl.sha256()


def test_stress_recipe_zero_and_subnormal_blocks():
    R, C = 512, 1024
    t = W.stress(R, C, seed=3).tensors[0]
    blk = t.x.reshape(-1, 32)
    nsel = int(0.01 * blk.shape[0])
    zero = np.all(blk == 0, axis=1)
    expo = (blk >> 7) & 0xFF
    sub = np.all((expo == 0) & ((blk & 0x7F) != 0), axis=1)
    assert zero.sum() == nsel and sub.sum() == nsel
    assert not np.any(zero & sub)
    # rows scaled by 2^k, k in [-20, 20]: row maxima span many binades
    live = ~(zero | sub)
    ex = expo.reshape(R, -1)
    assert ex.max() - ex[ex > 0].min() > 30


def test_algorithmic_bytes_formula():
    assert W.algorithmic_bytes(32768, 8192, True, True, True) == 1_627_406_336
    assert W.algorithmic_bytes(8192, 4096, True, True, True) == 203_431_936
    assert W.algorithmic_bytes(32, 256, False, True, True) == int(4.0625 * 32 * 256)


def test_random_bits_recipe():
    a = W.random_bits_fused(96, 256, seed=5, rows_per_draw=40).tensors[0]
    b = W.random_bits_fused(96, 256, seed=5, rows_per_draw=40).tensors[0]
    assert np.array_equal(a.x, b.x) and np.array_equal(a.gamma, b.gamma)
    expo = (a.x >> 7) & 0xFF
    assert expo.min() == 113 and expo.max() == 140
    sign = a.x >> 15
    assert 0.4 < sign.mean() < 0.6
    assert len(np.unique(a.x & 0x7F)) == 128


def test_wide_range_recipe():
    """Any row count; 2 % zero and 2 % sub-normal 32-element blocks, disjoint;
    rows 2^k-scaled with k in [-60, 60], so block exponents span far more than
    E4M3's range; the same seed gives the same bytes."""
    R, C = 37, 4096
    a = W.wide_range(R, C, seed=5)
    assert a.shape == (R, C) and a.dtype == np.uint16
    assert np.array_equal(a, W.wide_range(R, C, seed=5))
    assert not np.array_equal(a, W.wide_range(R, C, seed=6))
    blk = a.reshape(-1, 32)
    nsel = max(1, int(0.02 * blk.shape[0]))
    zero = np.all(blk == 0, axis=1)
    expo = (blk >> 7) & 0xFF
    sub = np.all((expo == 0) & ((blk & 0x7F) != 0), axis=1)
    assert zero.sum() == nsel and sub.sum() == nsel and not np.any(zero & sub)
    row_max = expo.reshape(R, -1).max(axis=1)
    assert row_max.max() - row_max.min() > 60
    assert W.wide_range(1, 32, seed=1).shape == (1, 32)
