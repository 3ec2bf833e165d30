"""Pins of the oracle's MXFP4 weights and their conversion to FP8 tiles (CPU only): the E2M1
grid in closed form, round-to-nearest-even on the grid (brute force and every tie written out
by hand), minimality of the sub-block exponent, the FP8 headroom (q * 2^t is an E4M3 value for
all q exactly when -8 <= t <= 6), the quantisation error bound, the headroom raise inside a
tile, and losslessness of the FP4 -> FP8 conversion."""
import numpy as np
import pytest

from oracle import fp8_weights as F8
from oracle import mxfp4_weights as M
from oracle import round_to_bf16


def test_e2m1_grid_closed_form():
    vals = M.e2m1_value(np.arange(16))
    assert list(vals[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(vals[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_rounding_ties_written_out():
    # every midpoint of the grid, with the neighbour whose mantissa bit is 0 (codes 0, 2, 4, 6)
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        for sgn in (1.0, -1.0):
            got = M.e2m1_value(M.round_to_e2m1_code(np.array([sgn * v])))[0]
            assert got == sgn * want or (want == 0.0 and got == 0.0), (v, sgn, got)
    assert M.round_to_e2m1_code(np.array([-0.0, -0.1]))[0] == 0        # zero stored as +0
    assert M.round_to_e2m1_code(np.array([-0.1]))[0] == 0


def test_rounding_brute_force():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-6, 6, 20000), M.GRID, -M.GRID])
    got = M.e2m1_value(M.round_to_e2m1_code(v))
    d = np.abs(np.concatenate([M.GRID, -M.GRID])[None, :] - v[:, None])
    assert (np.abs(got - v) == d.min(axis=1)).all()                     # always a nearest value


def test_block_exponent_is_the_smallest_that_fits():
    rng = np.random.default_rng(1)
    amax = np.concatenate([np.ldexp(rng.uniform(0.5, 1, 5000), rng.integers(-40, 40, 5000)),
                           6.0 * np.ldexp(1.0, np.arange(-30, 30)),
                           6.0 * np.ldexp(1.0, np.arange(-30, 30)) * (1 + 2.0 ** -40)])
    s = M.block_fit_exponent(amax)
    assert (amax <= 6.0 * np.ldexp(1.0, s)).all()
    assert (amax > 6.0 * np.ldexp(1.0, s - 1)).all()


def test_fp8_headroom_is_fourteen_binades():
    """q * 2^t is an E4M3 value for every E2M1 magnitude q iff -8 <= t <= 6."""
    for t in range(-12, 10):
        v = M.GRID[1:] * 2.0 ** t
        exact = bool((v <= 448).all()) and bool((F8.round_to_e4m3(np.minimum(v, 448)) == v).all())
        assert exact == (-8 <= t <= 6), t


def test_quantisation_error_bound_and_bf16_exactness():
    rng = np.random.default_rng(2)
    w = round_to_bf16(rng.normal(0, 0.02, (2, 256, 384)) * np.exp(rng.normal(0, 1, (2, 256, 1))))
    codes, exps = M.quantize_mxfp4(w)
    deq = M.dequantize_mxfp4(codes, exps)
    scale = np.ldexp(1.0, np.repeat(exps, 32, axis=-1))
    v = np.abs(w) / scale
    err = np.abs(deq - w) / scale
    # spacing 0.5 below 2, 1 in [2, 4), 2 in [4, 6]: at most half of it
    assert (err <= np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))).all()
    assert np.array_equal(round_to_bf16(deq), deq)
    assert (np.abs(deq) <= 6 * scale).all()


def test_headroom_raise_inside_a_tile():
    """A tile whose sub-block maxima span more than 14 binades: the small blocks' exponents are
    raised to the tile's largest minus 14; blocks in another tile are unaffected."""
    w = np.full((128, 256), 2.0 ** -30)
    w[0, :32] = 6.0                       # block exponent 0 in tile (0, 0)
    w[5, 32:64] = 6.0 * 2.0 ** -20        # would be -20: raised to -14
    codes, exps = M.quantize_mxfp4(w)
    assert exps[0, 0] == 0 and exps[5, 1] == -14
    assert (exps[:, :4] >= -14).all() and exps[:, :4].min() == -14
    assert (exps[:, 4:] == M.block_fit_exponent(np.array(2.0 ** -30))).all()   # tile (0, 1)
    assert exps[5, 1] == max(int(M.block_fit_exponent(np.array(6.0 * 2 ** -20))), -14)


def test_conversion_to_fp8_is_lossless():
    rng = np.random.default_rng(3)
    w = rng.normal(0, 1, (3, 200, 320)) * np.ldexp(1.0, rng.integers(-20, 6, (3, 200, 10)).repeat(32, -1))
    w[1, 128:, :128] = 0.0                # an all-zero FP8 tile
    w[2, 7, 64:96] = 0.0                  # an all-zero sub-block in a non-zero tile
    codes, exps = M.quantize_mxfp4(w)
    c8, e8 = M.mxfp4_to_fp8(codes, exps)
    assert c8.shape == codes.shape and e8.shape == (3, 2, 3)
    assert e8[1, 1, 0] == M.MIN_EXP - 6 and (exps[1, 128:, :4] == M.MIN_EXP).all()
    assert exps[2, 7, 2] == exps[2, :128, :4].max()      # zero sub-block: the tile's largest
    assert e8.min() >= -126 and exps.min() >= -128
    assert np.array_equal(F8.dequantize_fp8_tiles(c8, e8), M.dequantize_mxfp4(codes, exps))
    # the FP8 tile exponent is the tile's largest sub-block exponent minus 6
    assert e8[0, 0, 0] == exps[0, :128, :4].max() - 6


def test_conversion_rejects_exponents_beyond_the_headroom():
    codes = np.full((128, 128), 3, dtype=np.uint8)      # all 1.5
    exps = np.zeros((128, 4), dtype=np.int64)
    exps[3, 2] = -15       # 15 binades below the tile's largest: 1.5 * 2^-9 is no E4M3 value
    with pytest.raises(ValueError):
        M.mxfp4_to_fp8(codes, exps)


def test_rounding_matches_ml_dtypes_float4():
    """One rounding to E2M1 agrees with ml_dtypes' float4_e2m1fn conversion (round to nearest,
    ties to even) over the range, on the grid, on every midpoint and on its fp32 neighbours."""
    ml_dtypes = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(5)
    grid = np.concatenate([M.GRID, -M.GRID])
    mids = np.sort(M.GRID)
    mids = ((mids[1:] + mids[:-1]) / 2).astype(np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    v = np.concatenate([rng.uniform(-6, 6, 50000), grid, mids, -mids, near, -near]).astype(np.float32)
    ours = M.e2m1_value(M.round_to_e2m1_code(v.astype(np.float64)))
    ref = v.astype(ml_dtypes.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(np.abs(ours), np.abs(ref))
    assert np.array_equal(np.sign(ours), np.sign(ref) * (ref != 0))    # zero is stored as +0 here
