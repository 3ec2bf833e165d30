"""Pins of the oracle's FP8 weight quantisation (CPU only): E4M3 rounding against torch's own
float8_e4m3fn conversion, the closed-form E4M3 grid, minimality of the tile exponent, the
rounding error bound, exactness of the dequantised values in bf16, per-tile exponents on
partial tiles (brute force), and zero tiles."""
import numpy as np
import pytest
import torch

from oracle import fp8_weights as F
from oracle import round_to_bf16


def test_round_to_e4m3_matches_torch_conversion():
    """On fp32 inputs (what is rounded here: a bf16 weight times a power of two is exact in
    fp32), one rounding to E4M3 must agree with torch's float8_e4m3fn conversion of the fp32
    value -- over the whole range, on the grid, on every midpoint (ties to even) and on the fp32
    neighbours of every midpoint."""
    rng = np.random.default_rng(0)
    grid = F.e4m3_value(np.arange(0, 127, dtype=np.uint8))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
    v = np.concatenate([rng.uniform(-448, 448, 100000), np.ldexp(rng.uniform(-1, 1, 100000), rng.integers(-12, 9, 100000)),
                        grid, -grid, mids, -mids, near, -near]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ours = F.round_to_e4m3(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_grid_closed_form():
    vals = F.e4m3_value(np.arange(0, 0x7F, dtype=np.uint8))   # 0x7F is NaN
    expect = sorted(set([m * 2.0 ** -9 for m in range(8)] +
                        [(1 + j / 8) * 2.0 ** b for b in range(-6, 9) for j in range(8)]))
    expect = [x for x in expect if x <= 448]
    assert len(vals) == 127 and sorted(vals) == expect
    assert vals.max() == 448.0 and np.isnan(F.e4m3_value(np.uint8(0x7F)))
    # codes round-trip, sign bit included (zero maps to the positive code)
    codes = np.arange(0, 256, dtype=np.uint8)
    ok = (codes & 0x7F) != 0x7F
    back = F.e4m3_code(F.e4m3_value(codes[ok]))
    assert np.array_equal(back, np.where(codes[ok] == 0x80, 0, codes[ok]))


def test_tile_exponent_is_the_smallest_that_fits():
    rng = np.random.default_rng(1)
    amax = np.concatenate([np.ldexp(rng.uniform(0.5, 1, 5000), rng.integers(-30, 30, 5000)),
                           448.0 * np.ldexp(1.0, np.arange(-20, 20)),                # exactly at a boundary
                           448.0 * np.ldexp(1.0, np.arange(-20, 20)) * (1 + 2.0 ** -40),
                           np.ldexp(1.0, np.arange(-30, 30))])
    e = F.tile_exponent(amax)
    assert (amax <= 448.0 * np.ldexp(1.0, e)).all()
    assert (amax > 448.0 * np.ldexp(1.0, e - 1)).all()
    assert F.tile_exponent(0.0) == 0


def test_quantisation_error_bound_and_bf16_exactness():
    rng = np.random.default_rng(2)
    w = round_to_bf16(rng.normal(0, 0.02, (3, 256, 384)) * np.exp(rng.normal(0, 2, (3, 256, 1))))
    codes, exps = F.quantize_fp8_tiles(w)
    deq = F.dequantize_fp8_tiles(codes, exps)
    scale = np.ldexp(1.0, np.repeat(np.repeat(exps, 128, -2), 128, -1))
    normal = np.abs(w) / scale >= 2.0 ** -6
    err = np.abs(deq - w)
    assert (err[normal] <= 2.0 ** -4 * np.abs(w[normal])).all()        # half a step of 3 mantissa bits
    assert (err[~normal] <= 2.0 ** -10 * scale[~normal]).all()          # half the subnormal step
    assert np.array_equal(round_to_bf16(deq), deq)                       # every value is a bf16 value
    assert (np.abs(deq) <= 448.0 * scale).all()


def test_values_already_on_the_grid_round_trip_exactly():
    rng = np.random.default_rng(3)
    grid = F.e4m3_value(rng.integers(0, 0x7F, (128, 128)).astype(np.uint8)) * rng.choice([-1, 1], (128, 128))
    grid[5, 7] = 448.0                                                   # the tile's amax sits on the top
    w = grid * 2.0 ** -11
    codes, exps = F.quantize_fp8_tiles(w)
    assert exps[0, 0] == -11
    assert np.array_equal(F.dequantize_fp8_tiles(codes, exps), w)


def test_partial_tiles_brute_force():
    rng = np.random.default_rng(4)
    w = rng.normal(0, 1, (2, 200, 150)) * np.ldexp(1.0, rng.integers(-8, 8, (2, 200, 150)))
    w[1, 128:, :128] = 0.0                                               # an all-zero tile
    codes, exps = F.quantize_fp8_tiles(w)
    assert exps.shape == (2, 2, 2) and codes.shape == w.shape
    for n in range(2):
        for i in range(2):
            for j in range(2):
                blk = w[n, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                amax = np.abs(blk).max()
                e = 0 if amax == 0 else next(e for e in range(-60, 60) if amax <= 448.0 * 2.0 ** e)
                assert exps[n, i, j] == e
                for r in range(0, blk.shape[0], 37):
                    for c in range(0, blk.shape[1], 29):
                        x = blk[r, c] / 2.0 ** e
                        cand = F.e4m3_value(np.arange(0, 0x7F, dtype=np.uint8))
                        cand = np.concatenate([cand, -cand])
                        d = np.abs(cand - x)
                        best = cand[d == d.min()]
                        got = F.e4m3_value(codes[n, i * 128 + r, j * 128 + c])
                        assert got in best                               # a nearest grid value
    assert exps[1, 1, 0] == 0 and (codes[1, 128:, :128] == 0).all()


def test_round_to_e4m3_matches_ml_dtypes():
    """A second library: ml_dtypes' float8_e4m3fn conversion of fp32 values agrees too."""
    ml_dtypes = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(6)
    grid = F.e4m3_value(np.arange(0, 127, dtype=np.uint8))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    v = np.concatenate([rng.uniform(-448, 448, 50000), grid, -grid, mids, -mids,
                        np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    assert np.array_equal(F.round_to_e4m3(v.astype(np.float64)), v.astype(ml_dtypes.float8_e4m3fn).astype(np.float64))
