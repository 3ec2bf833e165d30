"""MXFP4 (E2M1) expert weights with one power-of-two scale per 1 x 32 sub-block, and their
lossless conversion to FP8 (E4M3) tiles with one scale per 128 x 128 tile -- oracle side.

TEST INFRASTRUCTURE (see the package docstring): used only by the tests, the smoke check and
the benchmark's CPU baseline.  Shares no code with the CUDA path.

What the pages fix ("DeepSeek-V4 MoE", section "FP4 QAT 怎么做到反量化无损"): expert weights in
FP4 E2M1 (1 sign, 2 exponent, 1 mantissa bit), one scale shared by each 1 x 32 sub-block; FP8
E4M3 tiles of 128 x 128 with one scale each; the FP4 -> FP8 dequantisation is lossless as long
as, inside each FP8 tile, the ratio of the largest to the smallest sub-block scale stays within
the FP8 exponent headroom; the forward pass computes on the FP8 form.  What they leave open, and
the reading taken here:
  * E2M1 values: exponent field 0 -> m * 0.5 (0 or 0.5), else (1 + m/2) * 2^(E-1): the grid
    {0, 0.5, 1, 1.5, 2, 3, 4, 6}; code = sign << 3 | E << 1 | m; zero is stored as +0;
  * sub-blocks are 32 consecutive elements of a row along K, counted from column 0;
  * the sub-block scale is 2^s with s the smallest integer for which the block's largest
    magnitude fits 6 * 2^s (no saturation), at least -114 -- then raised, where needed, to the
    largest s of its 128 x 128 tile minus 14, which is exactly the headroom: a value
    q * 2^t (q on the E2M1 grid) is an E4M3 value for every q iff -8 <= t <= 6, so with the FP8
    tile exponent E = (largest s of the tile) - 6 every sub-block has t = s - E in [-8, 6] and
    the conversion is exact.  An all-zero sub-block (its codes are 0) takes the largest s of
    its tile, MIN_EXP in an all-zero tile.  So every s fits an int8 (>= -128) and every tile
    exponent E is at least -120 (within the FP8 tiles' exponent range, >= -126);
  * codes are the round-to-nearest-even of w * 2^-s on the E2M1 grid.
"""
from __future__ import annotations

import numpy as np

from . import fp8_weights as F8

E2M1_MAX = 6.0
BLOCK = 32           # sub-block length along K
TILE = 128           # FP8 tile edge
HEADROOM = 14        # largest minus smallest sub-block exponent inside one FP8 tile
MIN_EXP = -114


def e2m1_value(code):
    """fp64 value of E2M1 codes (4-bit patterns, any integer array)."""
    c = np.asarray(code, dtype=np.int64) & 0xF
    s = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.ldexp(1.0, e - 1))
    return s * mag


GRID = e2m1_value(np.arange(8))  # the eight magnitudes, ascending with the code


def round_to_e2m1_code(v):
    """E2M1 code of the nearest grid value to each v (|v| <= 6), ties to the even mantissa
    bit (code bit 0 clear); zero (either sign) -> code 0."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    if (a > E2M1_MAX).any():
        raise ValueError("value outside the E2M1 range")
    d = np.abs(a[..., None] - GRID)                       # distance to each magnitude
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                                      # one or two nearest magnitudes
    even = cand & ((np.arange(8) & 1) == 0)
    pick = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    code = pick.astype(np.int64)
    return np.where((v < 0) & (code > 0), code | 8, code).astype(np.uint8)


def block_fit_exponent(amax):
    """Smallest integer s with amax <= 6 * 2^s, at least MIN_EXP.  With amax = m * 2^x,
    m in [0.5, 1): 6 = 0.75 * 2^3, so s = x - 3 when m <= 0.75, else x - 2."""
    amax = np.asarray(amax, dtype=np.float64)
    m, x = np.frexp(np.where(amax > 0, amax, 1.0))
    return np.maximum(np.where(m <= 0.75, x - 3, x - 2), MIN_EXP).astype(np.int64)


def quantize_mxfp4(w):
    """Quantise weight matrices w [..., R, K] (K a multiple of 32).  Returns (codes uint8
    [..., R, K] one 4-bit code per element, exps int64 [..., R, K/32])."""
    w = np.asarray(w, dtype=np.float64)
    R, K = w.shape[-2:]
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    lead = w.shape[:-2]
    blocks = w.reshape(lead + (R, K // BLOCK, BLOCK))
    amax = np.abs(blocks).max(axis=-1)                    # [..., R, K/32]
    fit = block_fit_exponent(amax)
    exps = np.empty_like(fit)
    for i in range(0, R, TILE):
        for j in range(0, K // BLOCK, TILE // BLOCK):
            f = fit[..., i:i + TILE, j:j + TILE // BLOCK]
            nz = amax[..., i:i + TILE, j:j + TILE // BLOCK] > 0
            top = np.where(nz, f, MIN_EXP).max(axis=(-2, -1), keepdims=True)
            floor = top - HEADROOM
            exps[..., i:i + TILE, j:j + TILE // BLOCK] = np.where(nz, np.maximum(f, floor), top)
    scaled = blocks * np.ldexp(1.0, -exps)[..., None]    # exact: power-of-two scaling
    codes = round_to_e2m1_code(scaled).reshape(w.shape)
    return codes, exps


def dequantize_mxfp4(codes, exps):
    """fp64 weights q * 2^s from codes [..., R, K] and sub-block exponents [..., R, K/32]."""
    codes = np.asarray(codes)
    scale = np.repeat(np.ldexp(1.0, np.asarray(exps, dtype=np.int64)), BLOCK, axis=-1)
    return e2m1_value(codes) * scale


def mxfp4_to_fp8(codes, exps):
    """The lossless conversion to FP8 tiles: for each 128 x 128 tile, E = (largest sub-block
    exponent of the tile) - 6 and each element's E4M3 code of q * 2^(s - E).  Returns (fp8 codes
    uint8 [..., R, K], tile exponents int64 [..., ceil(R/128), ceil(K/128)]) in the layout of
    fp8_weights.quantize_fp8_tiles."""
    codes = np.asarray(codes)
    exps = np.asarray(exps, dtype=np.int64)
    R, K = codes.shape[-2:]
    lead = codes.shape[:-2]
    nr, nk = -(-R // TILE), -(-K // TILE)
    tile_e = np.zeros(lead + (nr, nk), dtype=np.int64)
    out = np.zeros(codes.shape, dtype=np.uint8)
    for i in range(nr):
        for j in range(nk):
            s = exps[..., i * TILE:(i + 1) * TILE, j * (TILE // BLOCK):(j + 1) * (TILE // BLOCK)]
            E = s.max(axis=(-2, -1)) - 6
            tile_e[..., i, j] = E
            t = np.repeat(s, BLOCK, axis=-1) - E[..., None, None]
            q = e2m1_value(codes[..., i * TILE:(i + 1) * TILE, j * TILE:(j + 1) * TILE])
            v = q * np.ldexp(1.0, t)
            if (F8.round_to_e4m3(v) != v).any():
                raise ValueError("sub-block exponents exceed the FP8 headroom")
            out[..., i * TILE:(i + 1) * TILE, j * TILE:(j + 1) * TILE] = F8.e4m3_code(v)
    return out, tile_e
