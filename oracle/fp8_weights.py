"""FP8 (E4M3) expert weights with one scale per 128 x 128 tile -- oracle side.

TEST INFRASTRUCTURE (see the package docstring): used only by the tests, the smoke check and
the benchmark's CPU baseline.  Shares no code with the CUDA path.

What the pages fix ("DeepSeek-V4 MoE", section "FP4 QAT 怎么做到反量化无损"; "MoE compute and
communication", section 四.2): expert weights stored as FP8 E4M3 (1 sign, 4 exponent, 3
mantissa bits), one scale factor shared by each 128 x 128 tile of a weight matrix, which halves
the weight bytes a decode step reads.  What they leave open, and the reading taken here:
  * the scale is a power of two, 2^e, with e the smallest integer for which the tile's largest
    magnitude fits the E4M3 range (amax <= 448 * 2^e); codes are round-to-nearest-even of
    w / 2^e.  A power-of-two scale makes dequantisation q * 2^e exact, and every such value
    (at most 4 significant bits) is exactly a bf16 value, so the quantised layer is exactly
    the bf16 layer evaluated on the dequantised weights;
  * tiles are counted per weight matrix from its first row and column (the last ones may be
    partial); an all-zero tile has e = 0; e is at least -126 (2^-e stays a normal fp32 value).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0          # 1.75 * 2^8, the largest finite E4M3 value
E4M3_MIN_NORMAL_EXP = -6  # normals down to 2^-6
E4M3_MANT_BITS = 3        # subnormals in steps of 2^-9
TILE = 128


def round_to_e4m3(v):
    """Nearest E4M3 value to each v (|v| <= 448), ties to even, as fp64.  Inside the binade
    [2^b, 2^(b+1)) the spacing is 2^(b-3); below 2^-6 (subnormals) it is 2^-9."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    if (a > E4M3_MAX).any():
        raise ValueError("value outside the E4M3 range")
    _, ex = np.frexp(np.where(a > 0, a, 1.0))       # a = m * 2^ex, m in [0.5, 1)
    b = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)     # binade exponent, clamped to the normal minimum
    spacing = np.ldexp(1.0, b - E4M3_MANT_BITS)
    q = np.round(a / spacing) * spacing             # a / spacing is exact; np.round: half to even
    return np.where(a > 0, np.copysign(q, v), 0.0)


def e4m3_code(q):
    """Bit pattern (uint8) of E4M3 values q (already on the grid); zero (either sign) -> 0x00."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    sign = (q < 0).astype(np.uint8) << 7
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    b = ex - 1
    normal = a >= 2.0 ** E4M3_MIN_NORMAL_EXP
    exp_field = np.where(normal, b + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, b) - 1.0, a / 2.0 ** -9) * np.where(normal, 8, 1)
    mant = np.rint(mant).astype(np.int64)
    code = (exp_field.astype(np.int64) << 3) | mant
    code = np.where(a > 0, code | sign.astype(np.int64), 0)
    return code.astype(np.uint8)


def e4m3_value(code):
    """fp64 value of E4M3 bit patterns (0x7F / 0xFF are NaN)."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return s * val


def tile_exponent(amax):
    """Smallest integer e with amax <= 448 * 2^e (0 for amax == 0), but at least -126 so that
    2^-e stays a normal fp32 number (only tiles with amax below 448 * 2^-127 are affected; they
    still fit).  With amax = m * 2^x, m in [0.5, 1): 448 = 0.875 * 2^9, so e = x - 9 when
    m <= 0.875, else x - 8."""
    amax = np.asarray(amax, dtype=np.float64)
    m, x = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.maximum(np.where(m <= 0.875, x - 9, x - 8), -126)
    return np.where(amax > 0, e, 0).astype(np.int64)


def quantize_fp8_tiles(w, tile=TILE):
    """Quantise weight matrices w [..., R, K] tile by tile.  Returns (codes uint8 [..., R, K],
    exps int64 [..., ceil(R/tile), ceil(K/tile)])."""
    w = np.asarray(w, dtype=np.float64)
    R, K = w.shape[-2:]
    lead = w.shape[:-2]
    nr, nk = -(-R // tile), -(-K // tile)
    exps = np.zeros(lead + (nr, nk), dtype=np.int64)
    codes = np.zeros(w.shape, dtype=np.uint8)
    for i in range(nr):
        for j in range(nk):
            blk = w[..., i * tile:(i + 1) * tile, j * tile:(j + 1) * tile]
            e = tile_exponent(np.abs(blk).max(axis=(-2, -1)))
            exps[..., i, j] = e
            scaled = blk * np.ldexp(1.0, -e)[..., None, None]   # exact: power-of-two scaling
            codes[..., i * tile:(i + 1) * tile, j * tile:(j + 1) * tile] = e4m3_code(round_to_e4m3(scaled))
    return codes, exps


def dequantize_fp8_tiles(codes, exps, tile=TILE):
    """fp64 weights q * 2^e from codes [..., R, K] and tile exponents [..., nr, nk]."""
    codes = np.asarray(codes)
    exps = np.asarray(exps, dtype=np.int64)
    R, K = codes.shape[-2:]
    scale = np.repeat(np.repeat(exps, tile, axis=-2), tile, axis=-1)[..., :R, :K]
    return e4m3_value(codes) * np.ldexp(1.0, scale)
