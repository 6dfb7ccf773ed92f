"""FP8 KV-cache quantization, plain numpy (CPU oracle).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

"Baidu AI Cloud: Day-0 support for hybrid-architecture LLMs", Optimization 2,
item 2 (KV Cache FP8 Tiled Quantization): each token's K (and V) of each head
is quantized in tiles of 128 elements, one scale per tile.

Readings where the page is silent:
* the FP8 format is E4M3 as in the OCP 8-bit floating point specification:
  1 sign, 4 exponent (bias 7), 3 mantissa bits, subnormals, no infinities,
  the all-ones pattern S.1111.111 is NaN, largest finite value 448;
* scale = amax / 448 in fp32 (correctly rounded), or 1 when amax == 0;
* code = E4M3 round-to-nearest-even of the fp32 quotient x / scale
  (correctly rounded fp32 division), saturating to +-448;
* the dequantized value is decode(code) * scale, exact in float64.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Value of each E4M3 code (uint8 array) as float64; NaN for 0x7f/0xff."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = sign * (1.0 + man / 8.0) * np.power(2.0, exp - 7)
    sub = sign * (man / 8.0) * 2.0 ** -6
    out = np.where(exp == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


# all finite non-negative codes and their values, ascending (0x00 .. 0x7e)
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x):
    """E4M3 code of each float (float32/float64 array): round to nearest,
    ties to the even code (even mantissa), saturating at +-448. NaN input
    maps to 0x7f."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # index of the largest representable value <= a, and the next one up
    lo = np.searchsorted(_POS_VALUES, a, side="right") - 1
    hi = np.minimum(lo + 1, len(_POS_VALUES) - 1)
    vlo, vhi = _POS_VALUES[lo], _POS_VALUES[hi]
    d_lo, d_hi = a - vlo, vhi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi != lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code)  # the sign survives, also for zero
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_tiles(x, tile=128):
    """Quantize the last axis of x (float32 values, e.g. bf16 widened) in
    tiles of `tile` elements. Returns (codes uint8 same shape, scales float32
    with the last axis divided by tile)."""
    x = np.asarray(x, np.float32)
    d = x.shape[-1]
    assert d % tile == 0
    t = x.reshape(x.shape[:-1] + (d // tile, tile))
    amax = np.max(np.abs(t), axis=-1)
    scale = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    q = (t / scale[..., None]).astype(np.float32)  # IEEE fp32 division
    codes = e4m3_encode(q).reshape(x.shape)
    return codes, scale.astype(np.float32)


def dequantize_tiles(codes, scales, tile=128):
    """float64 values of quantized tiles (inverse of quantize_tiles up to rounding)."""
    c = np.asarray(codes, np.uint8)
    d = c.shape[-1]
    v = e4m3_decode(c).reshape(c.shape[:-1] + (d // tile, tile))
    return (v * np.asarray(scales, np.float64)[..., None]).reshape(c.shape)
