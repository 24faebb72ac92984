"""FP8 e4m3 codec and per-(head, block) scaled quantisation.

"SoulX-LiveAct" (youleyou.com), 技术内核 / 上手实践指南: adaptive FP8 precision
and an FP8 KV cache.  The format itself is the OCP 8-bit floating point
e4m3 ("E4M3FN"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
subnormals at exponent 0, no infinities, S.1111.111 is NaN, largest finite
magnitude 448.

Readings taken (the pages give no scale rule):
  * one fp32 scale per (head, block): scale = amax / 448 over that head's
    values of the block; an all-zero block gets scale 1;
  * code = e4m3(x * (448 / amax)) with round-to-nearest-even and saturation
    to +-448; both the reciprocal and the product are single fp32 roundings,
    because the code is an integer decided by floating point and both
    sides must decide it in the same precision;
  * dequantised value = decode(code) * scale.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode(code) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for the NaN codes)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


def _finite_table():
    codes = np.arange(0, 0x7F, dtype=np.uint8)           # positive finite codes
    return codes, decode(codes)


def encode(x) -> np.ndarray:
    """float values -> uint8 codes, round to nearest (ties to even code),
    saturating to +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    codes, vals = _finite_table()                        # ascending in value
    a = np.abs(x)
    a_clip = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(vals, a_clip, side="left")      # first vals[hi] >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a_clip - vals[lo]
    d_hi = vals[hi] - a_clip
    # nearest representable magnitude; an exact midpoint goes to the even code
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi] & 1) == 0))
    mag = np.where(pick_hi, codes[hi], codes[lo])
    out = mag.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    out = np.where(np.isnan(x), np.uint8(0x7F), out)
    return out.astype(np.uint8)


def quantize(x_f32: np.ndarray):
    """Quantise one (head, block) group of fp32 values.

    Returns (codes uint8 same shape, scale as np.float32, scaled fp32 values
    x * inv that decided the codes)."""
    x = np.asarray(x_f32, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    if amax == 0:
        return np.zeros(x.shape, np.uint8), np.float32(1.0), x.copy()
    inv = np.float32(E4M3_MAX) / amax
    scale = amax / np.float32(E4M3_MAX)
    y = (x * inv).astype(np.float32)
    return encode(y), np.float32(scale), y


def boundary_distance(y: np.ndarray) -> np.ndarray:
    """Relative distance of each scaled value from the nearest e4m3 rounding
    midpoint; small values mark codes that rounding noise could flip."""
    _, vals = _finite_table()
    mids = (vals[1:] + vals[:-1]) / 2.0
    a = np.minimum(np.abs(np.asarray(y, dtype=np.float64)), E4M3_MAX)
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))
    return d / np.maximum(a, 2.0 ** -9)
