"""E4M3 and bfloat16 codecs of the oracle (test infrastructure only).

E4M3 here is the OCP "E4M3FN" 8-bit float that FP8 GEMMs on Hopper and
Blackwell consume: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
no infinities, NaN = S.1111.111, largest finite 448, smallest subnormal 2^-9.

* decode: the value from the bits, exactly, in float64;
* encode: the nearest finite code to a float64 value, a tie going to the code
  whose mantissa LSB is 0, magnitudes beyond 448 saturating to 448, the sign
  kept on zero results (a reading: this is round-to-nearest-even with
  saturation, the behaviour of a saturating hardware conversion).

bfloat16 values are carried as uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values, straight from the bit fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    v = sign * np.where(e == 0, subnormal, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


# the 127 non-negative finite values, codes 0x00..0x7E, strictly increasing
_POS_VALUES = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
assert np.all(np.diff(_POS_VALUES) > 0)


def e4m3_encode(values, chunk: int = 1 << 22) -> np.ndarray:
    """float64 values -> uint8 codes: nearest finite E4M3 value, ties to the even
    code, saturating at +-448, sign kept on zero results, NaN -> 0x7F."""
    v = np.asarray(values, dtype=np.float64)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for s in range(0, flat.size, chunk):
        x = flat[s:s + chunk]
        a = np.abs(x)
        hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 1, 0x7E)
        lo = hi - 1
        d_lo = a - _POS_VALUES[lo]
        d_hi = _POS_VALUES[hi] - a
        tie_pick = np.where(lo % 2 == 0, lo, hi)
        code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, tie_pick))
        code = np.where(a >= E4M3_MAX, 0x7E, code)
        code = code | np.where(np.signbit(x), 0x80, 0)
        code = np.where(np.isnan(x), 0x7F, code)
        out[s:s + chunk] = code.astype(np.uint8)
    return out.reshape(v.shape)


def e4m3_encode_bruteforce(values) -> np.ndarray:
    """Reference for ``e4m3_encode``: scan every finite code for the nearest
    one.  Quadratic; for pinning on small inputs only."""
    v = np.asarray(values, dtype=np.float64).reshape(-1)
    out = np.empty(v.size, dtype=np.uint8)
    all_codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    table = e4m3_decode(np.array(all_codes, dtype=np.uint8))
    for i, x in enumerate(v):
        if np.isnan(x):
            out[i] = 0x7F
            continue
        best, best_d = None, None
        for c, val in zip(all_codes, table):
            if (c >> 7) != int(np.signbit(x)):
                continue                       # same sign only (keeps -0 for negative underflow)
            d = abs(min(max(x, -E4M3_MAX), E4M3_MAX) - val)
            if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
                best, best_d = c, d
        out[i] = best
    return out.reshape(np.shape(values))


def bf16_decode(bits) -> np.ndarray:
    """uint16 bfloat16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def bf16_encode(values) -> np.ndarray:
    """float64 -> uint16 bfloat16 bits, round to nearest even directly from float64
    (8 significant bits).  Results below 2^-126 in magnitude are outside this
    oracle's range and are flushed through float32."""
    v = np.asarray(values, dtype=np.float64)
    m, e = np.frexp(v)                      # v = m * 2^e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0)                  # numpy rint: ties to even
    y = np.ldexp(r, e - 8)                  # exactly representable in bfloat16
    y32 = y.astype(np.float32)
    bits = (y32.view(np.uint32) >> 16).astype(np.uint16)
    return np.where(np.isnan(v), np.uint16(0x7FC0), bits).astype(np.uint16)
