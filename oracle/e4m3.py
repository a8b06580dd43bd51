"""OCP OFP8 E4M3 ("FN") codec, written from the format definition. Oracle: test use only.

The pages store compact values as "FP8 E4M3" (knlp.io "Asymmetric K16/V8 KV cache":
"values in FP8 E4M3"; DPS paper Sec. 2 names E4M3 for weights). They do not spell out
the bit layout, so the OCP 8-bit floating point specification v1.0 (E4M3 variant
without infinities) is taken:

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* exponent field 0 encodes subnormals m * 2**-9;
* S.1111.111 is NaN (0x7F / 0xFF); there is no infinity;
* the largest finite magnitude is 448 (0x7E).

Encoding is round-to-nearest, ties-to-even (the rounding family the DPS paper uses for
its FP16 -> E4M3 path, Sec. 3 "NestedFP" carry bit), saturating to +-448 ("satfinite"),
with the sign kept for values that round to zero.
"""

import numpy as np

E4M3_MAX = 448.0


def decode_code(code):
    """Value of one E4M3 code (0..255) as a Python float; NaN for 0x7F/0xFF."""
    code = int(code) & 0xFF
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * man * 2.0 ** -9          # subnormal: (m / 8) * 2**(1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def decode_table():
    """float64[256]: value of every code."""
    return np.array([decode_code(c) for c in range(256)], dtype=np.float64)


_TABLE = decode_table()
# Non-negative finite codes 0x00..0x7E, whose values increase with the code.
_POS_VALUES = _TABLE[:0x7F].copy()


def decode(codes):
    """Dequantise an array of uint8 codes to float64 (exact)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode_rne_satfinite(y):
    """Nearest E4M3 code to each float64 value ``y`` (ties to even code), saturating.

    ``y`` must be finite. Values whose magnitude is >= 448 map to +-448. The sign bit
    is set for negative values and for -0.0, including those that round to zero.
    """
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        raise ValueError("encode_rne_satfinite: non-finite input")
    a = np.abs(y)
    a_clamped = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a_clamped, side="left")   # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    v_hi = _POS_VALUES[hi]
    v_lo = _POS_VALUES[lo]
    d_hi = v_hi - a_clamped          # exact: both are short dyadic rationals
    d_lo = a_clamped - v_lo
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(a_clamped == v_hi, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    neg = np.signbit(y)
    return (mag | np.where(neg, 0x80, 0).astype(np.uint8)).astype(np.uint8)
