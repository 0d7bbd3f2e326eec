"""bfloat16 encode/decode for the oracle (test infrastructure only).

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits (bias 127), 7 stored significand bits.  Decoding is exact.  Encoding
follows the IEEE-754 round-to-nearest, ties-to-even rule applied directly to
the fp64 value (no intermediate rounding to binary32):

    q = 2**(max(e, -126) - 7)      quantum of the binade of |x| (e = floor(log2|x|))
    n = nearest integer to |x|/q, ties to even
    result = sign * n * q          (overflow to infinity when n*q >= 2**128)

NaN encodes as the quiet NaN 0x7FC0 with the input's sign.
"""
from __future__ import annotations

import numpy as np


def to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def from_f64(x) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    inf = np.isinf(a)
    fin = ~(nan | inf)
    nz = fin & (a > 0)

    mant, exp = np.frexp(a[nz])            # a = mant * 2**exp, mant in [0.5, 1)
    e = exp.astype(np.int64) - 1           # a in [2**e, 2**(e+1))
    q_exp = np.maximum(e, -126) - 7
    n = np.rint(np.ldexp(a[nz], -q_exp))   # exact scaling; rint = ties-to-even
    val = np.ldexp(n, q_exp)
    over = val >= 2.0 ** 128
    val32 = np.where(over, np.inf, val).astype(np.float32)   # exact: val is a bf16 value
    mag = (val32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out[nz] = mag
    # zeros keep magnitude 0; infinities and NaNs
    out[inf] = np.uint16(0x7F80)
    out[nan] = np.uint16(0x7FC0)
    out = np.where(sign, out | np.uint16(0x8000), out).astype(np.uint16)
    return out


def round_f64(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, returned as float64."""
    return to_f64(from_f64(x))
