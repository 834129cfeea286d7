"""FP8 E4M3 codec, written from the OCP 8-bit floating point format (OFP8).

Test infrastructure only: a plain, slow CPU restatement used to check the
CUDA path.  Nothing in the library imports it.

The serving system stores its attention cache in FP8 ("Do It Once, at Write
Time" on the Runway Characters page); the pages do not say which FP8 format.
This oracle takes E4M3 in its "fn" form: 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448.  Subnormals have exponent field 0 and
value m * 2^-9.

Encoding rounds to nearest, ties to even, and saturates finite values beyond
the range to +-448 (the "satfinite" behaviour).  Negative zero and negative
values that round to zero keep their sign (0x80).
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
MIN_NORMAL = 2.0 ** -6
MIN_SUBNORMAL = 2.0 ** -9
NAN_CODE = 0x7F


def _decode_one(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)


def decode_table() -> np.ndarray:
    """The 256 code values as float64 (NaN at 0x7F and 0xFF)."""
    return _TABLE.copy()


def decode(codes: np.ndarray) -> np.ndarray:
    """Decode uint8 codes to float64 (exact)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x: np.ndarray) -> np.ndarray:
    """Encode float32/float64 values to E4M3 codes (RNE, saturating finite).

    Steps, per element, for a = |x|:
      * a < 2^-6 (subnormal range): m = RNE(a * 2^9) in [0, 8]; m = 8 is the
        smallest normal, whose code is also 8.
      * otherwise e = floor(log2 a) (from frexp), m = RNE(a / 2^(e-3)) in
        [8, 16]; m = 16 carries into the exponent (e+1, m = 8).
      * e > 8, or e = 8 with m > 14, saturates to 448 (code 0x7E).
      * code = (e + 7) << 3 | (m - 8); the sign bit is OR-ed in last.
    Inputs are widened to float64 first (exact for float32), so every
    scaling by a power of two is exact and RNE is ``numpy.rint``.
    """
    xa = np.asarray(x)
    x64 = xa.astype(np.float64)
    sign = np.signbit(x64).astype(np.uint8) << 7
    a = np.abs(x64)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    out = np.zeros(a.shape, dtype=np.int64)

    sub = a < MIN_NORMAL
    if np.any(sub):
        out[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)

    nrm = ~sub
    if np.any(nrm):
        an = a[nrm]
        an = np.minimum(an, 2.0 ** 20)            # anything this large saturates
        _, ex = np.frexp(an)                      # an = f * 2^ex, f in [0.5, 1)
        e = ex.astype(np.int64) - 1               # floor(log2 an)
        m = np.rint(an / np.ldexp(1.0, e - 3)).astype(np.int64)
        carry = m == 16
        e = np.where(carry, e + 1, e)
        m = np.where(carry, 8, m)
        sat = (e > 8) | ((e == 8) & (m > 14))
        code = ((e + 7) << 3) | (m - 8)
        out[nrm] = np.where(sat, 0x7E, code)

    codes = out.astype(np.uint8) | sign
    codes = np.where(nan, np.uint8(NAN_CODE) | sign, codes).astype(np.uint8)
    return codes.reshape(xa.shape)


def half_ulp(y: np.ndarray) -> np.ndarray:
    """Half the spacing of E4M3 values around |y| (for |y| <= 448).

    Subnormal range spacing is 2^-9; in binade [2^e, 2^(e+1)) it is 2^(e-3).
    """
    a = np.abs(np.asarray(y, dtype=np.float64))
    _, ex = np.frexp(np.maximum(a, MIN_NORMAL))
    e = ex.astype(np.int64) - 1
    return 0.5 * np.ldexp(1.0, e - 3)
