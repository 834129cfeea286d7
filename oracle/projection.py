"""QKV projection feeding the cache, plain CPU restatement.

Test infrastructure only; nothing in the library imports it.

The Runway Characters page names "fused pre-attention kernels" among the
changes that alter the model's numerics ("Judging Quality When Pixels
Can't"): the work between a block's input and its attention, i.e. the QKV
projection, the keys' and queries' RoPE and the FP8 quantisation that the
cache write and the attention then use.  The page gives no formula; this
oracle takes the plainest reading:

* the projection is ``y = x W^T`` of bf16 activations ``x [n, Dm]`` and bf16
  weights ``W [3 H d, Dm]`` (row-major, output by input, the layout of a
  linear layer's weight), summed without intermediate rounding and rounded
  once to bf16 (round to nearest, ties to even), the format a QKV projection
  emits;
* output columns [0, H d) are the queries, [H d, 2 H d) the keys and
  [2 H d, 3 H d) the values, each reshaped to [n, H, d];
* the keys and values then enter the ring exactly as a frame written with
  the write's arithmetic, and the queries are what the attention takes.

The sum is taken in float64: every bf16 x bf16 product is exact there, and
for the inputs the tests use (Dm up to a few thousand, exponents of
N(0, sigma^2) draws) the partial sums stay within float64's 53 bits, so the
float64 sum is the exact one (checked against rational arithmetic in the
tests); the single rounding to bf16 is done here from float64, not through
float32, so it is not a double rounding.
"""
from __future__ import annotations

import numpy as np

_BF16_MIN_NORMAL_EXP = -126       # smallest normal exponent (as in fp32)
_BF16_SUBNORMAL_STEP = 2.0 ** -133
_BF16_OVERFLOW = 2.0 ** 128       # |rounded| at or above this is infinite


def bf16_rne_from_f64(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of float64 values, rounded once to nearest,
    ties to even: 8 significant bits for normal values (exponent >= -126),
    a fixed step of 2^-133 below, infinity when the rounded magnitude reaches
    2^128; NaN becomes the quiet NaN 0x7FC0 with its sign."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(a)                       # a = m 2^e, m in [0.5, 1)
    normal = (a > 0) & np.isfinite(a) & (e - 1 >= _BF16_MIN_NORMAL_EXP)
    # normal: keep 8 significant bits, m 2^8 in [128, 256) rounded to even
    out[normal] = np.ldexp(np.round(np.ldexp(m[normal], 8)), e[normal] - 8)
    sub = (a > 0) & ~normal & np.isfinite(a)
    out[sub] = np.round(a[sub] / _BF16_SUBNORMAL_STEP) * _BF16_SUBNORMAL_STEP
    out[a == 0] = 0.0
    out[np.isinf(a)] = np.inf
    out[out >= _BF16_OVERFLOW] = np.inf
    out = np.copysign(out, x)
    bits = (out.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    bits[nan] = np.where(np.signbit(x[nan]), 0xFFC0, 0x7FC0).astype(np.uint16)
    return bits


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """float64 values of bf16 bit patterns."""
    b = np.asarray(b, dtype=np.uint16)
    with np.errstate(invalid="ignore"):      # NaN patterns widen to NaN
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def project_qkv(x_bits: np.ndarray, w_bits: np.ndarray, heads: int, head_dim: int):
    """(q, k, v) bf16 bit patterns, each [n, heads, head_dim], of the
    projection of ``x_bits [n, Dm]`` by ``w_bits [3 heads head_dim, Dm]``."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    n, dm = x.shape
    hd = heads * head_dim
    if w.shape != (3 * hd, dm):
        raise ValueError(f"weights must be [{3 * hd}, {dm}], got {w.shape}")
    y = x @ w.T                               # float64, [n, 3 H d]
    yb = bf16_rne_from_f64(y)
    return tuple(yb[:, i * hd:(i + 1) * hd].reshape(n, heads, head_dim) for i in range(3))
