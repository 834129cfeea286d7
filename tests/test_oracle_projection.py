"""Pins for the oracle's QKV projection (the step in front of the cache
write and the attention: bf16 activations times bf16 weights, summed, then
rounded once to bf16).

Checked against: an independent round-to-nearest-even built from the
sorted list of every finite bf16 value and exact rational arithmetic
(ties, one float64 step either side of a tie, subnormals, the overflow
threshold), torch's float32 -> bf16 conversion on values float32 holds
exactly, a brute-force projection in rationals on tiny inputs, identity and
scaled-identity weights, and the column blocks (queries, keys, values).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle.projection import bf16_rne_from_f64, bf16_to_f64, project_qkv

# every finite bf16 value, ascending, with a pattern for each (+0 for zero)
_PATS = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
_VALS = bf16_to_f64(_PATS)
_FIN = np.isfinite(_VALS) & ~((_PATS == 0x8000))
_ORDER = np.argsort(_VALS[_FIN], kind="stable")
_SORTED_VALS = [Fraction(float(v)) for v in _VALS[_FIN][_ORDER]]
_SORTED_PATS = _PATS[_FIN][_ORDER]
_MAX = _SORTED_VALS[-1]
_OVERFLOW_AT = _MAX + (Fraction(2) ** 127 * Fraction(1, 1 << 8))   # max + half its ulp


def _rne_exact(q: Fraction, negative_zero=False) -> int:
    """bf16 pattern nearest to the rational q (ties to the even pattern)."""
    if q >= _OVERFLOW_AT:
        return 0x7F80
    if q <= -_OVERFLOW_AT:
        return 0xFF80
    lo, hi = 0, len(_SORTED_VALS) - 1
    while hi - lo > 1:                       # bracket: sorted[lo] <= q <= sorted[hi]
        mid = (lo + hi) // 2
        if _SORTED_VALS[mid] <= q:
            lo = mid
        else:
            hi = mid
    if q >= _SORTED_VALS[hi]:
        lo = hi
    a, b = _SORTED_VALS[lo], _SORTED_VALS[min(lo + 1, len(_SORTED_VALS) - 1)]
    da, db = q - a, b - q
    if da < db or (da == db and int(_SORTED_PATS[lo]) & 1 == 0):
        pat = int(_SORTED_PATS[lo])
    else:
        pat = int(_SORTED_PATS[min(lo + 1, len(_SORTED_VALS) - 1)])
    if pat == 0 and (q < 0 or (q == 0 and negative_zero)):
        return 0x8000
    return pat


def _check(values):
    values = np.asarray(values, dtype=np.float64)
    got = bf16_rne_from_f64(values)
    want = [_rne_exact(Fraction(float(v)), np.signbit(v)) for v in values]
    bad = [(float(v), hex(int(g)), hex(w)) for v, g, w in zip(values, got, want) if int(g) != w]
    assert not bad, bad[:5]


def test_closed_form_roundings():
    cases = [(1.0, 0x3F80), (-2.0, 0xC000), (1 + 2 ** -8, 0x3F80), (1 + 3 * 2 ** -8, 0x3F82),
             (1 + 2 ** -8 + 2 ** -40, 0x3F81), (0.0, 0x0000), (-0.0, 0x8000),
             (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (1.5 * 2.0 ** -134, 0x0001),
             (3.0 * 2.0 ** -134, 0x0002), (float("inf"), 0x7F80), (2.0 ** 128, 0x7F80)]
    for x, bits in cases:
        assert int(bf16_rne_from_f64(np.array([x]))[0]) == bits, (x, hex(bits))
    assert int(bf16_rne_from_f64(np.array([np.nan]))[0]) == 0x7FC0


def test_ties_and_their_neighbours_against_exact_rounding():
    rng = np.random.default_rng(0)
    pats = rng.integers(0, 0x7F7F, 3000).astype(np.uint16)     # positive finite bf16
    base = bf16_to_f64(pats)
    nxt = bf16_to_f64(pats + 1)
    mid = (base + nxt) / 2                                    # exact in float64
    vals = np.concatenate([mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf), base])
    vals = np.concatenate([vals, -vals])
    _check(vals)


def test_random_values_all_ranges_against_exact_rounding():
    rng = np.random.default_rng(1)
    m = rng.uniform(0.5, 1.0, 4000)
    e = rng.integers(-140, 129, 4000)
    vals = np.ldexp(m, e) * rng.choice([-1.0, 1.0], 4000)
    edge = np.array([2.0 ** 127 * (2 - 2 ** -8), np.nextafter(2.0 ** 127 * (2 - 2 ** -8), 0),
                     2.0 ** -126, np.nextafter(2.0 ** -126, 0), 2.0 ** -126 - 2.0 ** -134])
    _check(np.concatenate([vals, edge, -edge]))


def test_agrees_with_torch_on_values_float32_holds():
    rng = np.random.default_rng(2)
    x32 = (rng.standard_normal(200_000) * np.exp2(rng.integers(-30, 30, 200_000))).astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_rne_from_f64(x32.astype(np.float64)), want)


def _bf16(rng, shape, scale=1.0):
    return bf16_rne_from_f64(rng.standard_normal(shape) * scale)


def test_projection_equals_rational_brute_force():
    rng = np.random.default_rng(3)
    H, d, n, dm = 2, 4, 3, 24
    x = _bf16(rng, (n, dm))
    w = _bf16(rng, (3 * H * d, dm), 0.2)
    q, k, v = project_qkv(x, w, H, d)
    xf = [[Fraction(float(a)) for a in row] for row in bf16_to_f64(x)]
    wf = [[Fraction(float(a)) for a in row] for row in bf16_to_f64(w)]
    for t in range(n):
        for c in range(3 * H * d):
            exact = sum(a * b for a, b in zip(xf[t], wf[c]))
            blk, hh, j = c // (H * d), (c % (H * d)) // d, c % d
            got = (q, k, v)[blk][t, hh, j]
            assert int(got) == _rne_exact(exact), (t, c)


def test_float64_sum_is_exact_at_production_width():
    """Dm = 5,120, N(0,1) activations and N(0, 0.02^2) weights: the float64
    sum equals the rational one (so the single rounding is the exact one)."""
    rng = np.random.default_rng(4)
    x = bf16_to_f64(_bf16(rng, (2, 5120)))
    w = bf16_to_f64(_bf16(rng, (3, 5120), 0.02))
    y = x @ w.T
    for t in range(2):
        for c in range(3):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(x[t], w[c]))
            assert Fraction(float(y[t, c])) == exact


def test_identity_blocks_and_column_order():
    rng = np.random.default_rng(5)
    H, d, n = 3, 8, 5
    hd = H * d
    x = _bf16(rng, (n, hd))
    eye = np.eye(hd)
    w = bf16_rne_from_f64(np.concatenate([eye, 2 * eye, -eye]))
    q, k, v = project_qkv(x, w, H, d)
    xf = bf16_to_f64(x).reshape(n, H, d)
    assert np.array_equal(bf16_to_f64(q), xf)
    assert np.array_equal(bf16_to_f64(k), 2 * xf)
    assert np.array_equal(bf16_to_f64(v), -xf)
    # only the key block non-zero: queries and values are +0
    w2 = bf16_rne_from_f64(np.concatenate([0 * eye, eye, 0 * eye]))
    q, k, v = project_qkv(x, w2, H, d)
    assert not q.any() and not v.any() and np.array_equal(bf16_to_f64(k), xf)
    with pytest.raises(ValueError):
        project_qkv(x, w[:-1], H, d)
