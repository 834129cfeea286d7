"""Pins for the oracle's FP8 E4M3 codec (OCP OFP8 E4M3, "fn" variant).

Every check here is independent of the codec's own code path: closed-form
values of the format, round-trip of all finite codes, ties-to-even at every
midpoint, saturation and signed-zero cases, a library cast (torch, and
ml_dtypes where installed), and the half-ulp error bound.
"""
import numpy as np
import pytest
import torch

from oracle import e4m3
from workloads import bf16_from_f32, f32_from_bf16


def test_closed_form_code_values():
    t = e4m3.decode_table()
    assert t[0x00] == 0.0 and not np.signbit(t[0x00])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == 2.0 ** -9            # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert t[0x08] == 2.0 ** -6            # smallest normal
    assert t[0x38] == 1.0
    assert t[0x3F] == 1.875
    assert t[0x40] == 2.0
    assert t[0x7E] == 448.0                # largest finite
    assert t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    finite = np.isfinite(t)
    assert finite.sum() == 254
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)        # codes 0..0x7E strictly increasing


def test_all_finite_codes_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes)
    assert np.array_equal(e4m3.encode(vals), codes)
    assert np.array_equal(e4m3.encode(vals.astype(np.float32)), codes)


def test_midpoints_round_to_even_and_neighbours_to_nearest():
    t = e4m3.decode_table()[:0x7F]          # 0 .. 448, increasing
    lo, hi = t[:-1], t[1:]
    mid = (lo + hi) / 2                    # exact in float64
    got = e4m3.encode(mid)
    lo_code = np.arange(0, 0x7E)
    want = np.where(lo_code % 2 == 0, lo_code, lo_code + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    eps = (hi - lo) * 1e-6
    assert np.array_equal(e4m3.encode(mid - eps), lo_code.astype(np.uint8))
    assert np.array_equal(e4m3.encode(mid + eps), (lo_code + 1).astype(np.uint8))
    # negative side mirrors with the sign bit
    assert np.array_equal(e4m3.encode(-mid), (want | 0x80).astype(np.uint8))


@pytest.mark.parametrize("x,code", [
    (448.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (465.0, 0x7E), (480.0, 0x7E),
    (1e30, 0x7E), (float(np.finfo(np.float32).max), 0x7E), (-1e30, 0xFE),
    (2.0 ** -10, 0x00),                 # half the smallest subnormal: tie to even 0
    (3 * 2.0 ** -11, 0x01),             # 0.75 of the smallest subnormal
    (3 * 2.0 ** -10, 0x02),             # 1.5 subnormal steps: tie to even 2
    (-(2.0 ** -11), 0x80),              # negative underflow keeps the sign
    (-0.0, 0x80), (0.0, 0x00),
    (15 * 2.0 ** -10, 0x08),            # 7.5 subnormal steps: rounds up to min normal
    (1.0625, 0x38), (1.0625 + 1e-7, 0x39), (1.1875, 0x3A),
])
def test_special_values(x, code):
    assert e4m3.encode(np.array([x]))[0] == code


def _torch_codes(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(x32, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_matches_torch_cast_on_all_bf16_patterns():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = f32_from_bf16(b)
    x = x[np.isfinite(x)]
    assert np.array_equal(e4m3.encode(x), _torch_codes(x))


def test_matches_torch_cast_on_random_float32():
    rng = np.random.default_rng(7)
    # mantissas uniform, exponents spanning the whole interesting range
    x = (rng.uniform(1, 2, 2_000_000) * np.exp2(rng.integers(-30, 12, 2_000_000))
         * rng.choice([-1, 1], 2_000_000)).astype(np.float32)
    assert np.array_equal(e4m3.encode(x), _torch_codes(x))


def test_matches_ml_dtypes_if_installed():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(500_000) * np.exp2(rng.integers(-14, 10, 500_000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    want = x.astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(e4m3.encode(x), want)


def test_half_ulp_error_bound():
    rng = np.random.default_rng(9)
    y = rng.uniform(-448, 448, 1_000_000) * np.exp2(-rng.integers(0, 16, 1_000_000))
    err = np.abs(e4m3.decode(e4m3.encode(y)) - y)
    assert np.all(err <= e4m3.half_ulp(y))


def test_bf16_helpers_round_to_nearest_even():
    # 1 + 2^-8 is a bf16 tie (between 1 and 1 + 2^-7): goes to even (1.0)
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5], dtype=np.float32)
    b = bf16_from_f32(x)
    assert list(f32_from_bf16(b)) == [1.0, 1.0 + 2.0 ** -6, -2.5]
