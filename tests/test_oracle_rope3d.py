"""Pins for the oracle's 3-D RoPE variant (temporal, row and column sections
of the rotation pairs, each its own RoPE; a reset turns only the temporal
pairs).

Checked against: the closed form of each section's angle ladder, the 1-D
RoPE when every pair is temporal, the relative-position property per axis
(q.k depends only on the three coordinate differences), each section
rotated on its own by the 1-D pinned arithmetic, cached keys within the
half-ulp bound of the exact rotation, the spatial codes untouched by a
reset, and attention over the ring invariant under a reset when the
queries' frame index moves with the keys'.
"""

import numpy as np
import pytest

from oracle import e4m3, Ring, TO_OLDEST
from oracle.attention import attention_exact
from oracle.rope import (Table, rotate_f64, rotate_f64_3d, rotate_pinned_f32, rows_3d, sections, theta,
                         theta_3d)
from workloads import TINY, f32_from_bf16, tiny_session

D = 128
T, Y = 16, 24          # 16 temporal pairs, 24 row pairs, 24 column pairs


def test_section_ladders_in_closed_form():
    th = theta_3d(D, 10000.0, T, Y)
    ax = sections(D, T, Y)
    assert list(np.bincount(ax)) == [T, Y, D // 2 - T - Y]
    for a, (lo, m) in enumerate([(0, T), (T, Y), (T + Y, D // 2 - T - Y)]):
        for j in range(m):
            assert th[lo + j] == pytest.approx(10000.0 ** (-j / m), rel=1e-15)
    assert np.array_equal(theta_3d(D, 10000.0, D // 2, 0), theta(D, 10000.0))
    with pytest.raises(ValueError):
        sections(D, 0, 8)


def test_all_temporal_is_the_1d_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, D))
    pos = rng.integers(0, 500, 5)
    p3 = np.stack([pos, rng.integers(0, 50, 5), rng.integers(0, 50, 5)], axis=1)
    a = rotate_f64_3d(x, p3, theta_3d(D, 10000.0, D // 2, 0), sections(D, D // 2, 0))
    assert np.abs(a - rotate_f64(x, pos, theta(D, 10000.0))).max() <= 1e-12


def test_dot_product_depends_only_on_coordinate_differences():
    rng = np.random.default_rng(1)
    th, ax = theta_3d(D, 10000.0, T, Y), sections(D, T, Y)
    q = rng.standard_normal((1, D))
    k = rng.standard_normal((1, D))
    a = np.array([[7, 3, 11]])
    b = np.array([[2, 9, 4]])
    ref = (rotate_f64_3d(q, a, th, ax) * rotate_f64_3d(k, b, th, ax)).sum()
    for shift in ([5, 0, 0], [0, 13, 0], [0, 0, 21], [40, 17, 3]):
        s = np.array([shift])
        got = (rotate_f64_3d(q, a + s, th, ax) * rotate_f64_3d(k, b + s, th, ax)).sum()
        assert got == pytest.approx(ref, abs=1e-9)
    # but not only on one axis: moving the row alone changes it
    moved = (rotate_f64_3d(q, a + [[0, 5, 0]], th, ax) * rotate_f64_3d(k, b, th, ax)).sum()
    assert abs(moved - ref) > 1e-6


def test_pinned_3d_rotation_is_each_section_rotated_on_its_own():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, D)).astype(np.float32)
    p3 = np.array([[3, 1, 2], [100, 7, 7], [0, 0, 0], [511, 63, 31]])
    full = Table(D, 10000.0, 1024, theta_3d(D, 10000.0, T, Y))
    c, s = rows_3d(full, sections(D, T, Y), p3)
    got = rotate_pinned_f32(x, c, s)
    for a, (lo, m) in enumerate([(0, T), (T, Y), (T + Y, D // 2 - T - Y)]):
        sect = Table(2 * m, 10000.0, 1024)              # a plain 1-D RoPE over 2m dims
        cs, ss = sect.rows(p3[:, a])
        want = rotate_pinned_f32(x[:, 2 * lo:2 * (lo + m)], cs, ss)
        assert np.array_equal(got[:, 2 * lo:2 * (lo + m)], want)


def _ring3d(prefix=0):
    return Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position, TINY.rope_base,
                prefix=prefix, rope3d=(8, 8))


def _pos3(frame_idx, n):
    """Frame index, then a 3 x 4 grid of row, column (12 tokens)."""
    t = np.arange(n)
    return np.stack([np.full(n, frame_idx), t // 4, t % 4], axis=1)


def _session3d(ring, frames, upto):
    ring.calibrate(f32_from_bf16(frames[0][1]), f32_from_bf16(frames[0][2]), _pos3(0, TINY.tokens))
    for i in range(upto):
        ring.write(f32_from_bf16(frames[i][1]), f32_from_bf16(frames[i][2]), _pos3(i, TINY.tokens))


def test_cached_keys_within_half_ulp_of_exact_3d_rope():
    frames = tiny_session()
    r = _ring3d()
    _session3d(r, frames, 3)
    for i in range(3):
        k = f32_from_bf16(frames[i][1]).astype(np.float64)
        y = r.rope_f64(k, _pos3(i, TINY.tokens)) / r.scale_k.astype(np.float64)[None, :, None]
        got = e4m3.decode(r.K[:, i * TINY.tokens:(i + 1) * TINY.tokens]).transpose(1, 0, 2)
        # half an e4m3 ulp plus the fp32 rotate / scale rounding; values past
        # the calibration frame's range saturate at 448
        inr = np.abs(y) <= 448.0
        assert np.all((np.abs(got - y) <= e4m3.half_ulp(y) + 4e-7 * (np.abs(y) + 1))[inr])
        assert np.all(np.abs(got[~inr]) == 448.0) and inr.mean() > 0.95
    assert np.array_equal(r.slot_pos[:36], np.repeat(np.arange(3), 12))


def test_reset_turns_only_temporal_pairs_and_keeps_attention():
    frames = tiny_session()
    r = _ring3d()
    _session3d(r, frames, 7)                 # 84 tokens in 48 slots: wrapped
    q = f32_from_bf16(frames[7][0])
    qpos = _pos3(7, TINY.queries)
    before = attention_exact(r, q, qpos)
    K0 = r.K.copy()
    d = r.delta_rotate(TO_OLDEST)
    assert d == 3                            # the oldest frame index left in the ring
    assert np.array_equal(r.K[:, :, 16:], K0[:, :, 16:])   # spatial codes untouched
    assert not np.array_equal(r.K[:, :, :16], K0[:, :, :16])
    after = attention_exact(r, q, qpos - [[d, 0, 0]])
    v_rms = np.sqrt(np.mean(f32_from_bf16(frames[0][2]).astype(np.float64) ** 2))
    err = np.abs(before - after).max()
    assert 0 < err < 0.05 * v_rms


def test_3d_needs_explicit_positions():
    r = _ring3d()
    x = np.zeros((2, TINY.heads, TINY.head_dim), np.float32)
    with pytest.raises(ValueError):
        r.calibrate(x, x)
    with pytest.raises(ValueError):
        r.calibrate(x, x, np.zeros(2, np.int64))
