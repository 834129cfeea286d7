"""Pins for the oracle's RoPE (RoFormer adjacent-pair form).

Checked against: textbook values of cos 1 and sin 1, the identity at
position 0, per-pair norm preservation, dependence of q·k on relative
position only, composition of rotations (the delta rotation's premise),
adjacency of the rotated pairs and the direction of rotation, and a rounding
bound for the pinned fp32 form.
"""
import math

import numpy as np

from oracle import rope

D, BASE = 64, 10000.0


def test_theta_geometric_progression():
    th = rope.theta(D, BASE)
    assert th[0] == 1.0
    ratio = th[1:] / th[:-1]
    assert np.allclose(ratio, BASE ** (-2.0 / D), rtol=1e-14)
    # the last frequency is base^(-(d-2)/d)
    assert math.isclose(th[-1], BASE ** (-(D - 2) / D), rel_tol=1e-14)


def test_table_textbook_values_and_identity():
    tab = rope.Table(D, BASE, 16)
    c0, s0 = tab.row(0)
    assert np.all(c0 == 1.0) and np.all(s0 == 0.0)
    c1, s1 = tab.row(1)
    # cos(1 rad), sin(1 rad) rounded to float32
    assert c1[0] == np.float32(0.5403023058681398)
    assert s1[0] == np.float32(0.8414709848078965)


def test_table_entries_are_rounded_libm_values():
    tab = rope.Table(D, BASE, 4096)
    th = rope.theta(D, BASE)
    for p in (0, 1, 7, 100, 1234, 4095):
        c, s = tab.row(p)
        ang = p * th
        assert np.all(np.abs(c.astype(np.float64) - np.cos(ang)) <= 2.0 ** -24 * np.abs(np.cos(ang)) + 1e-300)
        assert np.all(np.abs(s.astype(np.float64) - np.sin(ang)) <= 2.0 ** -24 * np.abs(np.sin(ang)) + 1e-300)


def test_rotation_acts_on_adjacent_pairs_counterclockwise():
    tab = rope.Table(D, BASE, 8)
    x = np.zeros((1, 1, D), np.float32)
    x[0, 0, 0] = 1.0
    c, s = tab.rows([1])
    y = rope.rotate_pinned_f32(x, c[:, None, :], s[:, None, :])
    assert y[0, 0, 0] == c[0, 0] and y[0, 0, 1] == s[0, 0]
    assert np.all(y[0, 0, 2:] == 0)
    yf = rope.rotate_f64(x.astype(np.float64), [1], tab.theta)
    assert math.isclose(yf[0, 0, 0], math.cos(1.0)) and math.isclose(yf[0, 0, 1], math.sin(1.0))
    assert np.all(yf[0, 0, 2:] == 0)


def test_pinned_position_zero_is_exact_identity():
    tab = rope.Table(D, BASE, 8)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, D)).astype(np.float32)
    c, s = tab.rows(np.zeros(5, int))
    assert np.array_equal(rope.rotate_pinned_f32(x, c[:, None, :], s[:, None, :]), x)
    assert np.array_equal(rope.unrotate_pinned_f32(x, c[0], s[0]), x)


def test_norm_of_each_pair_is_preserved():
    rng = np.random.default_rng(1)
    th = rope.theta(D, BASE)
    x = rng.standard_normal((50, 4, D))
    p = rng.integers(0, 100000, 50)
    y = rope.rotate_f64(x, p, th)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(nx, ny, rtol=1e-12, atol=1e-12)


def test_dot_product_depends_only_on_relative_position():
    rng = np.random.default_rng(2)
    th = rope.theta(D, BASE)
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    ref = None
    for a, b in [(10, 3), (17, 10), (1010, 1003), (40000, 39993)]:
        dot = float(np.sum(rope.rotate_f64(q, [a], th) * rope.rotate_f64(k, [b], th)))
        ref = dot if ref is None else ref
        assert math.isclose(dot, ref, rel_tol=1e-9, abs_tol=1e-9)
    # and it does change with the offset
    dot2 = float(np.sum(rope.rotate_f64(q, [11], th) * rope.rotate_f64(k, [3], th)))
    assert abs(dot2 - ref) > 1e-6


def test_rotations_compose():
    rng = np.random.default_rng(3)
    th = rope.theta(D, BASE)
    x = rng.standard_normal((20, 2, D))
    p = rng.integers(0, 50000, 20)
    delta = 31794
    back = rope.rotate_f64(rope.rotate_f64(x, p, th), np.full(20, -delta), th)
    direct = rope.rotate_f64(x, p - delta, th)
    assert np.allclose(back, direct, atol=1e-9)


def test_pinned_f32_within_rounding_of_exact_with_same_table():
    rng = np.random.default_rng(4)
    tab = rope.Table(D, BASE, 1000)
    x = rng.standard_normal((200, 3, D)).astype(np.float32)
    p = rng.integers(0, 1000, 200)
    c, s = tab.rows(p)
    y = rope.rotate_pinned_f32(x, c[:, None, :], s[:, None, :]).astype(np.float64)
    c64 = c.astype(np.float64)[:, None, :]
    s64 = s.astype(np.float64)[:, None, :]
    x0 = x[..., 0::2].astype(np.float64)
    x1 = x[..., 1::2].astype(np.float64)
    e0 = x0 * c64 - x1 * s64
    e1 = x0 * s64 + x1 * c64
    u = 2.0 ** -24
    b0 = u * (np.abs(x0 * c64) + np.abs(x1 * s64)) * (1 + u) + u * np.abs(e0)
    b1 = u * (np.abs(x0 * s64) + np.abs(x1 * c64)) * (1 + u) + u * np.abs(e1)
    assert np.all(np.abs(y[..., 0::2] - e0) <= b0 * 1.0001)
    assert np.all(np.abs(y[..., 1::2] - e1) <= b1 * 1.0001)
