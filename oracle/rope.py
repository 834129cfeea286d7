"""Rotary position embedding (RoPE), plain CPU restatement.

Test infrastructure only; nothing in the library imports it.

The Runway Characters page ("Do It Once, at Write Time") applies RoPE to each
new key once, as it enters the cache, and at each position reset applies one
"delta rotation" to the cached keys.  The pages do not give the RoPE variant;
this oracle takes the RoFormer form with adjacent pairs: for head size d and
pair index i < d/2, the pair (x[2i], x[2i+1]) is rotated by the angle
p * theta_i, theta_i = base^(-2i/d), at position p.

Two arithmetic forms are kept:

* ``rotate_f64`` -- the exact rotation in float64 with float64 cos/sin, used
  by the attention oracle and the closed-form checks.
* ``rotate_pinned_f32`` -- the form whose rounding is fixed so that cached
  FP8 bytes can be compared bit for bit: the table entries are
  c = fp32(cos(p*theta_i)), s = fp32(sin(p*theta_i)) from float64 libm, and
  y0 = fl(fl(x0*c) - fl(x1*s)), y1 = fl(fl(x0*s) + fl(x1*c)) in IEEE single
  precision, each product and sum rounded separately (no fused multiply-add).
  The delta rotation by -D uses the same table row for D with the signs
  flipped: y0 = fl(fl(a*c) + fl(b*s)), y1 = fl(fl(b*c) - fl(a*s)).

3-D variant (a video model's tokens carry a frame index t and a spatial row
y and column x; the pages give only "RoPE" and one position per token, so
this is a variant): the d/2 pairs are cut into a temporal section of T pairs,
then Y pairs for y, then X = d/2 - T - Y pairs for x.  Each section is a
RoPE of its own over its 2T (2Y, 2X) dimensions: local pair j of a section
of 2m dimensions turns by position_axis * base^(-2j/(2m)).  A token's
(t, y, x) position picks, for every pair, the coordinate of its section.
"""
from __future__ import annotations

import math

import numpy as np


def theta(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d) in float64, i < d/2 (libm pow per element)."""
    return np.array([math.pow(base, (-2.0 * i) / head_dim)
                     for i in range(head_dim // 2)], dtype=np.float64)


def sections(head_dim: int, pairs_t: int, pairs_y: int) -> np.ndarray:
    """Axis (0 = t, 1 = y, 2 = x) of every pair of the 3-D variant."""
    h = head_dim // 2
    if not (pairs_t >= 1 and pairs_y >= 0 and pairs_t + pairs_y <= h):
        raise ValueError("sections must fit the head")
    return np.r_[np.zeros(pairs_t, np.int64), np.ones(pairs_y, np.int64),
                 np.full(h - pairs_t - pairs_y, 2, np.int64)]


def theta_3d(head_dim: int, base: float, pairs_t: int, pairs_y: int) -> np.ndarray:
    """Per-pair angles of the 3-D variant: each section its own ladder
    base^(-2j/(2m)) over its m pairs (libm pow per element)."""
    ax = sections(head_dim, pairs_t, pairs_y)
    out = np.empty(head_dim // 2, dtype=np.float64)
    for a in range(3):
        idx = np.nonzero(ax == a)[0]
        m = len(idx)
        for j, i in enumerate(idx):
            out[i] = math.pow(base, (-2.0 * j) / (2 * m))
    return out


class Table:
    """fp32 cos/sin rows, built lazily from float64 libm cos/sin per element.

    ``th`` gives the per-pair angles (default: the 1-D ladder)."""

    def __init__(self, head_dim: int, base: float, max_position: int, th=None):
        self.head_dim = head_dim
        self.base = base
        self.max_position = max_position
        self.theta = theta(head_dim, base) if th is None else np.asarray(th, dtype=np.float64)
        self._rows: dict[int, tuple[np.ndarray, np.ndarray]] = {}

    def row(self, p: int):
        p = int(p)
        if not 0 <= p < self.max_position:
            raise ValueError(f"position {p} outside [0, {self.max_position})")
        r = self._rows.get(p)
        if r is None:
            ang = [float(p) * t for t in self.theta]
            c = np.array([math.cos(a) for a in ang], dtype=np.float64).astype(np.float32)
            s = np.array([math.sin(a) for a in ang], dtype=np.float64).astype(np.float32)
            r = (c, s)
            self._rows[p] = r
        return r

    def rows(self, positions):
        """(c, s) each [len(positions), d/2] float32."""
        cs = [self.row(p) for p in np.asarray(positions).reshape(-1)]
        c = np.stack([x[0] for x in cs]) if cs else np.zeros((0, self.head_dim // 2), np.float32)
        s = np.stack([x[1] for x in cs]) if cs else np.zeros((0, self.head_dim // 2), np.float32)
        return c, s


def rotate_pinned_f32(x: np.ndarray, c: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Rotate pairs of float32 ``x[..., d]`` by the angles whose fp32 cos/sin
    are ``c``, ``s`` (shape broadcastable to ``x[..., d/2]``).

    Every product and sum is rounded to float32 on its own.
    """
    x = np.asarray(x, dtype=np.float32)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    c = np.asarray(c, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    y = np.empty_like(x)
    y[..., 0::2] = (x0 * c) - (x1 * s)
    y[..., 1::2] = (x0 * s) + (x1 * c)
    return y


def unrotate_pinned_f32(x: np.ndarray, c: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Rotate pairs by the negated angle: the delta rotation's arithmetic."""
    x = np.asarray(x, dtype=np.float32)
    a = x[..., 0::2]
    b = x[..., 1::2]
    c = np.asarray(c, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    y = np.empty_like(x)
    y[..., 0::2] = (a * c) + (b * s)
    y[..., 1::2] = (b * c) - (a * s)
    return y


def rows_3d(table: Table, axis: np.ndarray, positions3: np.ndarray):
    """(c, s) [n, d/2] float32: pair i of token t takes the table row of its
    section's coordinate positions3[t, axis[i]]."""
    p3 = np.asarray(positions3, dtype=np.int64).reshape(-1, 3)
    n, h = p3.shape[0], len(axis)
    c = np.empty((n, h), np.float32)
    s = np.empty((n, h), np.float32)
    for t in range(n):
        for a in range(3):
            sel = axis == a
            if sel.any():
                cr, sr = table.row(int(p3[t, a]))
                c[t, sel] = cr[sel]
                s[t, sel] = sr[sel]
    return c, s


def rotate_f64_3d(x: np.ndarray, positions3: np.ndarray, th: np.ndarray, axis: np.ndarray) -> np.ndarray:
    """Exact-arithmetic 3-D rotation in float64: token t's pair i turns by
    positions3[t, axis[i]] * th[i] (token axis first in ``x``)."""
    x = np.asarray(x, dtype=np.float64)
    p3 = np.asarray(positions3, dtype=np.float64).reshape(-1, 3)
    ang = p3[:, axis] * th                                   # [n, d/2]
    ang = ang.reshape((ang.shape[0],) + (1,) * (x.ndim - 2) + (ang.shape[1],))
    c = np.cos(ang)
    s = np.sin(ang)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


def rotate_f64(x: np.ndarray, positions: np.ndarray, th: np.ndarray) -> np.ndarray:
    """Exact-arithmetic rotation in float64: x[..., t, :] by positions[t].

    ``x`` has shape [n, ..., d] with the token axis first; positions has n
    entries (any integer, negative allowed).
    """
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(positions, dtype=np.float64).reshape((-1,) + (1,) * (x.ndim - 1))
    ang = pos * th                      # [n, 1.., d/2]
    c = np.cos(ang)
    s = np.sin(ang)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y
