"""Pins for the oracle's float64 attention over the ring cache.

Checked against: closed forms (equal keys give the mean of the values, one
filled slot returns its value), a pure-Python brute force on a tiny case,
and torch's scaled_dot_product_attention in float64 (a library routine).
The kernel-mirroring diagnostic is checked to converge to the reference as
its FP8 term counts grow.  The split of the slots into parts merged by their
log-sum-exps is checked against the whole softmax for arbitrary cuts, a
two-slot closed form and its degenerate cases.
"""
import math

import numpy as np
import pytest
import torch

from oracle import e4m3, Ring
from oracle.attention import (attention_emulated, attention_exact, attention_part_f64, attention_split,
                              merge_parts_f64)
from oracle.rope import rotate_f64
from workloads import TINY, f32_from_bf16, tiny_session, prod_session, PROD


def _tiny_ring(frames_written=3):
    frames = tiny_session()
    r = Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position)
    r.calibrate(f32_from_bf16(frames[0][1]), f32_from_bf16(frames[0][2]))
    for f in range(frames_written):
        r.write(f32_from_bf16(frames[f][1]), f32_from_bf16(frames[f][2]))
    return r, frames


def test_equal_keys_give_mean_of_values():
    r, frames = _tiny_ring(2)
    r.K[:, :r.n_valid, :] = r.K[:, :1, :]          # every filled slot holds the same key
    q = f32_from_bf16(frames[2][0])
    o = attention_exact(r, q, np.arange(12))
    _, v, _ = r.dequantised()
    want = v.mean(axis=1)                           # [H, d]
    assert np.allclose(o, want[None], atol=1e-12)


def test_single_filled_slot_returns_its_value():
    r = Ring(2, 64, 48, 64)
    rng = np.random.default_rng(3)
    k = rng.standard_normal((1, 2, 64)).astype(np.float32)
    v = rng.standard_normal((1, 2, 64)).astype(np.float32)
    r.calibrate(k, v)
    r.write(k, v)
    q = rng.standard_normal((5, 2, 64)).astype(np.float32) * 10
    o = attention_exact(r, q, np.arange(5))
    vv = e4m3.decode(r.V[:, 0, :]) * r.scale_v.astype(np.float64)[:, None]
    assert np.allclose(o, vv[None], atol=1e-12)


def test_empty_ring_gives_zeros():
    r = Ring(2, 64, 48, 64)
    q = np.ones((3, 2, 64), np.float32)
    assert np.all(attention_exact(r, q, np.arange(3)) == 0)


def test_pure_python_brute_force_tiny():
    r, frames = _tiny_ring(5)                       # 60 tokens: wrapped
    q = f32_from_bf16(frames[5][0])[:2]
    qpos = np.array([70, 71])
    o = attention_exact(r, q, qpos)
    th = r.table.theta
    for t in range(2):
        for h in range(TINY.heads):
            # rotate the query by hand
            qt = []
            for i in range(TINY.head_dim // 2):
                a = qpos[t] * th[i]
                x0, x1 = float(q[t, h, 2 * i]), float(q[t, h, 2 * i + 1])
                qt += [x0 * math.cos(a) - x1 * math.sin(a), x0 * math.sin(a) + x1 * math.cos(a)]
            scores = []
            for j in range(r.C):
                kj = [float(e4m3.decode(r.K[h, j, i])) * float(r.scale_k[h]) for i in range(TINY.head_dim)]
                scores.append(sum(a * b for a, b in zip(qt, kj)) / math.sqrt(TINY.head_dim))
            mx = max(scores)
            w = [math.exp(s - mx) for s in scores]
            z = sum(w)
            for i in range(0, TINY.head_dim, 7):
                val = sum(w[j] * float(e4m3.decode(r.V[h, j, i])) * float(r.scale_v[h]) for j in range(r.C)) / z
                assert math.isclose(o[t, h, i], val, rel_tol=1e-10, abs_tol=1e-12)


def test_matches_torch_sdpa_float64():
    r, frames = _tiny_ring(6)
    q = f32_from_bf16(frames[6][0])
    qpos = np.arange(72, 84)
    o = attention_exact(r, q, qpos)
    qt = rotate_f64(q.astype(np.float64), qpos, r.table.theta)
    k, v, _ = r.dequantised()
    Q = torch.from_numpy(qt.transpose(1, 0, 2).copy())[None]       # [1, H, n, d]
    K = torch.from_numpy(k.copy())[None]
    V = torch.from_numpy(v.copy())[None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V)[0].numpy().transpose(1, 0, 2)
    assert np.allclose(o, ref, atol=1e-12)


def test_kernel_mirror_converges_to_reference():
    r, frames = _tiny_ring(6)
    q = f32_from_bf16(frames[6][0])
    qpos = np.arange(72, 84)
    ref = attention_exact(r, q, qpos)
    errs = []
    for qt, pt in [(1, 1), (2, 2), (3, 2)]:
        errs.append(np.abs(attention_emulated(r, q, qpos, qt, pt, tile=16) - ref).max())
    assert errs[0] > errs[1] > errs[2]
    assert errs[2] < 1e-3


def test_kernel_mirror_single_tile_equals_reference_structure():
    """With enough terms the mirror's normaliser and rescaling are exact:
    a tile size of 1 (a rescale at every slot) and of 128 agree."""
    r, frames = _tiny_ring(6)
    q = f32_from_bf16(frames[6][0])
    a = attention_emulated(r, q, np.arange(72, 84), 3, 2, tile=1, tau=0.0)
    b = attention_emulated(r, q, np.arange(72, 84), 3, 2, tile=128)
    assert np.abs(a - b).max() < 1e-3


def test_kernel_mirror_two_f16_probability_terms():
    """The level-4 mirror (four query terms, probabilities as an f16 value
    plus the f16 rounding of what it left) errs far less than three terms
    with single f16 probabilities, and its probability pair carries p to
    about 22 bits (a lower bound on what two 11-bit terms give)."""
    r, frames = _tiny_ring(6)
    q = f32_from_bf16(frames[6][0])
    qpos = np.arange(72, 84)
    ref = attention_exact(r, q, qpos)
    e3 = np.abs(attention_emulated(r, q, qpos, 3, "f16", tile=16, tau=8.0) - ref).max()
    e4 = np.abs(attention_emulated(r, q, qpos, 4, "f16x2", tile=16, tau=8.0) - ref).max()
    assert e4 < e3 / 4 and e4 < 5e-5, (e3, e4)
    p = np.random.default_rng(0).uniform(2.0 ** -6, 2.0 ** 15, 10000).astype(np.float32)
    hi = p.astype(np.float16)
    lo = (p - hi.astype(np.float32)).astype(np.float16)
    rel = np.abs(hi.astype(np.float64) + lo.astype(np.float64) - p) / p
    assert rel.max() <= 2.0 ** -21


# ---------------------------------------------------------------- split merge
# The slots of one query tile shared among several workers: each part's
# normalised output with its log-sum-exp, merged.  Pinned by the identity
# that the merged parts are the whole softmax, by a two-slot closed form,
# and by the degenerate cases.



def test_split_merge_equals_whole_softmax_for_any_cut():
    r, frames = _tiny_ring(5)                       # wrapped tiny ring
    q = f32_from_bf16(frames[5][0])
    want = attention_exact(r, q)
    nv = r.n_valid
    rng = np.random.default_rng(21)
    cuts = [[0, nv], [0, 1, nv], [0, nv - 1, nv], [0, nv // 2, nv // 2, nv],
            [0, 0, nv, nv]]                         # empty parts at either end and inside
    for s in (3, 5, 8):
        inner = np.sort(rng.integers(0, nv + 1, size=s - 1))
        cuts.append([0, *inner.tolist(), nv])
    for b in cuts:
        got = attention_split(r, q, b)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-13), b


def test_split_merge_order_of_parts_does_not_matter():
    rng = np.random.default_rng(5)
    qt = rng.standard_normal((4, 2, 16)) * 3
    k = rng.standard_normal((2, 30, 16))
    v = rng.standard_normal((2, 30, 16))
    parts = [attention_part_f64(qt, k[:, a:b], v[:, a:b]) for a, b in ((0, 7), (7, 7), (7, 19), (19, 30))]
    fwd = merge_parts_f64(parts)
    rev = merge_parts_f64(parts[::-1])
    assert np.allclose(fwd, rev, rtol=1e-14, atol=1e-15)


def test_split_merge_two_slots_closed_form():
    # one query, one head, d = 4: scores s1 = 2 / sqrt(4) = 1 and s2 = 0
    qt = np.array([[[1.0, 1.0, 0.0, 0.0]]])
    k = np.array([[[1.0, 1.0, 0.0, 0.0], [1.0, -1.0, 0.0, 0.0]]])
    v = np.array([[[3.0, 0.0, 0.0, 1.0], [-1.0, 2.0, 0.0, 1.0]]])
    p1 = attention_part_f64(qt, k[:, :1], v[:, :1])
    p2 = attention_part_f64(qt, k[:, 1:], v[:, 1:])
    assert p1[1][0, 0] == 1.0 and p2[1][0, 0] == 0.0    # a one-slot part's lse is its score
    e = math.e
    want = (e * v[0, 0] + 1.0 * v[0, 1]) / (e + 1.0)
    assert np.allclose(merge_parts_f64([p1, p2])[0, 0], want, rtol=1e-15)


def test_split_merge_single_part_and_empty_parts():
    rng = np.random.default_rng(8)
    qt = rng.standard_normal((3, 2, 8))
    k = rng.standard_normal((2, 5, 8))
    v = rng.standard_normal((2, 5, 8))
    whole = attention_part_f64(qt, k, v)
    assert np.array_equal(merge_parts_f64([whole]), whole[0])          # weight exp(0) = 1
    empty = attention_part_f64(qt, k[:, :0], v[:, :0])
    assert np.all(empty[0] == 0) and np.all(np.isneginf(empty[1]))
    assert np.array_equal(merge_parts_f64([empty, whole, empty]), whole[0])
    got = merge_parts_f64([empty, empty])
    assert np.all(got == 0) and not np.any(np.isnan(got))


def test_split_part_lse_is_the_log_of_the_sum_of_exponentials():
    rng = np.random.default_rng(13)
    qt = rng.standard_normal((2, 1, 8)) * 4
    k = rng.standard_normal((1, 6, 8))
    v = rng.standard_normal((1, 6, 8))
    _, lse = attention_part_f64(qt, k, v)
    s = np.einsum("thd,hjd->thj", qt, k) / math.sqrt(8)
    assert np.allclose(lse, np.log(np.exp(s).sum(axis=2)), rtol=1e-14)


def test_split_rejects_bounds_that_do_not_cut_the_slots():
    r, frames = _tiny_ring(2)
    q = f32_from_bf16(frames[2][0])
    for b in ([1, r.n_valid], [0, r.n_valid - 1], [0, 5, 3, r.n_valid]):
        with pytest.raises(ValueError):
            attention_split(r, q, b, np.arange(12))
