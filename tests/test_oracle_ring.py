"""Pins for the oracle's ring cache: calibration, write, delta rotation.

Checked against: the closed-form ring indexing, the calibration invariant
(each head's largest magnitude lands exactly on 448), the dequantised cache
against float64 RoPE within the half-ulp bound, a brute-force linear window
over the last ``capacity`` tokens, the page's own negative case (positions
by slot order go wrong after wrap-around), and the delta rotation against
float64 re-rotation and from-scratch quantisation.
"""
import numpy as np
import pytest

from oracle import e4m3, Ring, INT32_MIN, TO_OLDEST
from oracle.attention import (attention_exact, attention_linear_window,
                              attention_positions_by_slot_order,
                              attention_true_positions)
from oracle.rope import rotate_f64
from workloads import TINY, f32_from_bf16, tiny_session


def _ring(shape=TINY):
    return Ring(shape.heads, shape.head_dim, shape.capacity, shape.max_position, shape.rope_base)


def _f(x):
    return f32_from_bf16(x)


def test_ring_indexing_and_state():
    r = _ring()
    rng = np.random.default_rng(0)
    k = rng.standard_normal((30, TINY.heads, TINY.head_dim)).astype(np.float32)
    r.calibrate(k, k)
    total = 0
    for n in [12, 12, 20, 1, 47, 48, 5]:
        head_before = r.head
        slots = r.write(k[:1].repeat(n, 0), k[:1].repeat(n, 0))
        assert np.array_equal(slots, (head_before + np.arange(n)) % TINY.capacity)
        total += n
        assert r.head == total % TINY.capacity
        assert r.n_valid == min(total, TINY.capacity)
        assert r.next_pos == total
    with pytest.raises(ValueError):
        r.write(np.zeros((49, 2, 64), np.float32), np.zeros((49, 2, 64), np.float32))


def test_write_before_calibration_rejected():
    r = _ring()
    with pytest.raises(RuntimeError):
        r.write(np.zeros((1, 2, 64), np.float32), np.zeros((1, 2, 64), np.float32))


def test_calibration_maps_each_head_amax_to_448():
    frames = tiny_session()
    r = _ring()
    q, k, v = frames[0]
    r.calibrate(_f(k), _f(v))
    r.write(_f(k), _f(v))
    for h in range(TINY.heads):
        kc = r.K[h, :TINY.tokens]
        vc = r.V[h, :TINY.tokens]
        assert np.abs(e4m3.decode(kc)).max() == 448.0
        assert np.abs(e4m3.decode(vc)).max() == 448.0
    # scale is amax / 448 with amax taken after RoPE for keys
    kt = rotate_f64(_f(k).astype(np.float64), np.arange(TINY.tokens), r.table.theta)
    amax = np.abs(kt).max(axis=(0, 2))
    assert np.allclose(r.scale_k.astype(np.float64), amax / 448.0, rtol=1e-6)
    assert np.allclose(r.scale_v.astype(np.float64), np.abs(_f(v)).max(axis=(0, 2)) / 448.0, rtol=1e-7)


def test_zero_amax_gives_unit_scale():
    r = _ring()
    z = np.zeros((3, TINY.heads, TINY.head_dim), np.float32)
    r.calibrate(z, z)
    assert np.all(r.scale_k == 1.0) and np.all(r.inv_k == 1.0)


def test_dequantised_keys_within_half_ulp_of_exact_rope():
    frames = tiny_session()
    r = _ring()
    r.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    for f in range(3):
        r.write(_f(frames[f][1]), _f(frames[f][2]))
    k_all = np.concatenate([_f(frames[f][1]) for f in range(3)]).astype(np.float64)
    exact = rotate_f64(k_all, np.arange(36), r.table.theta)          # [36, H, d]
    sk = r.scale_k.astype(np.float64)[None, :, None]
    y = exact / sk
    got = e4m3.decode(r.K[:, :36, :]).transpose(1, 0, 2)
    # half an e4m3 ulp plus the fp32 rotate / scale rounding (a few 2^-24 relative);
    # later frames may exceed the calibration frame's range: those saturate at 448
    inr = np.abs(y) <= 448.0
    assert np.all((np.abs(got - y) <= e4m3.half_ulp(y) + 4e-7 * (np.abs(y) + 1))[inr])
    assert np.all(np.abs(got[~inr]) == 448.0) and inr.mean() > 0.99
    vexact = np.concatenate([_f(frames[f][2]) for f in range(3)]).astype(np.float64)
    yv = vexact / r.scale_v.astype(np.float64)[None, :, None]
    gotv = e4m3.decode(r.V[:, :36, :]).transpose(1, 0, 2)
    inr = np.abs(yv) <= 448.0
    assert np.all((np.abs(gotv - yv) <= e4m3.half_ulp(yv) + 4e-7 * (np.abs(yv) + 1))[inr])
    assert np.all(np.abs(gotv[~inr]) == 448.0)


def _run_tiny(reset_before=None):
    """Tiny workload through the oracle, keeping a time-ordered history."""
    frames = tiny_session()
    r = _ring()
    r.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    hist = []
    outs = []
    for f, (q, k, v) in enumerate(frames):
        if reset_before is not None and f == reset_before:
            r.delta_rotate(TO_OLDEST)
        pos = r.next_pos + np.arange(TINY.tokens)
        kc = r.quantise_keys(_f(k), pos)
        vc = r.quantise_values(_f(v))
        hist.append((kc, vc, pos))
        r.write(_f(k), _f(v))
        outs.append((r, q, pos))
    return r, hist


def test_wrapped_ring_equals_linear_window():
    frames = tiny_session()
    r = _ring()
    r.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    hist = []
    for f, (q, k, v) in enumerate(frames):
        pos = r.next_pos + np.arange(TINY.tokens)
        hist.append((r.quantise_keys(_f(k), pos), r.quantise_values(_f(v)), pos))
        r.write(_f(k), _f(v))
        o_ring = attention_exact(r, _f(q), pos)
        o_lin = attention_linear_window(hist, _f(q), pos, r)
        assert np.allclose(o_ring, o_lin, rtol=0, atol=1e-12), f
    assert r.total > TINY.capacity       # the ring wrapped


def test_slot_order_positions_wrong_only_after_wrap():
    """The page pins "ring + positions by slot order" as invalid."""
    frames = tiny_session()
    H, C, d = TINY.heads, TINY.capacity, TINY.head_dim
    raw_k = np.zeros((H, C, d))
    raw_v = np.zeros((H, C, d))
    slot_pos = np.full(C, INT32_MIN, dtype=np.int64)
    head, nv, nxt = 0, 0, 0
    r = _ring()
    seen_before = seen_after = False
    for f, (q, k, v) in enumerate(frames):
        n = TINY.tokens
        slots = (head + np.arange(n)) % C
        pos = nxt + np.arange(n)
        raw_k[:, slots, :] = _f(k).astype(np.float64).transpose(1, 0, 2)
        raw_v[:, slots, :] = _f(v).astype(np.float64).transpose(1, 0, 2)
        slot_pos[slots] = pos
        head, nv, nxt = (head + n) % C, min(C, nv + n), nxt + n
        good = attention_true_positions(raw_k, raw_v, slot_pos, _f(q), pos, r.table.theta)
        first = int(slot_pos[:nv].min())
        bad = attention_positions_by_slot_order(raw_k, raw_v, nv, _f(q), pos, r.table.theta, first)
        if nxt <= C or head == 0:
            # slot order equals time order: before wrap-around, or when the
            # head has come round to slot 0 again
            assert np.allclose(good, bad, atol=1e-12)
            seen_before = True
        else:
            assert np.abs(good - bad).max() > 1e-3
            seen_after = True
    assert seen_before and seen_after


def test_delta_zero_is_identity_and_rotation_is_deterministic():
    r, _ = _run_tiny()
    before = r.K.copy()
    r.delta_rotate(0)
    assert np.array_equal(r.K, before)
    r2, _ = _run_tiny()
    v_before = r.V.copy()
    r.delta_rotate(5)
    r2.delta_rotate(5)
    assert np.array_equal(r.K, r2.K)
    assert not np.array_equal(r.K, before)
    assert np.array_equal(r.V, v_before)          # values are never rotated


def test_delta_zero_keeps_negative_zero_codes():
    """A zero delta is the identity on every code, signed zeros included: a
    -0 code (0x80) paired with a positive value keeps its sign, in both
    positions of the pair, while a nonzero delta rotates it like any value."""
    r = _ring()
    k = np.zeros((TINY.tokens, TINY.heads, TINY.head_dim), np.float32)
    k[:, :, 0::2] = 1.0                 # positive first elements
    k[:, :, 3::4] = -1e-30              # second elements of odd pairs round to -0
    k[:, :, 2::4] = -1e-30              # first elements of odd pairs too, partners above
    k[:, :, 1::4] = 0.5
    v = np.ones_like(k)
    r.calibrate(k, v, np.zeros(TINY.tokens, np.int32))
    r.write(k, v, np.zeros(TINY.tokens, np.int32))
    assert (r.K[:, :TINY.tokens] == 0x80).any()
    before = r.K.copy()
    assert r.delta_rotate(TO_OLDEST) == 0          # the window already starts at position 0
    assert np.array_equal(r.K, before)
    r.delta_rotate(0)
    assert np.array_equal(r.K, before)
    r.delta_rotate(3)
    assert not np.array_equal(r.K, before)


def test_delta_to_oldest_reads_the_oldest_slot():
    frames = tiny_session()
    r = _ring()
    r.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    for f in range(7):
        r.write(_f(frames[f][1]), _f(frames[f][2]))
    # 84 tokens written into 48 slots: window holds positions 36..83
    assert r.slot_pos.min() == 36 and r.slot_pos.max() == 83
    d = r.delta_rotate(TO_OLDEST)
    assert d == 36
    assert sorted(r.slot_pos.tolist()) == list(range(48))
    assert r.next_pos == 48


def test_delta_rotation_matches_reference_rotation_within_format_error():
    frames = tiny_session()
    r = _ring()
    r.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    ks = []
    for f in range(7):
        r.write(_f(frames[f][1]), _f(frames[f][2]))
        ks.append(_f(frames[f][1]))
    cached = e4m3.decode(r.K).copy()                    # scaled units, [H, C, d]
    pos_before = r.slot_pos.copy()
    delta = r.delta_rotate(TO_OLDEST)
    after = e4m3.decode(r.K)
    th = r.table.theta
    # (i) float64 re-rotation of the same cached values by -delta
    rot = rotate_f64(cached.transpose(1, 0, 2), np.full(r.C, -delta), th).transpose(1, 0, 2)
    inr = np.abs(rot) <= 448.0          # a rotated pair can leave the range: saturates
    assert np.all((np.abs(after - rot) <= e4m3.half_ulp(rot) + 1e-5 * (np.abs(rot) + 1))[inr])
    assert np.all(np.abs(after[~inr]) == 448.0)
    frac_equal = np.mean(e4m3.encode(np.clip(rot, -448, 448)) == r.K)
    assert frac_equal > 0.99
    # (ii) from-scratch quantisation of the original keys at p - delta
    k_all = np.concatenate(ks)[-r.C:]                     # time order, last 48 tokens
    order = np.argsort(pos_before)                        # slots sorted by time
    exact = rotate_f64(k_all.astype(np.float64), pos_before[order] - delta, th)
    y = exact / r.scale_k.astype(np.float64)[None, :, None]
    got = after[:, order, :].transpose(1, 0, 2)
    # the cached pair (a, b) erred by at most half an ulp of each component at
    # write time; rotating keeps that error vector's length, then the reset
    # rounds once more
    y0 = rotate_f64(k_all.astype(np.float64), pos_before[order], th) / r.scale_k.astype(np.float64)[None, :, None]
    pair_max = np.maximum(np.abs(y0[..., 0::2]), np.abs(y0[..., 1::2])).repeat(2, axis=-1)
    bound = np.sqrt(2) * e4m3.half_ulp(pair_max) + e4m3.half_ulp(y) + 1e-5 * (np.abs(y) + 1)
    # keep pairs whose norm (kept by every rotation) leaves both components in
    # range at write time and after the reset, with room for the FP8 error
    pair_norm = np.sqrt(y[..., 0::2] ** 2 + y[..., 1::2] ** 2).repeat(2, axis=-1)
    keep = pair_norm <= 420.0
    assert keep.mean() > 0.9
    assert np.all((np.abs(got - y) <= bound)[keep])


def test_attention_invariant_under_reset_up_to_format_error():
    frames = tiny_session()
    r = _ring()
    r.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    for f in range(7):
        r.write(_f(frames[f][1]), _f(frames[f][2]))
    q = _f(frames[7][0])
    qpos = np.arange(84, 96)
    o_before = attention_exact(r, q, qpos)
    delta = r.delta_rotate(TO_OLDEST)
    o_after = attention_exact(r, q, qpos - delta)
    v_rms = np.sqrt(np.mean(_f(frames[0][2]).astype(np.float64) ** 2))
    err = np.abs(o_before - o_after).max()
    assert err < 0.05 * v_rms          # only the requantisation of the keys differs
    assert err > 0                     # ... and it does differ a little
