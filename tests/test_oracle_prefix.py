"""Pins for the oracle's pinned-prefix variant of the ring.

The reading (the pages give 5,788 = 7 x 757 + 489 slots and do not say
whether a part of the cache is never evicted): the first P slots keep the
first P tokens ever written; later tokens cycle over the other C - P slots;
a position reset rotates only those rolling slots and, by default, puts the
oldest rolling position right after the prefix.

Checked against: a token-by-token simulation of slot assignment with an
explicit cursor (no modular formula), the brute-force window (the first P
tokens plus the last C - P tokens in time order, each quantised at its own
position), the prefix bytes staying unchanged through writes and resets, and
attention over the rolling slots being invariant under a reset when the
queries move with the keys.
"""
import numpy as np
import pytest

from oracle import e4m3, Ring, INT32_MIN, TO_OLDEST
from oracle.attention import attention_exact, softmax_attention_f64
from oracle.rope import rotate_f64
from workloads import TINY, f32_from_bf16, tiny_session

P = 10


def _ring(prefix=P):
    return Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position, TINY.rope_base, prefix=prefix)


def _f(x):
    return f32_from_bf16(x)


def _cursor_slots(sizes, C, prefix):
    """Slot of every token, by moving a cursor one token at a time: prefix
    slots in order first, then around the rolling slots, back to slot
    ``prefix`` after slot C - 1."""
    out, cur = [], 0
    for n in sizes:
        s = []
        for _ in range(n):
            s.append(cur)
            cur += 1
            if cur == C:
                cur = prefix
        out.append(np.array(s))
    return out


def test_slots_follow_a_cursor_over_prefix_then_rolling_slots():
    r = _ring()
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, TINY.heads, TINY.head_dim)).astype(np.float32)
    r.calibrate(k, k)
    sizes = [4, 4, 12, 38, 1, 37, 20, 38, 5]
    expect = _cursor_slots(sizes, TINY.capacity, P)
    total = 0
    for n, e in zip(sizes, expect):
        got = r.write(k.repeat(n, 0), k.repeat(n, 0))
        assert np.array_equal(got, e)
        total += n
        assert r.n_valid == min(total, TINY.capacity)
        assert r.next_pos == total
    with pytest.raises(ValueError):          # a frame larger than the rolling part
        r.write(k.repeat(39, 0), k.repeat(39, 0))


def test_prefix_must_leave_rolling_slots():
    with pytest.raises(ValueError):
        _ring(prefix=TINY.capacity)
    with pytest.raises(ValueError):
        _ring(prefix=-1)


def _session(ring, frames, upto):
    ring.calibrate(_f(frames[0][1]), _f(frames[0][2]))
    hist = []
    for f in range(upto):
        pos = ring.next_pos + np.arange(TINY.tokens)
        hist.append((ring.quantise_keys(_f(frames[f][1]), pos), ring.quantise_values(_f(frames[f][2])), pos))
        ring.write(_f(frames[f][1]), _f(frames[f][2]))
    return hist


def test_window_is_first_prefix_tokens_plus_latest_tokens():
    frames = tiny_session()
    r = _ring()
    hist = _session(r, frames, 10)           # 120 tokens: the rolling part wrapped twice
    kc = np.concatenate([h[0] for h in hist])
    vc = np.concatenate([h[1] for h in hist])
    pos = np.concatenate([h[2] for h in hist])
    keep = np.r_[np.arange(P), np.arange(len(pos) - (TINY.capacity - P), len(pos))]
    by_pos = {int(p): i for i, p in enumerate(pos)}
    valid = np.nonzero(r.slot_pos != INT32_MIN)[0]
    assert sorted(int(p) for p in r.slot_pos[valid]) == sorted(int(pos[i]) for i in keep)
    for s in valid:
        i = by_pos[int(r.slot_pos[s])]
        assert np.array_equal(r.K[:, s, :], kc[i]) and np.array_equal(r.V[:, s, :], vc[i])
    # attention over the ring equals attention over the brute-force window
    q = _f(frames[9][0])
    qpos = pos[-TINY.queries:]
    k = e4m3.decode(kc[keep]).transpose(1, 0, 2) * r.scale_k.astype(np.float64)[:, None, None]
    v = e4m3.decode(vc[keep]).transpose(1, 0, 2) * r.scale_v.astype(np.float64)[:, None, None]
    qt = rotate_f64(q.astype(np.float64), qpos, r.table.theta)
    want = softmax_attention_f64(qt, k, v)
    assert np.abs(attention_exact(r, q, qpos) - want).max() <= 1e-12


def test_prefix_bytes_never_change_through_writes_and_resets():
    frames = tiny_session()
    r = _ring()
    _session(r, frames, 1)                   # 12 tokens >= P: prefix full
    K0, V0, p0 = r.K[:, :P].copy(), r.V[:, :P].copy(), r.slot_pos[:P].copy()
    for f in range(1, 10):
        if f == 7:
            r.delta_rotate(TO_OLDEST)
        r.write(_f(frames[f][1]), _f(frames[f][2]))
        assert np.array_equal(r.K[:, :P], K0) and np.array_equal(r.V[:, :P], V0)
        assert np.array_equal(r.slot_pos[:P], p0)
    r.delta_rotate(5)
    assert np.array_equal(r.K[:, :P], K0) and np.array_equal(r.slot_pos[:P], p0)


def test_default_reset_puts_the_window_right_after_the_prefix():
    frames = tiny_session()
    r = _ring()
    _session(r, frames, 7)                   # 84 tokens, wrapped
    prefix_end = int(r.slot_pos[P - 1]) + 1
    rolling = r.slot_pos[P:r.n_valid].copy()
    d = r.delta_rotate(TO_OLDEST)
    assert d == int(rolling.min()) - prefix_end
    assert int(r.slot_pos[P:r.n_valid].min()) == prefix_end
    assert np.array_equal(r.slot_pos[P:r.n_valid], rolling - d)
    assert r.next_pos == 84 - d


def test_attention_over_rolling_slots_invariant_under_reset():
    """Keys and queries move together, so only the requantisation of the
    rotated keys changes the rolling part's attention."""
    frames = tiny_session()
    r = _ring()
    _session(r, frames, 7)
    q = _f(frames[7][0])
    qpos = np.arange(84, 96)

    def rolling_attention(ring, qp):
        sl = np.arange(P, ring.n_valid)
        k = e4m3.decode(ring.K[:, sl]) * ring.scale_k.astype(np.float64)[:, None, None]
        v = e4m3.decode(ring.V[:, sl]) * ring.scale_v.astype(np.float64)[:, None, None]
        qt = rotate_f64(q.astype(np.float64), qp, ring.table.theta)
        return softmax_attention_f64(qt, k, v)

    before = rolling_attention(r, qpos)
    d = r.delta_rotate(TO_OLDEST)
    after = rolling_attention(r, qpos - d)
    v_rms = np.sqrt(np.mean(_f(frames[0][2]).astype(np.float64) ** 2))
    err = np.abs(before - after).max()
    assert 0 < err < 0.05 * v_rms


def test_zero_prefix_is_the_plain_ring():
    frames = tiny_session()
    a, b = _ring(prefix=0), Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position, TINY.rope_base)
    for ring in (a, b):
        _session(ring, frames, 7)
        ring.delta_rotate(TO_OLDEST)
        ring.write(_f(frames[7][1]), _f(frames[7][2]))
    assert np.array_equal(a.K, b.K) and np.array_equal(a.slot_pos, b.slot_pos) and a.head == b.head
