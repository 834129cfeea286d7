"""Pins of the legacy-upkeep oracle (the path the ring replaced).

* window bookkeeping against token identities: slot i holds token
  total - fill + i, in time order, across fills and wrap-arounds;
* with the ring's calibrated scales forced in, every token's key and value
  codes equal the ring oracle's codes for the same token (same position,
  same pinned RoPE, same conversion): two independently written models agree;
* with window scales, every head's largest key and value code is 448 (the
  window maximum maps to E4M3's maximum), and the scale is that maximum / 448.
"""
import numpy as np

from oracle import Ring, e4m3
from oracle.legacy import LegacyWindow
from oracle.rope import rotate_f64, theta
from workloads import TINY, frame, tiny_session, f32_from_bf16


def test_window_holds_the_last_tokens_in_time_order():
    H, d, C = 2, 64, 48
    w = LegacyWindow(H, d, C, 512)
    total = 0
    for n in (12, 12, 20, 7, 30, 48, 5):
        ids = np.arange(total, total + n, dtype=np.float32)
        k = np.broadcast_to(ids[:, None, None], (n, H, d)).copy()
        w.shift_in(k, -k)
        total += n
        fill = min(total, C)
        assert w.fill == fill and w.total == total and w.base() == total - fill
        want = np.arange(total - fill, total, dtype=np.float32)
        assert np.array_equal(w.k[:fill, 0, 0], want)
        assert np.array_equal(w.v[:fill, 1, 3], -want)


def test_codes_match_the_ring_oracle_token_by_token_with_the_same_scales():
    frames = tiny_session(frames=7)
    ring = Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position)
    ring.calibrate(f32_from_bf16(frames[0][1]), f32_from_bf16(frames[0][2]))
    w = LegacyWindow(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position)
    for _, k, v in frames:
        ring.write(f32_from_bf16(k), f32_from_bf16(v))
        w.shift_in(f32_from_bf16(k), f32_from_bf16(v))
        w.requantise(ring.scale_k, ring.scale_v)
        for i in range(w.fill):
            t = w.base() + i                     # the token in window slot i
            slot = t % TINY.capacity             # its ring slot (head starts at 0)
            assert ring.slot_pos[slot] == t == w.slot_pos[i]
            assert np.array_equal(w.K[:, i, :], ring.K[:, slot, :]), (t, i)
            assert np.array_equal(w.V[:, i, :], ring.V[:, slot, :]), (t, i)


def test_window_scales_map_each_heads_maximum_to_448():
    rng = np.random.default_rng(5)
    H, d, C = 3, 64, 40
    w = LegacyWindow(H, d, C, 1024)
    sig = np.array([0.3, 1.0, 7.0])
    for _ in range(5):
        _, k, v = frame(rng, TINY.__class__(heads=H, head_dim=d, capacity=C, tokens=16, queries=16,
                                            max_position=1024), 16, sig, sig[::-1])
        w.upkeep(f32_from_bf16(k), f32_from_bf16(v))
        for h in range(H):
            kc = e4m3.decode(w.K[h, :w.fill, :])
            vc = e4m3.decode(w.V[h, :w.fill, :])
            assert np.abs(kc).max() == 448.0 and np.abs(vc).max() == 448.0
        # the key scale is the rotated window's maximum over 448 (float64 RoPE
        # agrees with the pinned fp32 rotation to a few ulp)
        pos = w.base() + np.arange(w.fill)
        y = rotate_f64(w.k[:w.fill].astype(np.float64), pos, theta(d, 10000.0))
        amax = np.abs(y).max(axis=(0, 2))
        assert np.allclose(w.scale_k.astype(np.float64) * 448.0, amax, rtol=1e-6)
        assert np.allclose(w.scale_v.astype(np.float64) * 448.0, np.abs(w.v[:w.fill]).max(axis=(0, 2)), rtol=1e-6)
