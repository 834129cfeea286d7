"""Pinned-prefix variant on the GPU against the oracle, bit for bit (codes,
scales, slot positions, ring state), with position resets, attention within
tolerance, the batched write and reset against the single-ring calls, and
the host-side limits of the variant."""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring, TO_OLDEST
from oracle.attention import attention_exact
from workloads import PROD, TINY, prod_session, tiny_session

from _ringcheck import MAX_ABS, MEAN_ABS, assert_ring_equal, attn_errors, dev, export_np, f

pytestmark = pytest.mark.gpu

TINY_P = 10
PROD_P = 489   # 5,788 = 7 x 757 + 489


def _pair(shape, prefix, **kw):
    ring = kv.KvRing(shape.heads, shape.head_dim, shape.capacity, max(shape.tokens, shape.queries),
                     shape.max_position, shape.rope_base, pinned_prefix=prefix, **kw)
    orc = Ring(shape.heads, shape.head_dim, shape.capacity, shape.max_position, shape.rope_base, prefix=prefix)
    return ring, orc


def test_tiny_prefix_session_bit_exact_with_resets_and_attention():
    frames = tiny_session()
    ring, orc = _pair(TINY, TINY_P)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    for i, (q, k, v) in enumerate(frames):
        if i in (5, 8):
            ring.delta_rotate(kv.TO_OLDEST)
            assert orc.delta_rotate(TO_OLDEST) > 0
            assert_ring_equal(ring, orc, f"after reset before frame {i}")
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
        assert_ring_equal(ring, orc, f"after write {i}")
        out = ring.attention(dev(q))
        torch.cuda.synchronize()
        mx, mn = attn_errors(out.cpu().numpy(), attention_exact(orc, f(q)))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, mx, mn)
    ring.delta_rotate(3)                      # an explicit delta as well
    orc.delta_rotate(3)
    assert_ring_equal(ring, orc, "after an explicit delta")


def test_production_prefix_wrap_reset_and_attention():
    sk, sv, frames = prod_session(frames=9)
    ring, orc = _pair(PROD, PROD_P, max_kv_splits=16)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    for i in range(8):                        # 6,056 tokens: the rolling part wraps
        ring.write(dev(frames[i][1]), dev(frames[i][2]))
        orc.write(f(frames[i][1]), f(frames[i][2]))
    assert_ring_equal(ring, orc, "after 8 frames")
    ring.delta_rotate(kv.TO_OLDEST)
    assert orc.delta_rotate(TO_OLDEST) > 0
    assert_ring_equal(ring, orc, "after the reset")
    ring.write(dev(frames[8][1]), dev(frames[8][2]))
    orc.write(f(frames[8][1]), f(frames[8][2]))
    assert_ring_equal(ring, orc, "after the next frame")
    out = ring.attention(dev(frames[8][0]))
    torch.cuda.synchronize()
    rows = np.arange(0, PROD.queries, 12)
    ref = attention_exact(orc, f(frames[8][0][rows]), orc.next_pos - PROD.queries + rows)
    mx, mn = attn_errors(out.cpu().numpy()[rows], ref)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_batched_prefix_write_and_reset_equal_single_ring_calls():
    frames = tiny_session()
    many = [_pair(TINY, TINY_P)[0] for _ in range(3)]
    single = [_pair(TINY, TINY_P)[0] for _ in range(3)]
    for r in many + single:
        r.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    for i in range(7):
        ks = [dev(frames[(i + j) % 10][1]) for j in range(3)]
        vs = [dev(frames[(i + j) % 10][2]) for j in range(3)]
        kv.write_frames_many(many, ks, vs)
        for j in range(3):
            single[j].write(ks[j], vs[j])
    kv.delta_rotate_many(many, kv.TO_OLDEST)
    for r in single:
        r.delta_rotate(kv.TO_OLDEST)
    for a, b in zip(many, single):
        ea, eb = export_np(a), export_np(b)
        for key in ("k", "v", "slot_pos", "state"):
            assert np.array_equal(ea[key], eb[key]), key


def test_prefix_limits_on_the_host():
    frames = tiny_session()
    ring, _ = _pair(TINY, 40)                 # 8 rolling slots
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    with pytest.raises(kv.KvRingError) as e:
        ring.write(dev(frames[0][1]), dev(frames[0][2]))   # 12 tokens > 8
    assert e.value.status == 3
    plain = kv.KvRing(TINY.heads, TINY.head_dim, TINY.capacity, TINY.tokens, TINY.max_position)
    with pytest.raises(kv.KvRingError):
        kv.write_frames_many([ring, plain], [dev(frames[0][1])] * 2, [dev(frames[0][2])] * 2)
    win = [torch.zeros((TINY.capacity, TINY.heads, TINY.head_dim), dtype=torch.bfloat16, device="cuda")
           for _ in range(4)]
    with pytest.raises(kv.KvRingError) as e:  # the original upkeep had no prefix
        kv.kvring_legacy_upkeep(ring.handle, *win, dev(frames[0][1][:8]), dev(frames[0][2][:8]), 8, None)
    assert e.value.status == 4
