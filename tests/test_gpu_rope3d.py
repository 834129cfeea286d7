"""3-D RoPE variant on the GPU against the oracle, bit for bit (codes,
scales, slot positions, ring state), with position resets that turn only
the temporal pairs, attention within tolerance, the batched write and reset
against the single-ring calls, and the host-side checks of the variant."""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring, TO_OLDEST
from oracle.attention import attention_exact
from workloads import PROD, TINY, prod_session, tiny_session

from _ringcheck import MAX_ABS, MEAN_ABS, assert_ring_equal, attn_errors, dev, export_np, f

pytestmark = pytest.mark.gpu

TINY_SEC = (8, 8)       # of 32 pairs: 8 temporal, 8 row, 16 column
PROD_SEC = (16, 24)     # of 64 pairs: 16 temporal, 24 row, 24 column


def _pair(shape, sec, prefix=0, **kw):
    ring = kv.KvRing(shape.heads, shape.head_dim, shape.capacity, max(shape.tokens, shape.queries),
                     shape.max_position, shape.rope_base, pinned_prefix=prefix, rope3d=sec, **kw)
    orc = Ring(shape.heads, shape.head_dim, shape.capacity, shape.max_position, shape.rope_base,
               prefix=prefix, rope3d=sec)
    return ring, orc


def _pos3(frame_idx, n, width):
    t = np.arange(n)
    return np.stack([np.full(n, frame_idx), t // width, t % width], axis=1).astype(np.int32)


def _d(p):
    return torch.from_numpy(np.ascontiguousarray(p)).cuda()


@pytest.mark.parametrize("prefix", [0, 10])
def test_tiny_3d_session_bit_exact_with_resets_and_attention(prefix):
    frames = tiny_session()
    ring, orc = _pair(TINY, TINY_SEC, prefix)
    p0 = _pos3(0, TINY.tokens, 4)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]), _d(p0))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]), p0)
    for i, (q, k, v) in enumerate(frames):
        if i in (5, 8):
            ring.delta_rotate(kv.TO_OLDEST)
            orc.delta_rotate(TO_OLDEST)
            assert_ring_equal(ring, orc, f"after reset before frame {i}")
        # frame index: one past the newest cached frame (resets lower them all)
        p = _pos3(int(orc.slot_pos.max()) + 1 if orc.n_valid else 0, TINY.tokens, 4)
        ring.write(dev(k), dev(v), _d(p))
        orc.write(f(k), f(v), p)
        assert_ring_equal(ring, orc, f"after write {i}")
        out = ring.attention(dev(q), qpos=_d(p))
        torch.cuda.synchronize()
        mx, mn = attn_errors(out.cpu().numpy(), attention_exact(orc, f(q), p))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, mx, mn)


def test_production_3d_wrap_reset_and_attention():
    sk, sv, frames = prod_session(frames=9)
    ring, orc = _pair(PROD, PROD_SEC, max_kv_splits=16)
    pos = [_pos3(i, PROD.tokens, 29) for i in range(9)]
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]), _d(pos[0]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]), pos[0])
    for i in range(8):                        # 6,056 tokens in 5,788 slots: wraps
        ring.write(dev(frames[i][1]), dev(frames[i][2]), _d(pos[i]))
        orc.write(f(frames[i][1]), f(frames[i][2]), pos[i])
    assert_ring_equal(ring, orc, "after 8 frames")
    ring.delta_rotate(kv.TO_OLDEST)
    assert orc.delta_rotate(TO_OLDEST) == 0   # frame 0 still has slots: the window starts at frame 0
    ring.delta_rotate(1)
    orc.delta_rotate(1)
    assert_ring_equal(ring, orc, "after resets")
    p8 = pos[8].copy()
    p8[:, 0] = 7
    ring.write(dev(frames[8][1]), dev(frames[8][2]), _d(p8))
    orc.write(f(frames[8][1]), f(frames[8][2]), p8)
    assert_ring_equal(ring, orc, "after the next frame")
    out = ring.attention(dev(frames[8][0]), qpos=_d(p8))
    torch.cuda.synchronize()
    rows = np.arange(0, PROD.queries, 12)
    ref = attention_exact(orc, f(frames[8][0][rows]), p8[rows])
    mx, mn = attn_errors(out.cpu().numpy()[rows], ref)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_batched_3d_write_and_reset_equal_single_ring_calls():
    frames = tiny_session()
    many = [_pair(TINY, TINY_SEC)[0] for _ in range(3)]
    single = [_pair(TINY, TINY_SEC)[0] for _ in range(3)]
    p0 = _d(_pos3(0, TINY.tokens, 4))
    for r in many + single:
        r.calibrate(dev(frames[0][1]), dev(frames[0][2]), p0)
    for i in range(7):
        ks = [dev(frames[(i + j) % 10][1]) for j in range(3)]
        vs = [dev(frames[(i + j) % 10][2]) for j in range(3)]
        ps = [_d(_pos3(i + j, TINY.tokens, 4)) for j in range(3)]
        kv.write_frames_many(many, ks, vs, ps)
        for j in range(3):
            single[j].write(ks[j], vs[j], ps[j])
    kv.delta_rotate_many(many, kv.TO_OLDEST)
    for r in single:
        r.delta_rotate(kv.TO_OLDEST)
    for a, b in zip(many, single):
        ea, eb = export_np(a), export_np(b)
        for key in ("k", "v", "slot_pos", "state"):
            assert np.array_equal(ea[key], eb[key]), key


def test_3d_positions_required():
    frames = tiny_session()
    ring, _ = _pair(TINY, TINY_SEC)
    with pytest.raises(ValueError):
        ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    st = kv.lib().kvring_write_frame(ring.handle, dev(frames[0][1]).data_ptr(), dev(frames[0][2]).data_ptr(),
                                     None, TINY.tokens, None)
    assert st == 1                            # INVALID_ARG: no positions given
