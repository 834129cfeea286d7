"""Cache kernels (calibration, write, delta rotation) against the oracle, bit
for bit: key and value codes, scales and their reciprocals, the slot-to-
position map and the ring state, on the tiny and production-shaped
workloads, plus varied frame sizes, explicit positions and host-side
argument errors."""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring, TO_OLDEST
from oracle.attention import attention_exact
from workloads import PROD, TINY, RingShape, frame, prod_session, tiny_session

from _ringcheck import MAX_ABS, MEAN_ABS, assert_ring_equal, attn_errors, dev, f, make_pair

pytestmark = pytest.mark.gpu


def test_tiny_session_bit_exact_with_reset_and_attention():
    frames = tiny_session()
    ring, orc = make_pair(TINY, Ring)
    q0, k0, v0 = frames[0]
    ring.calibrate(dev(k0), dev(v0))
    orc.calibrate(f(k0), f(v0))
    assert_ring_equal(ring, orc, "after calibration")
    for i, (q, k, v) in enumerate(frames):
        if i == 7:
            ring.delta_rotate(kv.TO_OLDEST)
            assert orc.delta_rotate(TO_OLDEST) == 36
            assert_ring_equal(ring, orc, "after reset")
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
        assert_ring_equal(ring, orc, f"after write {i}")
        out = ring.attention(dev(q))
        torch.cuda.synchronize()
        mx, mn = attn_errors(out.cpu().numpy(), attention_exact(orc, f(q)))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, mx, mn)


@pytest.fixture(scope="module")
def prod_pair():
    sk, sv, frames = prod_session(frames=9)
    ring, orc = make_pair(PROD, Ring, max_kv_splits=16)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    return ring, orc, frames


def test_production_writes_wrap_bit_exact(prod_pair):
    ring, orc, frames = prod_pair
    for i in range(9):            # 6,813 tokens into 5,788 slots: wraps mid-frame
        ring.write(dev(frames[i][1]), dev(frames[i][2]))
        orc.write(f(frames[i][1]), f(frames[i][2]))
        if i in (0, 7, 8):
            assert_ring_equal(ring, orc, f"write {i}")
    assert orc.total > PROD.capacity


def test_production_attention_within_tolerance(prod_pair):
    ring, orc, frames = prod_pair
    q = frames[8][0]
    out = ring.attention(dev(q))
    torch.cuda.synchronize()
    ref = attention_exact(orc, f(q))
    mx, mn = attn_errors(out.cpu().numpy(), ref)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_production_delta_rotation_bit_exact(prod_pair):
    ring, orc, frames = prod_pair
    ring.delta_rotate(kv.TO_OLDEST)
    d = orc.delta_rotate(TO_OLDEST)
    assert d > 0
    e = assert_ring_equal(ring, orc, "reset")
    assert e["state"][kv.STATE["last_delta"]] == d
    ring.delta_rotate(0)          # explicit zero delta: identity
    assert_ring_equal(ring, orc, "zero delta")


@pytest.mark.parametrize("first", [1, 127, 128, 129, 757, 5788])
def test_varied_first_write_sizes(first):
    rng = np.random.default_rng(first)
    shape = RingShape(heads=4, head_dim=128, capacity=5788, tokens=first, queries=129,
                      max_position=20000)
    ring, orc = make_pair(shape, Ring, max_tokens=5788)
    q, k, v = frame(rng, shape, first)
    ring.calibrate(dev(k), dev(v))
    orc.calibrate(f(k), f(v))
    ring.write(dev(k), dev(v))
    orc.write(f(k), f(v))
    for n in (757, 1000):          # later frames of other sizes, wrapping
        _, k2, v2 = frame(rng, shape, n)
        ring.write(dev(k2), dev(v2))
        orc.write(f(k2), f(v2))
    assert_ring_equal(ring, orc, f"first={first}")
    for nq in (1, 129):
        qq, _, _ = frame(rng, shape, nq)
        out = ring.attention(dev(qq))
        torch.cuda.synchronize()
        mx, mn = attn_errors(out.cpu().numpy(), attention_exact(orc, f(qq)))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (first, nq, mx, mn)


def test_head_dim_64_and_explicit_positions():
    rng = np.random.default_rng(5)
    shape = RingShape(heads=3, head_dim=64, capacity=300, tokens=100, queries=100, max_position=5000)
    ring, orc = make_pair(shape, Ring)
    pos0 = rng.integers(0, 4000, 100).astype(np.int32)
    q, k, v = frame(rng, shape, 100)
    ring.calibrate(dev(k), dev(v), torch.from_numpy(pos0).cuda())
    orc.calibrate(f(k), f(v), pos0)
    for i in range(5):
        pos = rng.integers(0, 4000, 100).astype(np.int32)
        q, k, v = frame(rng, shape, 100)
        ring.write(dev(k), dev(v), torch.from_numpy(pos).cuda())
        orc.write(f(k), f(v), pos)
    assert_ring_equal(ring, orc, "explicit positions")
    qpos = rng.integers(0, 4000, 100).astype(np.int32)
    out = ring.attention(dev(q), torch.from_numpy(qpos).cuda())
    torch.cuda.synchronize()
    mx, mn = attn_errors(out.cpu().numpy(), attention_exact(orc, f(q), qpos))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_zero_head_calibrates_to_unit_scale():
    shape = RingShape(heads=2, head_dim=64, capacity=64, tokens=8, queries=8, max_position=64)
    ring, orc = make_pair(shape, Ring)
    rng = np.random.default_rng(1)
    q, k, v = frame(rng, shape, 8)
    k[:, 1, :] = 0                # head 1 of K all zero
    ring.calibrate(dev(k), dev(v))
    orc.calibrate(f(k), f(v))
    ring.write(dev(k), dev(v))
    orc.write(f(k), f(v))
    e = assert_ring_equal(ring, orc, "zero head")
    assert e["scales"][1] == 1.0


def test_host_argument_errors():
    ring = kv.KvRing(2, 64, 48, 12, 256)
    k = torch.zeros((12, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kv.KvRingError) as ei:
        ring.write(k, k)
    assert ei.value.status == 2                       # not calibrated
    with pytest.raises(kv.KvRingError) as ei:
        ring.attention(k)
    assert ei.value.status == 2
    ring.calibrate(k, k)
    big = torch.zeros((13, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kv.KvRingError) as ei:
        ring.write(big, big)
    assert ei.value.status == 3                       # more than max_tokens
    with pytest.raises(kv.KvRingError) as ei:
        ring.delta_rotate(256)
    assert ei.value.status == 1                       # outside the RoPE table
    with pytest.raises(ValueError):
        ring.write(k.float(), k)                      # wrong dtype caught in the binding


def test_device_position_out_of_table_sets_error_word():
    ring = kv.KvRing(2, 64, 48, 12, 256)
    k = torch.ones((12, 2, 64), dtype=torch.bfloat16, device="cuda")
    ring.calibrate(k, k)
    pos = torch.arange(12, dtype=torch.int32, device="cuda")
    pos[3] = 999
    ring.write(k, k, pos)
    st = ring.export()["state"].cpu().numpy()
    assert st[kv.STATE["error"]] & kv.DEVERR_POSITION


def test_write_floor_leaves_the_ring_unchanged():
    """The measurement kernel for the write's fixed cost (the write's grid,
    launch, wait, state read, ticket and state publication with no data)
    leaves codes, positions and state exactly as they were, before and after
    the ring has wrapped, and a write after it still matches the oracle."""
    frames = tiny_session()
    ring, orc = make_pair(TINY, Ring)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    for i, (q, k, v) in enumerate(frames):
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
        if i in (1, 6):
            for _ in range(3):
                ring.write_floor(TINY.tokens)
            assert_ring_equal(ring, orc, f"after floor launches at frame {i}")
    assert_ring_equal(ring, orc, "after the last write")
    with pytest.raises(kv.KvRingError):
        ring.write_floor(TINY.capacity + 1)


@pytest.mark.parametrize("prefix", [0, 10])
def test_writes_on_alternating_rings_match_the_oracle(prefix):
    """Writes and resets whose preceding kernel touches another ring (the host
    then lets the whole call -- state read, codes, ticket, publication --
    happen before its wait for that kernel), mixed with writes that follow a
    kernel on their own ring, and attention calls, eager and captured in a
    CUDA graph, with and without a pinned prefix: every ring equals the
    oracle byte for byte and every attention meets the bar."""
    frames = tiny_session(frames=12)
    pairs = [(kv.KvRing(TINY.heads, TINY.head_dim, TINY.capacity, TINY.tokens, TINY.max_position,
                        TINY.rope_base, pinned_prefix=prefix),
              Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position, TINY.rope_base, prefix=prefix))
             for _ in range(2)]
    for ring, orc in pairs:
        ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
        orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    dframes = [tuple(dev(x) for x in fr) for fr in frames]
    outs = [torch.empty((TINY.queries, TINY.heads, TINY.head_dim), device="cuda") for _ in pairs]
    s = torch.cuda.Stream()

    def step(i, eager_check):
        q, k, v = dframes[i]
        for j, (ring, orc) in enumerate(pairs):
            if i == 9 and j == 1:
                ring.delta_rotate(kv.TO_OLDEST, stream=s)     # a reset on one ring only
                if eager_check:
                    orc.delta_rotate(TO_OLDEST)
            ring.write(k, v, stream=s)
            if i % 3 == 2:
                ring.write(k, v, stream=s)                    # right after a write on the same ring
            ring.attention(q, out=outs[j], stream=s)

    for i in range(6):
        with torch.cuda.stream(s):
            step(i, True)
        s.synchronize()
        for j, (ring, orc) in enumerate(pairs):
            orc.write(f(frames[i][1]), f(frames[i][2]))
            if i % 3 == 2:
                orc.write(f(frames[i][1]), f(frames[i][2]))
            assert_ring_equal(ring, orc, f"eager step {i}, ring {j}")
            mx, mn = attn_errors(outs[j].cpu().numpy(), attention_exact(orc, f(frames[i][0])))
            assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, j, mx, mn)
    # steps 6-11 captured once (the reset before step 9 on ring 1 included) and replayed
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(6, 12):
            step(i, False)
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    for i in range(6, 12):
        for j, (ring, orc) in enumerate(pairs):
            if i == 9 and j == 1:
                orc.delta_rotate(TO_OLDEST)
            orc.write(f(frames[i][1]), f(frames[i][2]))
            if i % 3 == 2:
                orc.write(f(frames[i][1]), f(frames[i][2]))
    for j, (ring, orc) in enumerate(pairs):
        assert_ring_equal(ring, orc, f"after the graph, ring {j}")
        mx, mn = attn_errors(outs[j].cpu().numpy(), attention_exact(orc, f(frames[11][0])))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (j, mx, mn)
