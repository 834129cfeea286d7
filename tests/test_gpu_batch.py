"""Batched write and delta rotation over several rings in one launch.

Each ring must end exactly as the oracle says (codes, scales, slot map,
state) and as the single-ring entry points leave it; argument errors are
refused on the host before anything is launched.
"""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring, TO_OLDEST
from workloads import PROD, TINY, frame, prod_session

from _ringcheck import assert_ring_equal, dev, export_np, f, make_pair

pytestmark = pytest.mark.gpu


def test_batched_tiny_sessions_bit_exact_with_resets():
    """Five tiny rings with their own inputs; ring 1 takes explicit positions."""
    m = 5
    rngs = [np.random.default_rng(40 + i) for i in range(m)]
    pairs = [make_pair(TINY, Ring) for _ in range(m)]
    rings = [p[0] for p in pairs]
    orcs = [p[1] for p in pairs]
    for i in range(m):
        _, k, v = frame(rngs[i], TINY, TINY.tokens)
        rings[i].calibrate(dev(k), dev(v))
        orcs[i].calibrate(f(k), f(v))
    for step in range(10):
        ks, vs, poss = [], [], []
        for i in range(m):
            _, k, v = frame(rngs[i], TINY, TINY.tokens)
            ks.append(dev(k))
            vs.append(dev(v))
            if i == 1:
                p = np.arange(TINY.tokens, dtype=np.int32) * 3 + step
                poss.append(torch.from_numpy(p).cuda())
                orcs[i].write(f(k), f(v), p)
            else:
                poss.append(None)
                orcs[i].write(f(k), f(v))
        kv.write_frames_many(rings, ks, vs, poss)
        for i in range(m):
            assert_ring_equal(rings[i], orcs[i], f"ring {i} after batched write {step}")
        if step == 6:
            kv.delta_rotate_many(rings, kv.TO_OLDEST)
            for i in range(m):
                orcs[i].delta_rotate(TO_OLDEST)
                assert_ring_equal(rings[i], orcs[i], f"ring {i} after batched reset")
        if step == 8:
            kv.delta_rotate_many(rings, 5)
            for i in range(m):
                orcs[i].delta_rotate(5)
                assert_ring_equal(rings[i], orcs[i], f"ring {i} after batched delta 5")


def test_batched_equals_single_calls_on_production_shape():
    """Three production-shaped rings written and reset in batches end byte for
    byte as three rings driven one call at a time."""
    m = 3
    sessions = [prod_session(seed=60 + i, frames=9)[2] for i in range(m)]
    single = [kv.KvRing(PROD.heads, PROD.head_dim, PROD.capacity, PROD.tokens, PROD.max_position) for _ in range(m)]
    batch = [kv.KvRing(PROD.heads, PROD.head_dim, PROD.capacity, PROD.tokens, PROD.max_position) for _ in range(m)]
    for i in range(m):
        k0, v0 = dev(sessions[i][0][1]), dev(sessions[i][0][2])
        single[i].calibrate(k0, v0)
        batch[i].calibrate(k0, v0)
    for step in range(9):
        ks = [dev(sessions[i][step][1]) for i in range(m)]
        vs = [dev(sessions[i][step][2]) for i in range(m)]
        for i in range(m):
            single[i].write(ks[i], vs[i])
        kv.write_frames_many(batch, ks, vs)
        if step == 7:
            for i in range(m):
                single[i].delta_rotate(kv.TO_OLDEST)
            kv.delta_rotate_many(batch, kv.TO_OLDEST)
    for i in range(m):
        a, b = export_np(single[i]), export_np(batch[i])
        for key in ("k", "v", "slot_pos", "scales", "state"):
            assert np.array_equal(a[key], b[key]), (i, key)


def test_batched_argument_errors():
    a = kv.KvRing(2, 64, 48, 12, 256)
    b = kv.KvRing(2, 64, 48, 12, 256)
    c = kv.KvRing(2, 64, 96, 12, 256)          # another capacity
    u = kv.KvRing(2, 64, 48, 12, 256)          # never calibrated
    x = torch.zeros((12, 2, 64), dtype=torch.bfloat16, device="cuda")
    for r in (a, b, c):
        r.calibrate(x, x)

    def status(fn):
        with pytest.raises(kv.KvRingError) as e:
            fn()
        return e.value.status

    assert status(lambda: kv.write_frames_many([a, c], [x, x], [x, x])) == 1      # shapes differ
    assert status(lambda: kv.write_frames_many([a, a], [x, x], [x, x])) == 1      # repeated ring
    assert status(lambda: kv.write_frames_many([a, u], [x, x], [x, x])) == 2      # not calibrated
    big = torch.zeros((60, 2, 64), dtype=torch.bfloat16, device="cuda")
    assert status(lambda: kv.write_frames_many([a, b], [big, big], [big, big])) == 3   # n > capacity
    assert status(lambda: kv.delta_rotate_many([a, c], 0)) == 1
    assert status(lambda: kv.delta_rotate_many([a, b], 256)) == 1                 # >= max_position
    L = kv.lib()
    assert L.kvring_delta_rotate_many(None, 1, 0, None) == 1
    assert L.kvring_delta_rotate_many(kv._ptr_array([a.handle]), 0, 0, None) == 1
    torch.cuda.synchronize()
    st = export_np(a)["state"]
    assert st[kv.STATE["n_valid"]] == 0      # nothing was launched on a refused call
