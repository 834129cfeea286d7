"""The attention kernel's bounded waits, made to give up on purpose.

Every wait in the attention kernel has a wall-time limit; a wait that gives
up sets KVRING_DEVERR_TIMEOUT in the ring's error word, and the kernel drains
its in-flight copies and MMAs, frees its tensor memory and returns, so the
CUDA context stays usable.  The test support entry point
kvring_debug_set_attention_wait shortens the limit and makes the kernel's QK
issuer first wait on a barrier that nothing ever completes (a flag nothing
sets): no fault, trap or endless wait is involved, the abort comes only from
the limit running out.  One key/value split, so no cluster peers are
involved.
"""
import time

import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring
from oracle.attention import attention_exact
from workloads import RingShape, frame

from _ringcheck import MAX_ABS, MEAN_ABS, attn_errors, dev, f, make_pair

pytestmark = pytest.mark.gpu

SHAPE = RingShape(heads=2, head_dim=128, capacity=700, tokens=350, queries=200, max_position=2000)


def _loaded(seed):
    rng = np.random.default_rng(seed)
    ring, orc = make_pair(SHAPE, Ring, max_tokens=350, max_kv_splits=1)
    for i in range(3):                       # 1,050 tokens: six key/value tiles, wrapped
        q, k, v = frame(rng, SHAPE, 350)
        if i == 0:
            ring.calibrate(dev(k), dev(v))
            orc.calibrate(f(k), f(v))
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    q, _, _ = frame(rng, SHAPE, 200)
    return ring, orc, q


def test_wait_limit_is_checked_on_the_host():
    ring, _, _ = _loaded(30)
    L = kv.lib()
    assert L.kvring_debug_set_attention_wait(ring.handle, 10, 0) == 1            # below 1 us
    assert L.kvring_debug_set_attention_wait(ring.handle, 10 ** 11, 0) == 1      # above 60 s
    assert L.kvring_debug_set_attention_wait(ring.handle, 10 ** 6, 2) == 1       # stall is 0 or 1
    assert L.kvring_debug_set_attention_wait(None, 10 ** 6, 0) == 1
    assert L.kvring_debug_set_attention_wait(ring.handle, 10 ** 9, 0) == 0


def test_a_wait_that_gives_up_reports_timeout_and_leaves_the_context_usable():
    ring, orc, q = _loaded(31)
    ring.set_attention_wait(2_000_000, stall=True)          # 2 ms, then give up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(2):                                      # two aborted calls in a row
        ring.attention(dev(q))
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    err = ring.export()["state"][kv.STATE["error"]].item()
    assert err & kv.DEVERR_TIMEOUT, err
    assert elapsed < 2.0, elapsed                           # each call ended near its limit

    # normal calls again: on the same ring (its error word keeps the bit) and
    # on a fresh ring, both match the float64 reference
    ring.set_attention_wait()
    want = attention_exact(orc, f(q))
    mx, mn = attn_errors(ring.attention(dev(q)).cpu().numpy(), want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)
    fresh, orc2, q2 = _loaded(32)
    mx, mn = attn_errors(fresh.attention(dev(q2)).cpu().numpy(), attention_exact(orc2, f(q2)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)
    assert fresh.export()["state"][kv.STATE["error"]].item() == 0
