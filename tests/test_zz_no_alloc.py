"""The attention entry point that allocates nothing.

Some callers cannot give the library device memory: a plugin inside a host
program that owns the whole device pool, or a real-time loop where an
allocation would stall the device.  kvring_attention_noalloc serves them:
it computes what kvring_attention computes, with its scratch in a fixed
static device array inside the library.

Checked through the C ABI (ctypes, no binding helpers): two calls in a row
each match the existing entry point's output for the same inputs, and the
float64 reference on an oracle ring fed the same frames, within the
attention tolerance the other tests use; a call whose split choice exceeds
the eight splits a cluster merges (so the entry point narrows it to eight)
matches the reference too; and a call with more (query tile, head) units
than the static array holds levels for is refused with KVRING_ERR_CAPACITY
before anything is launched.  This file is named to run last, so a failure
here comes after every other test ran.
"""
import ctypes

import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring
from oracle.attention import attention_exact
from workloads import PROD, RingShape, frame, prod_session

from _ringcheck import MAX_ABS, MEAN_ABS, attn_errors, dev, f, make_pair, sampled_attention_errors

ROWS = np.random.default_rng(77).choice(PROD.queries, 48, replace=False)

pytestmark = pytest.mark.gpu


def _call(fn, ring, q, out):
    s = torch.cuda.current_stream().cuda_stream
    return fn(ctypes.c_void_p(ring.handle), ctypes.c_void_p(q.data_ptr()), None, q.shape[0],
              ctypes.c_void_p(out.data_ptr()), 0, ctypes.c_void_p(s))


def test_noalloc_matches_attention_on_two_calls_in_a_row():
    L = kv.lib()
    sk, sv, frames = prod_session(seed=21, frames=10)
    ring = kv.KvRing(PROD.heads, PROD.head_dim, PROD.capacity, PROD.tokens, PROD.max_position,
                     max_kv_splits=16)
    orc = Ring(PROD.heads, PROD.head_dim, PROD.capacity, PROD.max_position)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    for q, k, v in frames[:8]:
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    for step in (8, 9):
        q, k, v = frames[step]
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
        qd = dev(q)
        want = torch.empty((PROD.queries, PROD.heads, PROD.head_dim), dtype=torch.float32, device="cuda")
        got = torch.full_like(want, float("nan"))
        assert _call(L.kvring_attention, ring, qd, want) == 0
        assert _call(L.kvring_attention_noalloc, ring, qd, got) == 0
        torch.cuda.synchronize()
        err = (got.double() - want.double()).abs()
        assert torch.isfinite(got).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (step, err.max().item())
        # and against the float64 reference on sampled rows of every head
        mx, mn, _ = sampled_attention_errors(orc, q, got.cpu().numpy(), ROWS)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (step, mx, mn)


def test_noalloc_narrows_more_than_eight_splits():
    """One query tile of two heads over a full 5,788-slot ring: the split
    choice is sixteen (two units on a GPU of 152 SMs); the entry point merges
    at most eight inside a cluster and needs no partials, so it narrows the
    call to eight splits of six tiles.  Its output matches the reference."""
    L = kv.lib()
    rng = np.random.default_rng(23)
    shape = RingShape(heads=2, head_dim=128, capacity=5788, tokens=757, queries=128, max_position=8000)
    ring, orc = make_pair(shape, Ring, max_tokens=757, max_kv_splits=16)
    for i in range(8):
        _, k, v = frame(rng, shape, 757)
        if i == 0:
            ring.calibrate(dev(k), dev(v))
            orc.calibrate(f(k), f(v))
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    q, _, _ = frame(rng, shape, 128)
    want = attention_exact(orc, f(q))
    for _ in range(2):
        got = torch.full((128, 2, 128), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(L.kvring_attention_noalloc, ring, dev(q), got) == 0
        torch.cuda.synchronize()
        mx, mn = attn_errors(got.cpu().numpy(), want)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_noalloc_refuses_what_does_not_fit():
    L = kv.lib()
    # 64 heads x 513 query tiles = 32,832 (tile, head) levels > 128 KiB / 4 B
    n_big = 513 * 128
    ring = kv.KvRing(64, 128, 256, n_big, 4096, max_kv_splits=1)
    x = torch.zeros((8, 64, 128), dtype=torch.bfloat16, device="cuda")
    ring.calibrate(x, x)
    q = torch.zeros((n_big, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((n_big, 64, 128), dtype=torch.float32, device="cuda")
    assert _call(L.kvring_attention_noalloc, ring, q, out) == 3      # KVRING_ERR_CAPACITY
    small = torch.zeros((128, 64, 128), dtype=torch.bfloat16, device="cuda")
    out_small = torch.empty((128, 64, 128), dtype=torch.float32, device="cuda")
    assert _call(L.kvring_attention_noalloc, ring, small, out_small) == 0
    torch.cuda.synchronize()
    assert np.all(out_small.cpu().numpy() == 0)                      # empty ring: zeros
