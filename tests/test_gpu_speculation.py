"""The attention's early query preparation, against the float64 reference.

With default positions the kernel rotates and splits its queries before it
waits for the preceding kernel, for the positions implied by the ring's
next-position hint (which every write leaves as it starts), and after the
wait checks them against the ring's next position, preparing the queries
again if the guess was wrong.  These tests make the guess wrong on purpose
(kvring_debug_attention_guess: off by max_position, so also outside the
RoPE table, which must not be reported as an error) and chain writes and
attention calls with no host synchronisation, where the hint the attention
reads may still be a write's early guess; every output must match the
reference, and the error word must report only real position errors.
"""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring
from oracle.attention import attention_exact
from workloads import PROD, RingShape, frame, prod_session, to_torch_bf16

from _ringcheck import MAX_ABS, MEAN_ABS, attn_errors, dev, f, make_pair, sampled_attention_errors

pytestmark = pytest.mark.gpu

SHAPE = RingShape(heads=3, head_dim=128, capacity=900, tokens=300, queries=300, max_position=4000)


def _loaded(seed, frames=4):
    rng = np.random.default_rng(seed)
    ring, orc = make_pair(SHAPE, Ring)
    for i in range(frames):                   # 1,200 tokens: wrapped
        q, k, v = frame(rng, SHAPE, 300)
        if i == 0:
            ring.calibrate(dev(k), dev(v))
            orc.calibrate(f(k), f(v))
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    return rng, ring, orc


def _error_word(ring):
    return ring.export()["state"][kv.STATE["error"]].item()


def test_guess_setting_is_checked_on_the_host():
    _, ring, _ = _loaded(40, frames=1)
    assert kv.lib().kvring_debug_attention_guess(ring.handle, 2) == 1
    assert kv.lib().kvring_debug_attention_guess(None, 0) == 1


def test_wrong_guess_is_redone():
    rng, ring, orc = _loaded(41)
    q, _, _ = frame(rng, SHAPE, 300)
    ring.set_attention_guess(True)
    out = ring.attention(dev(q)).cpu().numpy()
    mx, mn = attn_errors(out, attention_exact(orc, f(q)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)
    assert _error_word(ring) == 0            # the guessed positions were out of range: not reported
    ring.set_attention_guess(False)
    out = ring.attention(dev(q)).cpu().numpy()
    mx, mn = attn_errors(out, attention_exact(orc, f(q)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)
    assert _error_word(ring) == 0


def test_real_position_errors_still_reported():
    """Default positions below zero (more queries than tokens written), with
    the guess right and with it wrong: the error bit is set either way and
    the rows with valid positions match the reference."""
    for wrong in (False, True):
        rng = np.random.default_rng(42)
        ring, orc = make_pair(SHAPE, Ring)
        q, k, v = frame(rng, SHAPE, 300)
        ring.calibrate(dev(k), dev(v))
        orc.calibrate(f(k), f(v))
        ring.write(dev(k[:200]), dev(v[:200]))
        orc.write(f(k[:200]), f(v[:200]))
        ring.set_attention_guess(wrong)
        out = ring.attention(dev(q)).cpu().numpy()      # default positions -100 .. 199
        assert _error_word(ring) & kv.DEVERR_POSITION, wrong
        rows = np.arange(100, 300)
        mx, mn = attn_errors(out[rows], attention_exact(orc, f(q[rows]), rows - 100))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (wrong, mx, mn)


def test_chained_writes_then_attention():
    """Two writes and an attention on one ring enqueued back to back (the
    second write's early hint is taken before the first has published, so
    the attention may start from a wrong guess), then attention calls after
    a delta rotation; every output matches the reference."""
    sk, sv, fr = prod_session(seed=43, frames=12)
    ring, orc = make_pair(PROD, Ring)
    t = [(to_torch_bf16(q).cuda(), to_torch_bf16(k).cuda(), to_torch_bf16(v).cuda()) for q, k, v in fr]
    ring.calibrate(t[0][1], t[0][2])
    orc.calibrate(f(fr[0][1]), f(fr[0][2]))
    rows = np.random.default_rng(6).choice(PROD.queries, 32, replace=False)
    torch.cuda.synchronize()
    for i in range(0, 12, 2):
        ring.write(t[i][1], t[i][2])
        ring.write(t[i + 1][1], t[i + 1][2])
        out = ring.attention(t[i + 1][0])
        if i == 6:
            ring.delta_rotate(kv.TO_OLDEST)
            out2 = ring.attention(t[i + 1][0])
        orc.write(f(fr[i][1]), f(fr[i][2]))
        orc.write(f(fr[i + 1][1]), f(fr[i + 1][2]))
        torch.cuda.synchronize()
        mx, mn, _ = sampled_attention_errors(orc, fr[i + 1][0], out.cpu().numpy(), rows)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, mx, mn)
        if i == 6:
            orc.delta_rotate()
            mx, mn, _ = sampled_attention_errors(orc, fr[i + 1][0], out2.cpu().numpy(), rows)
            assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, "after reset", mx, mn)
    assert _error_word(ring) == 0
