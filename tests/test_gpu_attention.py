"""FP8 attention kernel against the oracle.

* the float64 reference (unquantised queries, exact softmax) over the same
  FP8 cache, within max-abs 2e-2 / mean-abs 2e-3, at every precision level;
* the kernel-mirroring diagnostic (same FP8 query terms, same lazy maximum,
  probabilities rounded to f16, one key/value split) much more tightly,
  which separates kernel bugs from format error;
* closed forms: an empty ring gives zeros, a single filled slot gives its
  value, and the split-KV merge matches the single-split result.
"""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring
from oracle.attention import attention_emulated, attention_exact
from workloads import RingShape, TINY, frame, tiny_session

from _ringcheck import MAX_ABS, MEAN_ABS, attn_errors, dev, f, make_pair

pytestmark = pytest.mark.gpu


def _tiny_loaded(frames_written, **kw):
    frames = tiny_session()
    ring, orc = make_pair(TINY, Ring, **kw)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    for i in range(frames_written):
        ring.write(dev(frames[i][1]), dev(frames[i][2]))
        orc.write(f(frames[i][1]), f(frames[i][2]))
    return ring, orc, frames


@pytest.mark.parametrize("level", [1, 2, 3, 4])
def test_kernel_matches_its_mirror_tightly(level):
    """Level 1 is only chosen automatically for tiny-magnitude heads; forced
    here, its output must still match its mirror (format error aside).
    Level 4 carries the probabilities as two f16 terms."""
    ring, orc, frames = _tiny_loaded(6, max_kv_splits=1, attn_precision=level)
    q = frames[6][0]
    out = ring.attention(dev(q)).cpu().numpy()
    # the kernel's probability shift (2^7) and rescale threshold (8, log2 units)
    mirror = attention_emulated(orc, f(q), None, level, "f16x2" if level == 4 else "f16",
                                p_shift=7.0, tau=8.0)
    mx, mn = attn_errors(out, mirror)
    scale = np.abs(mirror).max()
    assert mx <= 2e-3 * scale, (level, mx, scale)
    if level >= 2:
        ref = attention_exact(orc, f(q))
        mx2, mn2 = attn_errors(out, ref)
        assert mx2 <= MAX_ABS and mn2 <= MEAN_ABS


def test_levels_reported_and_automatic_choice_is_in_range():
    ring, orc, frames = _tiny_loaded(3)
    ring.attention(dev(frames[3][0]))
    lv = ring.levels().cpu().numpy()
    assert lv.shape[1] == TINY.heads and np.all((lv[0] >= 1) & (lv[0] <= 4))


def _loaded(shape, frames, **kw):
    ring, orc = make_pair(shape, Ring, **kw)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    for _, k, v in frames:
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    return ring, orc


def test_automatic_level_1_on_small_heads_meets_the_bar():
    """Heads whose keys and values are small (sigma 0.08: L = max|q| max|k|
    about 2, V = max|v| about 0.35) are given one query term by the automatic
    rule; the output still meets the float64 reference's bar."""
    rng = np.random.default_rng(12)
    shape = RingShape(heads=2, head_dim=128, capacity=700, tokens=300, queries=256, max_position=2000)
    sig = np.array([0.08, 0.06])
    frames = [frame(rng, shape, 300, sig, sig) for _ in range(3)]
    ring, orc = _loaded(shape, frames)
    q, _, _ = frame(rng, shape, 256)
    out = ring.attention(dev(q)).cpu().numpy()
    lv = ring.levels().cpu().numpy()[:2]
    assert np.all(lv == 1), lv
    mx, mn = attn_errors(out, attention_exact(orc, f(q)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_automatic_level_4_on_heavy_tailed_heads_meets_the_bar():
    """Heavy-tailed heads with large values (Student-t keys and values, 3
    degrees of freedom, scales up to 10: V = max|v| in the hundreds) are given
    four query terms and two-term f16 probabilities by the automatic rule, and
    meet the float64 reference's absolute bar."""
    rng = np.random.default_rng(13)
    shape = RingShape(heads=2, head_dim=128, capacity=1500, tokens=700, queries=256, max_position=4000)
    sk, sv = np.array([6.0, 2.5]), np.array([10.0, 4.0])
    frames = [frame(rng, shape, 700, sk, sv, dist="student_t") for _ in range(3)]
    ring, orc = _loaded(shape, frames, max_tokens=700)
    q, _, _ = frame(rng, shape, 256)
    out = ring.attention(dev(q)).cpu().numpy()
    lv = ring.levels().cpu().numpy()[:2]
    assert np.all(lv == 4), lv
    want = attention_exact(orc, f(q))
    mx, mn = attn_errors(out, want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn, np.abs(want).max())


def test_empty_ring_gives_zeros():
    ring = kv.KvRing(2, 64, 48, 12, 256)
    x = torch.randn((12, 2, 64), device="cuda").bfloat16()
    ring.calibrate(x, x)
    out = ring.attention(x)
    assert torch.count_nonzero(out) == 0


def test_single_filled_slot_returns_its_value():
    rng = np.random.default_rng(2)
    shape = RingShape(heads=2, head_dim=128, capacity=300, tokens=1, queries=200, max_position=1000)
    ring, orc = make_pair(shape, Ring, max_tokens=200)
    q, k, v = frame(rng, shape, 1)
    ring.calibrate(dev(k), dev(v))
    orc.calibrate(f(k), f(v))
    ring.write(dev(k), dev(v))
    orc.write(f(k), f(v))
    qq, _, _ = frame(rng, shape, 200)
    out = ring.attention(dev(qq), torch.zeros(200, dtype=torch.int32, device="cuda")).cpu().numpy()
    want = attention_exact(orc, f(qq), np.zeros(200, int))
    assert np.allclose(out, want, atol=1e-5 * np.abs(want).max())


def test_default_positions_up_to_the_table_end_and_before_enough_tokens():
    """Default query positions are the last n_q positions written.  When all
    of them lie in the RoPE table (here up to its last row, in both query
    tiles) the output matches the reference and no error is recorded.  When
    fewer than n_q tokens were ever written, the first rows' positions are
    negative: the device error word records it, and the rows whose positions
    are valid still match."""
    rng = np.random.default_rng(7)
    shape = RingShape(heads=2, head_dim=128, capacity=300, tokens=150, queries=150, max_position=450)
    ring, orc = make_pair(shape, Ring)
    for i in range(3):                        # positions 0..449: the table's last row is used
        q, k, v = frame(rng, shape, 150)
        if i == 0:
            ring.calibrate(dev(k), dev(v))
            orc.calibrate(f(k), f(v))
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    out = ring.attention(dev(q)).cpu().numpy()
    mx, mn = attn_errors(out, attention_exact(orc, f(q)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)
    assert ring.export()["state"][kv.STATE["error"]].item() == 0

    ring, orc = make_pair(shape, Ring)
    q, k, v = frame(rng, shape, 150)
    ring.calibrate(dev(k), dev(v))
    orc.calibrate(f(k), f(v))
    ring.write(dev(k[:100]), dev(v[:100]))
    orc.write(f(k[:100]), f(v[:100]))
    out = ring.attention(dev(q)).cpu().numpy()      # default positions -50 .. 99
    assert ring.export()["state"][kv.STATE["error"]].item() & kv.DEVERR_POSITION
    rows = np.arange(50, 150)
    mx, mn = attn_errors(out[rows], attention_exact(orc, f(q[rows]), rows - 50))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 8, 16])
def test_split_merge_consistent(splits):
    """2..8 splits merge inside a thread-block cluster, more through global
    partials; both must agree with the float64 reference."""
    rng = np.random.default_rng(3)
    shape = RingShape(heads=2, head_dim=128, capacity=2000, tokens=700, queries=300, max_position=4000)
    ring, orc = make_pair(shape, Ring, max_tokens=700, max_kv_splits=splits)
    for i in range(3):
        q, k, v = frame(rng, shape, 700)
        if i == 0:
            ring.calibrate(dev(k), dev(v))
            orc.calibrate(f(k), f(v))
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    q, _, _ = frame(rng, shape, 300)
    out = ring.attention(dev(q)).cpu().numpy()
    mx, mn = attn_errors(out, attention_exact(orc, f(q)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (splits, mx, mn)


@pytest.mark.parametrize("heads,out_dtype", [(4, torch.float32), (8, torch.bfloat16), (20, torch.float32)])
def test_cluster_merge_production_scale(heads, out_dtype):
    """The cluster merge at production scale: a 757-query call over a wrapped
    5,788-slot ring on 4, 8 or 20 heads makes the host choose about 6, 3 or
    2 splits of each query tile (each CTA of the cluster owns 128 / splits
    rows, not a multiple of 32 for most split counts); sampled rows of every
    query tile and head must match the float64 reference, in f32 and bf16
    output."""
    rng = np.random.default_rng(11 + heads)
    shape = RingShape(heads=heads, head_dim=128, capacity=5788, tokens=757, queries=757, max_position=40960)
    ring, orc = make_pair(shape, Ring, max_kv_splits=16)
    for i in range(9):                       # 6,813 tokens: wrapped
        q, k, v = frame(rng, shape, 757)
        if i == 0:
            ring.calibrate(dev(k), dev(v))
            orc.calibrate(f(k), f(v))
        ring.write(dev(k), dev(v))
        orc.write(f(k), f(v))
    q, _, _ = frame(rng, shape, 757)
    out = ring.attention(dev(q), out_dtype=out_dtype).float().cpu().numpy()
    rows = np.concatenate([np.arange(0, 757, 41), [36, 37, 38, 63, 64, 127, 128, 756]])
    want = attention_exact(orc, f(q[rows]), orc.next_pos - 757 + rows)
    mx, mn = attn_errors(out[rows], want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (heads, mx, mn)
    assert ring.export()["state"][kv.STATE["error"]].item() == 0


def test_bf16_output_close_to_f32_output():
    ring, orc, frames = _tiny_loaded(5)
    q = dev(frames[5][0])
    o32 = ring.attention(q)
    o16 = ring.attention(q, out_dtype=torch.bfloat16)
    assert torch.allclose(o16.float(), o32, rtol=2 ** -7, atol=1e-6)


@pytest.mark.parametrize("splits", [4, 8, 12])
def test_split_merge_with_empty_splits_and_bf16_output(splits):
    """A ring one-third full: the last splits of each query tile own no
    key/value tiles and contribute nothing; the merged bf16 output must
    still match the reference, and so must the f32 output."""
    rng = np.random.default_rng(4)
    shape = RingShape(heads=2, head_dim=128, capacity=2000, tokens=700, queries=300, max_position=4000)
    ring, orc = make_pair(shape, Ring, max_tokens=700, max_kv_splits=splits)
    q, k, v = frame(rng, shape, 700)
    ring.calibrate(dev(k), dev(v))
    orc.calibrate(f(k), f(v))
    ring.write(dev(k), dev(v))
    orc.write(f(k), f(v))
    q, _, _ = frame(rng, shape, 300)
    want = attention_exact(orc, f(q))
    out = ring.attention(dev(q)).cpu().numpy()
    mx, mn = attn_errors(out, want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (splits, mx, mn)
    outb = ring.attention(dev(q), out_dtype=torch.bfloat16).float().cpu().numpy()
    mx, mn = attn_errors(outb, want)
    assert mx <= MAX_ABS + 2.0 ** -8 * np.abs(want).max() and mn <= MEAN_ABS + 1e-3, (splits, mx, mn)
