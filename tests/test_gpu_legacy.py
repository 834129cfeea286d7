"""The legacy upkeep (window copy + RoPE of every key + re-quantisation at
every call) against its oracle, bit for bit: the bf16 windows, the FP8 codes,
the window scales, the positions and the ring state, on the tiny workload
(wrapping twice) and the production-shaped one; attention over the rebuilt
cache against the float64 reference."""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle.attention import attention_exact
from oracle.legacy import LegacyWindow
from workloads import PROD, TINY, bf16_from_f32, prod_session, tiny_session

from _ringcheck import MAX_ABS, MEAN_ABS, attn_errors, dev, export_np, f

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check(ring, win, w, what):
    e = export_np(ring)
    H, C, fill = w.H, w.C, w.fill
    assert np.array_equal(e["k"][:, :fill], w.K[:, :fill]), f"{what}: key codes"
    assert np.array_equal(e["v"][:, :fill], w.V[:, :fill]), f"{what}: value codes"
    assert np.array_equal(e["slot_pos"][:fill].astype(np.int64), w.slot_pos[:fill]), f"{what}: positions"
    sc = e["scales"].view(np.uint32)
    assert np.array_equal(sc[:H], w.scale_k.view(np.uint32)), f"{what}: scale_k"
    assert np.array_equal(sc[H:2 * H], w.scale_v.view(np.uint32)), f"{what}: scale_v"
    st = e["state"]
    assert st[kv.STATE["n_valid"]] == fill and st[kv.STATE["next_pos"]] == w.total, what
    wk, wv = win.window()
    assert np.array_equal(_bits(wk)[:fill], bf16_from_f32(w.k[:fill])), f"{what}: key window"
    assert np.array_equal(_bits(wv)[:fill], bf16_from_f32(w.v[:fill])), f"{what}: value window"


def test_legacy_tiny_session_bit_exact():
    frames = tiny_session()
    ring = kv.KvRing(TINY.heads, TINY.head_dim, TINY.capacity, TINY.tokens, TINY.max_position)
    win = kv.LegacyWindows(ring)
    w = LegacyWindow(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position)
    for i, (q, k, v) in enumerate(frames):
        win.upkeep(dev(k), dev(v))
        w.upkeep(f(k), f(v))
        _check(ring, win, w, f"tiny call {i}")
        out = ring.attention(dev(q)).cpu().numpy()
        mx, mn = attn_errors(out, attention_exact(w.as_ring(TINY.max_position), f(q)))
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, mx, mn)


def test_legacy_production_shape_bit_exact_and_attention():
    _, _, frames = prod_session(seed=31, frames=9)
    ring = kv.KvRing(PROD.heads, PROD.head_dim, PROD.capacity, PROD.tokens, PROD.max_position)
    win = kv.LegacyWindows(ring)
    w = LegacyWindow(PROD.heads, PROD.head_dim, PROD.capacity, PROD.max_position)
    for i, (q, k, v) in enumerate(frames):
        win.upkeep(dev(k), dev(v))
        w.upkeep(f(k), f(v))
        if i in (0, 7, 8):
            _check(ring, win, w, f"production call {i}")
    q = frames[8][0]
    out = ring.attention(dev(q)).cpu().numpy()
    mx, mn = attn_errors(out, attention_exact(w.as_ring(PROD.max_position), f(q)))
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_legacy_argument_errors():
    ring = kv.KvRing(2, 64, 48, 12, 256)
    win = kv.LegacyWindows(ring)
    x = torch.zeros((12, 2, 64), dtype=torch.bfloat16, device="cuda")
    L = kv.lib()
    s = torch.cuda.current_stream().cuda_stream
    a, b = win.k[0].data_ptr(), win.k[1].data_ptr()
    va, vb = win.v[0].data_ptr(), win.v[1].data_ptr()
    assert L.kvring_legacy_upkeep(ring.handle, a, va, a, vb, x.data_ptr(), x.data_ptr(), 12, s) == 1   # aliased
    big = torch.zeros((60, 2, 64), dtype=torch.bfloat16, device="cuda")
    assert L.kvring_legacy_upkeep(ring.handle, a, va, b, vb, big.data_ptr(), big.data_ptr(), 60, s) == 3
    assert L.kvring_legacy_upkeep(ring.handle, a, va, b, vb, None, x.data_ptr(), 12, s) == 1
