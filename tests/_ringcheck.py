"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
export a ring, and compare it with the oracle bit for bit."""
import numpy as np
import torch

import ring_kv_cache_gb300 as kv
from oracle import INT32_MIN
from workloads import f32_from_bf16, to_torch_bf16

# Attention tolerance against the float64 oracle fed the same FP8 cache.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev(u16):
    return to_torch_bf16(u16).cuda()


def f(u16):
    return f32_from_bf16(u16)


def make_pair(shape, oracle_cls, **kw):
    """A device ring and an oracle ring of the same shape."""
    ring = kv.KvRing(shape.heads, shape.head_dim, shape.capacity, kw.pop("max_tokens", max(shape.tokens, shape.queries)),
                     shape.max_position, shape.rope_base, **kw)
    orc = oracle_cls(shape.heads, shape.head_dim, shape.capacity, shape.max_position, shape.rope_base)
    return ring, orc


def export_np(ring):
    e = ring.export()
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in e.items()}


def assert_ring_equal(ring, orc, what=""):
    e = export_np(ring)
    H = orc.H
    assert np.array_equal(e["k"], orc.K), f"{what}: key codes differ at {np.argwhere(e['k'] != orc.K)[:5]}"
    assert np.array_equal(e["v"], orc.V), f"{what}: value codes differ at {np.argwhere(e['v'] != orc.V)[:5]}"
    sp = e["slot_pos"].astype(np.int64)
    want = orc.slot_pos.copy()
    assert np.array_equal(sp, want), f"{what}: slot positions differ"
    sc = e["scales"].view(np.uint32)
    assert np.array_equal(sc[:H], orc.scale_k.view(np.uint32)), f"{what}: scale_k"
    assert np.array_equal(sc[H:2 * H], orc.scale_v.view(np.uint32)), f"{what}: scale_v"
    assert np.array_equal(sc[2 * H:3 * H], orc.inv_k.view(np.uint32)), f"{what}: inv_k"
    assert np.array_equal(sc[3 * H:], orc.inv_v.view(np.uint32)), f"{what}: inv_v"
    st = e["state"]
    assert st[kv.STATE["head"]] == orc.head, what
    assert st[kv.STATE["n_valid"]] == orc.n_valid, what
    total = int(np.uint32(st[kv.STATE["total_lo"]])) | (int(np.uint32(st[kv.STATE["total_hi"]])) << 32)
    assert total == orc.total, what
    assert st[kv.STATE["next_pos"]] == orc.next_pos, what
    assert st[kv.STATE["calibrated"]] == int(orc.calibrated), what
    assert st[kv.STATE["error"]] == 0, f"{what}: device error word {st[kv.STATE['error']]}"
    return e


def attn_errors(got, want):
    err = np.abs(np.asarray(got, np.float64) - want)
    return float(err.max()), float(err.mean())


def bf16_bits(t):
    """bf16 CUDA tensor -> numpy uint16 bit patterns (for the oracle)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_from_ring(ring, max_position, rope_base=10000.0):
    """An oracle Ring holding exactly the device ring's current contents."""
    from oracle import Ring
    e = export_np(ring)
    H = ring.H
    orc = Ring(ring.H, ring.d, ring.C, max_position, rope_base)
    orc.K = e["k"].copy()
    orc.V = e["v"].copy()
    orc.slot_pos = e["slot_pos"].astype(np.int64)
    sc = e["scales"].astype(np.float32)
    orc.scale_k, orc.scale_v = sc[:H].copy(), sc[H:2 * H].copy()
    orc.inv_k, orc.inv_v = sc[2 * H:3 * H].copy(), sc[3 * H:].copy()
    st = e["state"]
    orc.head = int(st[kv.STATE["head"]])
    orc.n_valid = int(st[kv.STATE["n_valid"]])
    orc.total = int(np.uint32(st[kv.STATE["total_lo"]])) | (int(np.uint32(st[kv.STATE["total_hi"]])) << 32)
    orc.next_pos = int(st[kv.STATE["next_pos"]])
    orc.calibrated = bool(st[kv.STATE["calibrated"]])
    return orc


def sampled_attention_errors(orc, q_bits, out, rows, qpos=None):
    """Max/mean abs error of device output rows against the float64 oracle."""
    from oracle.attention import attention_exact
    n = q_bits.shape[0]
    if qpos is None:
        qpos = orc.next_pos - n + np.arange(n)
    ref = attention_exact(orc, f32_from_bf16(q_bits[rows]), np.asarray(qpos)[rows])
    got = out[rows].astype(np.float64)
    err = np.abs(got - ref)
    return float(err.max()), float(err.mean()), ref
