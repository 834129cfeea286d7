"""QKV projection with the cache write fused in, against the oracle: the
bf16 projection outputs (queries, and keys and values when stored) against
the oracle's exactly rounded projection, and the ring's bytes, positions and
state against the oracle ring written with the oracle's projected keys and
values.

The tensor cores sum in fp32, in their own order, so an output can round to
a different bf16 value than the exactly rounded sum: one step where the
exact sum lies close to a rounding midpoint, and many steps for outputs near
zero, where the sum cancels and a bf16 step is tiny against the terms.  The
test bounds every output by what fp32 accumulation allows,
|got - exact| <= half a bf16 step of the exact sum + d_model * 2^-24 *
sum_i |x_i w_i| (the worst-case error of an fp32 sum of d_model exact
products in any order), caps the share of outputs that differ from the
exact rounding at 5e-3 and prints it (about 3e-3 for d_model 5,120), and
requires every cache row whose bf16 inputs equal the exactly rounded ones to
be bit-exact, and the slot positions and ring state to be exact.
"""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring, e4m3
from oracle.projection import project_qkv
from workloads import PROD, TINY, bf16_from_f32

from _ringcheck import MAX_ABS, MEAN_ABS, dev, export_np, f, sampled_attention_errors

pytestmark = pytest.mark.gpu


def _weights(rng, rows, dm, scale):
    return bf16_from_f32((rng.standard_normal((rows, dm)) * scale).astype(np.float32))


def _acts(rng, n, dm):
    return bf16_from_f32(rng.standard_normal((n, dm)).astype(np.float32))


def _bf16_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bound(x, w, heads, d):
    """Per-output allowance [3][n][H][d]: half a bf16 step of the exact sum
    plus the fp32 accumulation bound d_model * 2^-24 * sum_i |x_i w_i|."""
    xf, wf = _bf16_f64(x), _bf16_f64(w)
    exact = xf @ wf.T
    absum = np.abs(xf) @ np.abs(wf).T
    e = np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -133)))
    half_step = np.ldexp(1.0, (np.maximum(e, -126) - 8).astype(int))
    allow = half_step + xf.shape[1] * 2.0 ** -24 * absum
    n, hd = x.shape[0], heads * d
    split = lambda a: [a[:, i * hd:(i + 1) * hd].reshape(n, heads, d) for i in range(3)]
    return split(exact), split(allow)


RATES = []


def _compare_bf16(got, want, exact, allow, what, rate=5e-3):
    err = np.abs(_bf16_f64(got) - exact)
    assert np.all(err <= allow), (what, float((err / allow).max()), np.argwhere(err > allow)[:4])
    diff = got != want
    assert diff.mean() <= rate, (what, float(diff.mean()))
    RATES.append((what, float(diff.mean())))
    return ~diff


def _codes_within(a, b, dx, inv, pairs):
    """Codes a, b [H, n, d] of rows written from bf16 inputs that differ by
    dx [H, n, d] (absolute): with RoPE (pairs) a pair's two components mix,
    so each output of the pair may move by (|dx0| + |dx1|) * inv_scale,
    without it by |dx| * inv_scale; plus one E4M3 step of rounding."""
    da, db = e4m3.decode(a), e4m3.decode(b)
    m = np.maximum(np.abs(da), np.abs(db))
    step = np.where(m >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(m, 2.0 ** -6))) - 3), 2.0 ** -9)
    if pairs:
        dx = np.repeat(dx[..., 0::2] + dx[..., 1::2], 2, axis=-1)
    move = dx * np.asarray(inv, np.float64)[:, None, None]
    return np.abs(da - db) <= move * (1 + 1e-6) + step


def _session(shape, dm, frames, seed, scale):
    rng = np.random.default_rng(seed)
    w = _weights(rng, 3 * shape.heads * shape.head_dim, dm, scale)
    xs = [_acts(rng, shape.tokens, dm) for _ in range(frames)]
    return w, xs


@pytest.mark.parametrize("shape,dm,frames,scale", [(TINY, 128, 8, 0.1), (PROD, 5120, 9, 0.015)])
def test_projection_write_matches_oracle(shape, dm, frames, scale):
    w, xs = _session(shape, dm, frames, 21, scale)
    H, d = shape.heads, shape.head_dim
    ring = kv.KvRing(H, d, shape.capacity, max(shape.tokens, shape.queries), shape.max_position, shape.rope_base)
    orc = Ring(H, d, shape.capacity, shape.max_position, shape.rope_base)
    wd = dev(w)
    # session start: the first frame's keys and values calibrate both rings
    q0, k0, v0 = project_qkv(xs[0], w, H, d)
    (eq, ek, ev), (aq, ak, av) = _bound(xs[0], w, H, d)
    q_out, kv_out = ring.project_write(dev(xs[0]), wd, write=False, store_kv=True)
    torch.cuda.synchronize()
    _compare_bf16(q_out.view(torch.int16).cpu().numpy().view(np.uint16), q0, eq, aq, "q")
    kvn = kv_out.view(torch.int16).cpu().numpy().view(np.uint16)
    _compare_bf16(kvn[0], k0, ek, ak, "k")
    _compare_bf16(kvn[1], v0, ev, av, "v")
    ring.calibrate(dev(k0), dev(v0))
    orc.calibrate(f(k0), f(v0))
    for i in range(frames):
        q, k, v = project_qkv(xs[i], w, H, d)
        (eq, ek, ev), (aq, ak, av) = _bound(xs[i], w, H, d)
        q_out, kv_out = ring.project_write(dev(xs[i]), wd, store_kv=True)
        slots = orc.write(f(k), f(v))
        torch.cuda.synchronize()
        kvn = kv_out.view(torch.int16).cpu().numpy().view(np.uint16)
        same_k = _compare_bf16(kvn[0], k, ek, ak, f"k {i}").all(axis=2)      # [n, H] rows whose inputs agree
        same_v = _compare_bf16(kvn[1], v, ev, av, f"v {i}").all(axis=2)
        _compare_bf16(q_out.view(torch.int16).cpu().numpy().view(np.uint16), q, eq, aq, f"q {i}")
        e = export_np(ring)
        for t in range(shape.tokens):
            s = slots[t]
            for h in range(H):
                if same_k[t, h]:
                    assert np.array_equal(e["k"][h, s], orc.K[h, s]), (i, t, h)
                if same_v[t, h]:
                    assert np.array_equal(e["v"][h, s], orc.V[h, s]), (i, t, h)
        assert same_k.mean() > 0.5 and same_v.mean() > 0.5, (same_k.mean(), same_v.mean())
        # every code written now, including rows whose inputs differ, within
        # what the input difference and one rounding allow
        dk = np.abs(_bf16_f64(kvn[0]) - _bf16_f64(k)).transpose(1, 0, 2)
        dv = np.abs(_bf16_f64(kvn[1]) - _bf16_f64(v)).transpose(1, 0, 2)
        assert _codes_within(e["k"][:, slots], orc.K[:, slots], dk, orc.inv_k, True).all()
        assert _codes_within(e["v"][:, slots], orc.V[:, slots], dv, orc.inv_v, False).all()
        assert np.array_equal(e["slot_pos"].astype(np.int64), orc.slot_pos)
        st = e["state"]
        assert st[kv.STATE["head"]] == orc.head and st[kv.STATE["n_valid"]] == orc.n_valid
        assert st[kv.STATE["next_pos"]] == orc.next_pos and st[kv.STATE["error"]] == 0
    worst = max(RATES, key=lambda x: x[1])
    print(f"{shape.heads}x{shape.head_dim}, d_model {dm}: outputs off the exact bf16 rounding: "
          f"worst {worst[1]:.2e} ({worst[0]}), mean {np.mean([r for _, r in RATES]):.2e}")
    RATES.clear()


def test_projection_argument_errors():
    ring = kv.KvRing(TINY.heads, TINY.head_dim, TINY.capacity, TINY.tokens, TINY.max_position)
    x = torch.zeros((TINY.tokens, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((3 * TINY.heads * TINY.head_dim, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kv.KvRingError) as e:          # write before calibration
        ring.project_write(x, w)
    assert e.value.status == 2
    with pytest.raises(ValueError):                   # d_model not a multiple of 64
        ring.project_write(x[:, :96].contiguous(), w[:, :96].contiguous(), write=False)


def test_projection_outputs_consumed_at_once():
    """The projection's outputs read by the very next call on the stream, with
    no host synchronisation between: its stored keys and values by a write,
    its queries by an attention.  The projection lets its dependents start
    before it has stored them, so both calls must read those inputs only
    after waiting for it -- the library's per-stream record of the buffers
    its last kernel writes makes them do so (counted by late_reads) -- and
    the results match the oracle.  Inputs no library kernel wrote are still
    read before the wait."""
    shape, dm, scale = PROD, 5120, 0.015
    w, xs = _session(shape, dm, 8, 33, scale)
    H, d = shape.heads, shape.head_dim
    ring = kv.KvRing(H, d, shape.capacity, max(shape.tokens, shape.queries), shape.max_position, shape.rope_base)
    orc = Ring(H, d, shape.capacity, shape.max_position, shape.rope_base)
    wd = dev(w)
    rows = np.random.default_rng(5).choice(shape.queries, 48, replace=False)
    q0, k0, v0 = project_qkv(xs[0], w, H, d)
    (_, ek, ev), (_, ak, av) = _bound(xs[0], w, H, d)
    ring.calibrate(dev(k0), dev(v0))
    orc.calibrate(f(k0), f(v0))
    # frame 0: stored keys and values, written by a separate write at once
    x0 = dev(xs[0])
    before = kv.late_reads()
    _, kv_out = ring.project_write(x0, wd, write=False, store_kv=True)
    ring.write(kv_out[0], kv_out[1])
    assert kv.late_reads() == before + 1
    slots = orc.write(f(k0), f(v0))
    torch.cuda.synchronize()
    kvn = kv_out.view(torch.int16).cpu().numpy().view(np.uint16)
    same_k = _compare_bf16(kvn[0], k0, ek, ak, "k").all(axis=2)
    same_v = _compare_bf16(kvn[1], v0, ev, av, "v").all(axis=2)
    e = export_np(ring)
    for t in range(shape.tokens):
        for h in range(H):
            if same_k[t, h]:
                assert np.array_equal(e["k"][h, slots[t]], orc.K[h, slots[t]]), (t, h)
            if same_v[t, h]:
                assert np.array_equal(e["v"][h, slots[t]], orc.V[h, slots[t]]), (t, h)
    assert np.array_equal(e["slot_pos"].astype(np.int64), orc.slot_pos)
    # frames 1-7 (the ring wraps in frame 7): the fused write, then an
    # attention over the queries it just stored
    for i in range(1, 8):
        q, k, v = project_qkv(xs[i], w, H, d)
        x = dev(xs[i])
        before = kv.late_reads()
        q_out, _ = ring.project_write(x, wd)
        out = ring.attention(q_out)
        assert kv.late_reads() == before + 1, i
        orc.write(f(k), f(v))
        torch.cuda.synchronize()
        mx, mn, _ = sampled_attention_errors(orc, q, out.cpu().numpy(), rows)
        assert mx <= MAX_ABS and mn <= MEAN_ABS, (i, mx, mn)
        assert export_np(ring)["state"][kv.STATE["error"]] == 0
    # a frame and queries uploaded by the caller: read before the wait
    q, k, v = project_qkv(xs[0], w, H, d)
    kd, vd, qd = dev(k), dev(v), dev(q)
    torch.cuda.synchronize()
    before = kv.late_reads()
    ring.write(kd, vd)
    ring.attention(qd)
    assert kv.late_reads() == before
