"""Attention of a new frame's queries over the ring cache, plain CPU model.

Test infrastructure only; nothing in the library imports it.

"Where the Time Went" and "Blackwell and Beyond Four GPUs" on the Runway
Characters page: every attention call of a step reads its layer's cache of
5,788 slots, with FP8 keys and values that carry per-head scales.  Keys
already hold their rotation (RoPE at write time), so slot order does not
matter; queries are rotated by their own positions.  The pages give no
softmax scale or mask; this oracle takes the usual 1/sqrt(d), no causal mask
(every query sees every filled slot), and leaves empty slots out.

``attention_exact`` is the reference the CUDA path is judged against: the
queries in float64 without any quantisation, keys and values dequantised
from the same FP8 cache bytes (code value times the fp32 scale, in float64),
and a float64 softmax with the row maximum subtracted.

``attention_part_f64`` / ``merge_parts_f64`` / ``attention_split`` restate
the split of one query tile's slots among several workers: each part's
normalised output with its log-sum-exp, and their combination, which is
exact up to rounding (the merged parts equal the whole softmax).

``attention_emulated`` is a diagnostic that repeats the CUDA kernel's
choices (queries split into FP8 terms with a per-row scale, probabilities
scaled by 2^7 relative to a lazily raised running maximum and carried as FP8
terms, in half precision, or as two half-precision terms) in float64, so
that format error and kernel bugs can be told apart.
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3
from .rope import rotate_f64

INT32_MIN = -(2 ** 31)


def softmax_attention_f64(qt: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """o[t,h,:] = sum_j softmax_j(qt[t,h]·k[h,j] / sqrt(d)) v[h,j,:] in float64.

    qt [n, H, d]; k, v [H, m, d].  m = 0 gives zeros.
    """
    n, H, d = qt.shape
    if k.shape[1] == 0:
        return np.zeros((n, H, d), dtype=np.float64)
    s = np.einsum("thd,hjd->thj", qt, k) / math.sqrt(d)
    s = s - s.max(axis=2, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=2, keepdims=True)
    return np.einsum("thj,hjd->thd", p, v)


def attention_exact(ring, q: np.ndarray, qpos=None) -> np.ndarray:
    """Reference attention of queries q (float32 [n, H, d]) over ``ring``.

    qpos defaults to the n positions just before ``ring.next_pos``; with the
    3-D RoPE variant it is an explicit [n, 3] array of (t, y, x).
    """
    q = np.asarray(q, dtype=np.float64)
    n = q.shape[0]
    if qpos is None:
        qpos = ring.next_pos - n + np.arange(n)
    qt = ring.rope_f64(q, qpos)
    k, v, _ = ring.dequantised()
    return softmax_attention_f64(qt, k, v)


def attention_part_f64(qt: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Attention over one part of the slots, normalised within the part.

    Returns (o, lse): o[t,h,:] = sum_j softmax_j(s) v[h,j,:] over the part's
    slots j only, with s = qt[t,h]·k[h,j] / sqrt(d), and lse[t,h] =
    log sum_j exp(s), the part's log-sum-exp in float64.  An empty part gives
    zeros and lse = -inf.  This is the partial result a split of the keys
    produces when one query tile's slots are shared among several workers.
    """
    n, H, d = qt.shape
    if k.shape[1] == 0:
        return np.zeros((n, H, d), dtype=np.float64), np.full((n, H), -np.inf)
    s = np.einsum("thd,hjd->thj", qt, k) / math.sqrt(d)
    m = s.max(axis=2)
    p = np.exp(s - m[:, :, None])
    ell = p.sum(axis=2)
    o = np.einsum("thj,hjd->thd", p, v) / ell[:, :, None]
    return o, m + np.log(ell)


def merge_parts_f64(parts) -> np.ndarray:
    """Combine partial results (o_s, lse_s) of disjoint parts of the slots.

    With M = max_s lse_s and w_s = exp(lse_s - M), the whole softmax is
    o = sum_s w_s o_s / sum_s w_s, because exp(lse_s) is part s's sum of
    exponentials and o_s its normalised output.  Parts with lse = -inf
    weigh nothing; a row whose parts are all empty is zero.
    """
    os_ = np.stack([np.asarray(o, dtype=np.float64) for o, _ in parts])      # [S, n, H, d]
    lse = np.stack([np.asarray(l, dtype=np.float64) for _, l in parts])      # [S, n, H]
    M = lse.max(axis=0)
    finite = np.isfinite(M)
    w = np.where(np.isfinite(lse), np.exp(lse - np.where(finite, M, 0.0)[None]), 0.0)
    den = w.sum(axis=0)
    num = (w[..., None] * os_).sum(axis=0)
    return np.where(den[..., None] > 0, num / np.where(den > 0, den, 1.0)[..., None], 0.0)


def attention_split(ring, q: np.ndarray, bounds, qpos=None) -> np.ndarray:
    """``attention_exact`` computed in parts and merged: the filled slots (in
    the ring's slot order) are cut at ``bounds`` (0 = b_0 <= b_1 <= ... <= b_S
    = the number of filled slots; equal neighbours give empty parts), each
    part gives its normalised output and log-sum-exp, and ``merge_parts_f64``
    combines them."""
    q = np.asarray(q, dtype=np.float64)
    n = q.shape[0]
    if qpos is None:
        qpos = ring.next_pos - n + np.arange(n)
    qt = ring.rope_f64(q, qpos)
    k, v, _ = ring.dequantised()
    b = [int(x) for x in bounds]
    if b[0] != 0 or b[-1] != k.shape[1] or any(x > y for x, y in zip(b, b[1:])):
        raise ValueError(f"bounds {b} do not cut the {k.shape[1]} filled slots")
    parts = [attention_part_f64(qt, k[:, b0:b1], v[:, b0:b1]) for b0, b1 in zip(b, b[1:])]
    return merge_parts_f64(parts)


def attention_linear_window(history, q, qpos, ring) -> np.ndarray:
    """Brute force over the last ``capacity`` written tokens in time order.

    ``history`` is a list of (k_codes [n,H,d], v_codes [n,H,d], positions)
    as they were quantised at write time.  Uses the ring's scales.
    """
    kc = np.concatenate([h[0] for h in history], axis=0)
    vc = np.concatenate([h[1] for h in history], axis=0)
    kc = kc[-ring.C:]
    vc = vc[-ring.C:]
    k = e4m3.decode(kc).transpose(1, 0, 2) * ring.scale_k.astype(np.float64)[:, None, None]
    v = e4m3.decode(vc).transpose(1, 0, 2) * ring.scale_v.astype(np.float64)[:, None, None]
    qt = rotate_f64(np.asarray(q, np.float64), np.asarray(qpos, np.int64), ring.table.theta)
    return softmax_attention_f64(qt, k, v)


def attention_positions_by_slot_order(raw_k, raw_v, n_valid, q, qpos, th,
                                      first_position: int = 0) -> np.ndarray:
    """The combination the page pins as invalid: keys cached without rotation
    in a ring, rotated at read time with positions assigned by slot order
    (slot j gets ``first_position + j``).

    raw_k, raw_v float64 [H, C, d] (unrotated, unquantised); uses slots
    [0, n_valid).  Correct only while slot order equals time order.
    """
    k = raw_k[:, :n_valid, :]
    v = raw_v[:, :n_valid, :]
    pos = first_position + np.arange(n_valid)
    kt = rotate_f64(k.transpose(1, 0, 2), pos, th).transpose(1, 0, 2)
    qt = rotate_f64(np.asarray(q, np.float64), np.asarray(qpos, np.int64), th)
    return softmax_attention_f64(qt, kt, v)


def attention_true_positions(raw_k, raw_v, slot_pos, q, qpos, th) -> np.ndarray:
    """Same raw ring, each slot rotated by its own recorded position."""
    sl = np.nonzero(np.asarray(slot_pos) != INT32_MIN)[0]
    k = raw_k[:, sl, :]
    v = raw_v[:, sl, :]
    kt = rotate_f64(k.transpose(1, 0, 2), np.asarray(slot_pos)[sl], th).transpose(1, 0, 2)
    qt = rotate_f64(np.asarray(q, np.float64), np.asarray(qpos, np.int64), th)
    return softmax_attention_f64(qt, kt, v)


def _split_terms(u: np.ndarray, m: int):
    """Split float values into m FP8 terms by successive residuals."""
    terms = []
    r = u.astype(np.float32)
    for _ in range(m):
        c = e4m3.decode(e4m3.encode(r))
        terms.append(c)
        r = (r - c.astype(np.float32)).astype(np.float32)
    return terms


def attention_emulated(ring, q, qpos=None, q_terms=1, p_terms=1, tile=128,
                       p_shift=7.0, tau=1.5) -> np.ndarray:
    """Diagnostic: the CUDA kernel's quantisation choices, in float64.

    q_terms may be an int or a per-head sequence.  p_terms is the number of
    E4M3 terms of the probabilities (1 or 2; the normaliser then sums the
    same FP8 values), or "f16": probabilities rounded to IEEE half precision
    for the value product while the normaliser sums the unrounded values, or
    "f16x2": the same with two half-precision terms, the rounded value and
    the rounding of what it left (p - hi taken in float32, where it is exact).
    """
    q = np.asarray(q, dtype=np.float64)
    n, H, d = q.shape
    if qpos is None:
        qpos = ring.next_pos - n + np.arange(n)
    qt = ring.rope_f64(q, qpos).astype(np.float32)
    amax = np.abs(qt).max(axis=2)                                # [n, H]
    sq = (amax / np.float32(448.0)).astype(np.float32)
    sq = np.where(sq >= np.float32(2.0 ** -126), sq, np.float32(1.0)).astype(np.float32)
    invq = (np.float32(1.0) / sq).astype(np.float32)
    u = (qt * invq[:, :, None]).astype(np.float32)
    qt_terms = np.broadcast_to(np.asarray(q_terms), (H,))
    p_f16 = isinstance(p_terms, str)
    if p_f16 and p_terms not in ("f16", "f16x2"):
        raise ValueError(p_terms)
    pt_terms = None if p_f16 else np.broadcast_to(np.asarray(p_terms), (H,))
    out = np.zeros((n, H, d), dtype=np.float64)
    nv = ring.n_valid
    log2e = 1.0 / math.log(2.0)
    for h in range(H):
        qsum = sum(_split_terms(u[:, h, :], int(qt_terms[h])))   # float64 [n, d]
        kc = e4m3.decode(ring.K[h, :nv, :])
        vc = e4m3.decode(ring.V[h, :nv, :])
        f = (sq[:, h].astype(np.float64) * float(ring.scale_k[h]) * log2e / math.sqrt(d))
        m = np.full(n, -np.inf)
        O = np.zeros((n, d))
        ell = np.zeros(n)
        for j0 in range(0, nv, tile):
            x = (qsum @ kc[j0:j0 + tile].T) * f[:, None]
            mt = x.max(axis=1)
            upd = (mt > m + tau) | ~np.isfinite(m)
            alpha = np.where(upd & np.isfinite(m), np.exp2(m - mt), 1.0)
            alpha = np.where(np.isfinite(m), alpha, 0.0)
            m = np.where(upd, mt, m)
            O *= alpha[:, None]
            ell *= alpha
            p = np.exp2(x - m[:, None] + p_shift).astype(np.float32)
            if p_f16:
                hi = p.astype(np.float16)
                pv = hi.astype(np.float64)
                if p_terms == "f16x2":
                    lo = (p - hi.astype(np.float32)).astype(np.float16)
                    pv = pv + lo.astype(np.float64)
                O += pv @ vc[j0:j0 + tile]
                ell += p.astype(np.float64).sum(axis=1)
            else:
                ps = sum(_split_terms(p, int(pt_terms[h])))
                O += ps @ vc[j0:j0 + tile]
                ell += ps.sum(axis=1)
        out[:, h, :] = np.where(ell[:, None] > 0, O / np.maximum(ell, 1e-300)[:, None], 0.0) \
            * float(ring.scale_v[h])
    return out
