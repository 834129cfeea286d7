"""Seeded synthetic inputs for the rolling FP8 attention cache.

This module only draws random numbers and packs them as bf16 bit patterns.
It holds none of the cache's arithmetic (no RoPE, no quantisation, no ring
indexing, no attention), so both the CPU oracle and the CUDA path can take
their inputs from here without sharing any of the method.

Workloads follow the shapes of the serving system in "Runway Characters:
Serving a 57B Video Diffusion Transformer for Real-Time Conversation",
section "Where the Time Went": every attention call reads a cache of 5,788
slots of which 757 are new, 60 blocks, 4 passes per step.  Head count and
head size are not on the pages; 10 heads of 128 (40 heads split four ways)
is the assumed production split.

bf16 tensors are carried as ``numpy.uint16`` bit patterns (numpy has no
bf16 type); ``to_torch_bf16`` reinterprets them for the GPU side.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "RingShape", "TINY", "PROD", "STRESS",
    "bf16_from_f32", "f32_from_bf16", "to_torch_bf16",
    "log_uniform", "frame", "tiny_session", "prod_session",
    "stress_prompt_length", "ROPE_BASE",
]

ROPE_BASE = 10000.0


@dataclass(frozen=True)
class RingShape:
    heads: int
    head_dim: int
    capacity: int
    tokens: int          # new tokens written per frame
    queries: int         # queries per attention call
    max_position: int    # rows of the RoPE table
    rope_base: float = ROPE_BASE


# Tiny: 2 heads of 64, 48 slots, 12 tokens per frame, 10 frames (wraps twice).
TINY = RingShape(heads=2, head_dim=64, capacity=48, tokens=12, queries=12,
                 max_position=256)
# Production-shaped call: 10 heads of 128, 5,788 slots, 757 new per frame.
PROD = RingShape(heads=10, head_dim=128, capacity=5788, tokens=757,
                 queries=757, max_position=40960)
# Stress: the whole unsharded head set.
STRESS = RingShape(heads=40, head_dim=128, capacity=5788, tokens=757,
                   queries=757, max_position=40960)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def f32_from_bf16(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_torch_bf16(b: np.ndarray):
    """Reinterpret uint16 bf16 bit patterns as a CPU ``torch.bfloat16`` tensor."""
    import torch
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)


def log_uniform(rng: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    """n values whose logarithm is uniform on [log lo, log hi]."""
    return np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))


def frame(rng: np.random.Generator, shape: RingShape, n: int,
          sigma_k=None, sigma_v=None, sigma_q=None, dist: str = "normal",
          nu: float = 3.0):
    """One frame of bf16 (q, k, v), each ``[n, heads, head_dim]`` uint16.

    ``sigma_*`` are per-head multipliers (None = 1).  ``dist`` is "normal"
    (standard normal draws) or "student_t" (Student-t with ``nu`` degrees of
    freedom, heavy tailed).
    """
    H, d = shape.heads, shape.head_dim

    def draw():
        if dist == "normal":
            return rng.standard_normal((n, H, d))
        if dist == "student_t":
            return rng.standard_t(nu, size=(n, H, d))
        raise ValueError(dist)

    def scaled(sig):
        x = draw()
        if sig is not None:
            x = x * np.asarray(sig, dtype=np.float64)[None, :, None]
        return bf16_from_f32(x.astype(np.float32))

    q = scaled(sigma_q)
    k = scaled(sigma_k)
    v = scaled(sigma_v)
    return q, k, v


def tiny_session(seed: int = 1, frames: int = 10):
    """Tiny workload: ``frames`` frames of N(0,1) q/k/v for the TINY shape.

    Positions are frame_idx * 12 + token_idx; the caller applies them.
    """
    rng = np.random.default_rng(seed)
    return [frame(rng, TINY, TINY.tokens) for _ in range(frames)]


def prod_session(seed: int = 2, frames: int = 9, shape: RingShape = PROD,
                 lo: float = 0.25, hi: float = 4.0):
    """Production-shaped workload.

    Per-head standard deviations for K and V are drawn independently,
    log-uniform on [lo, hi]; Q is N(0,1).  Returns (sigma_k, sigma_v, frames).
    """
    rng = np.random.default_rng(seed)
    sigma_k = log_uniform(rng, shape.heads, lo, hi)
    sigma_v = log_uniform(rng, shape.heads, lo, hi)
    fr = [frame(rng, shape, shape.tokens, sigma_k, sigma_v) for _ in range(frames)]
    return sigma_k, sigma_v, fr


def stress_prompt_length(seed: int = 5) -> int:
    """First-forward prompt length for the stress workload, uniform in [100, 2000]."""
    return int(np.random.default_rng(seed).integers(100, 2001))


# ---------------------------------------------------------------------------
# Device-side draws for the large workloads (full step, reset cycle, stress):
# a seeded torch CUDA generator, bf16 tensors [n, H, d] on the GPU.  Only
# random numbers and the bf16 cast; nothing of the cache's arithmetic.
def cuda_generator(seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def cuda_frame(gen, heads: int, head_dim: int, n: int, sigma_k=None, sigma_v=None,
               dist: str = "normal", device="cuda"):
    """(q, k, v) bf16 [n, heads, head_dim] on the GPU.

    dist "normal": N(0,1) draws; "student_t3": Student-t with 3 degrees of
    freedom, built as z / sqrt((z1^2 + z2^2 + z3^2) / 3) from standard normals.
    sigma_k / sigma_v scale each head (None = 1).
    """
    import torch

    def draw():
        z = torch.randn((n, heads, head_dim), generator=gen, device=device)
        if dist == "normal":
            return z
        if dist == "student_t3":
            c = torch.randn((3, n, heads, head_dim), generator=gen, device=device)
            return z / torch.sqrt((c * c).sum(0) / 3.0)
        raise ValueError(dist)

    def scaled(sig):
        x = draw()
        if sig is not None:
            x = x * torch.as_tensor(sig, dtype=torch.float32, device=device)[None, :, None]
        return x.to(torch.bfloat16).contiguous()

    q = scaled(None)
    k = scaled(sigma_k)
    v = scaled(sigma_v)
    return q, k, v
