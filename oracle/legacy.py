"""The original cache upkeep, as a plain CPU model (the comparison path).

Test infrastructure only; nothing in the library imports it.

"Where the Time Went" on the Runway Characters page describes what every
attention call did before the ring: re-apply RoPE to every cached key,
re-quantise the cache to FP8 and shift the window by copying it (69.7 ms of
a 239.2 ms step, against 6.2 ms once the work moved to write time).  The
pages give no code; the readings taken here (listed in the design notes):

* the window keeps the unrotated bf16 keys and values of the last C tokens
  in time order; a call copies the window shifted by the n new tokens (the
  n oldest leave once it is full) and appends the new frame at its end;
* the key in window slot i gets RoPE at its position, base + i, where base
  is the position of the oldest token in the window (token positions are
  their index in the session, as for the ring's default positions);
* per-head scales are recomputed from the whole window at every call (amax
  of the rotated keys, of the values, over 448; a scale that is not a
  normal fp32 number becomes 1), and the whole window is quantised with
  them, with the same pinned fp32 RoPE and E4M3 conversion as the ring.

The FP8 cache it produces has slot order = time order, so the same
attention reads it.
"""
from __future__ import annotations

import numpy as np

from . import e4m3
from .ring import INT32_MIN, Ring, scale_from_amax
from .rope import Table, rotate_pinned_f32


class LegacyWindow:
    """bf16 windows (as float32 values) [C, H, d] in time order, and the FP8
    cache rebuilt from them at every call."""

    def __init__(self, heads: int, head_dim: int, capacity: int,
                 max_position: int, rope_base: float = 10000.0):
        self.H, self.d, self.C = heads, head_dim, capacity
        self.table = Table(head_dim, rope_base, max_position)
        self.k = np.zeros((capacity, heads, head_dim), dtype=np.float32)
        self.v = np.zeros((capacity, heads, head_dim), dtype=np.float32)
        self.fill = 0       # tokens in the window
        self.total = 0      # tokens seen; the next token's position
        self.K = np.zeros((heads, capacity, head_dim), dtype=np.uint8)
        self.V = np.zeros((heads, capacity, head_dim), dtype=np.uint8)
        self.slot_pos = np.full(capacity, INT32_MIN, dtype=np.int64)
        self.scale_k = np.ones(heads, dtype=np.float32)
        self.scale_v = np.ones(heads, dtype=np.float32)

    def shift_in(self, k_new: np.ndarray, v_new: np.ndarray) -> None:
        """The window copy: the n oldest tokens leave once full, the frame enters."""
        k_new = np.asarray(k_new, dtype=np.float32)
        v_new = np.asarray(v_new, dtype=np.float32)
        n = k_new.shape[0]
        if not 1 <= n <= self.C:
            raise ValueError("frame must hold 1..capacity tokens")
        keep = min(self.fill, self.C - n)              # old tokens that stay
        old_k, old_v = self.k[self.fill - keep:self.fill], self.v[self.fill - keep:self.fill]
        k = np.zeros_like(self.k)
        v = np.zeros_like(self.v)
        k[:keep], v[:keep] = old_k, old_v
        k[keep:keep + n], v[keep:keep + n] = k_new, v_new
        self.k, self.v = k, v
        self.fill = keep + n
        self.total += n

    def base(self) -> int:
        """Position of the oldest token in the window."""
        return self.total - self.fill

    def rotated_keys(self, scales=None) -> np.ndarray:
        """RoPE of every key in the window at its position (pinned fp32)."""
        pos = self.base() + np.arange(self.fill, dtype=np.int64)
        c, s = self.table.rows(pos)
        return rotate_pinned_f32(self.k[:self.fill], c[:, None, :], s[:, None, :])

    def requantise(self, scale_k=None, scale_v=None) -> None:
        """Rebuild the FP8 cache from the window.  Scales from the window's
        maxima unless given (the given form pins this model to the ring's)."""
        y = self.rotated_keys()
        v = self.v[:self.fill]
        if scale_k is None:
            scale_k = scale_from_amax(np.abs(y).max(axis=(0, 2)))
            scale_v = scale_from_amax(np.abs(v).max(axis=(0, 2)))
        self.scale_k = np.asarray(scale_k, dtype=np.float32)
        self.scale_v = np.asarray(scale_v, dtype=np.float32)
        inv_k = (np.float32(1.0) / self.scale_k).astype(np.float32)
        inv_v = (np.float32(1.0) / self.scale_v).astype(np.float32)
        f = self.fill
        self.K[:] = 0
        self.V[:] = 0
        self.K[:, :f, :] = e4m3.encode(y * inv_k[None, :, None]).transpose(1, 0, 2)
        self.V[:, :f, :] = e4m3.encode(v * inv_v[None, :, None]).transpose(1, 0, 2)
        self.slot_pos[:] = INT32_MIN
        self.slot_pos[:f] = self.base() + np.arange(f, dtype=np.int64)

    def upkeep(self, k_new: np.ndarray, v_new: np.ndarray) -> None:
        """One call of the original upkeep: shift, RoPE everything, re-quantise."""
        self.shift_in(k_new, v_new)
        self.requantise()

    def as_ring(self, max_position: int, rope_base: float = 10000.0) -> Ring:
        """An oracle Ring holding this FP8 cache (to run the attention oracle on it)."""
        r = Ring(self.H, self.d, self.C, max_position, rope_base)
        r.K[:] = self.K
        r.V[:] = self.V
        r.slot_pos[:] = self.slot_pos
        r.scale_k, r.scale_v = self.scale_k.copy(), self.scale_v.copy()
        r.inv_k = (np.float32(1.0) / r.scale_k).astype(np.float32)
        r.inv_v = (np.float32(1.0) / r.scale_v).astype(np.float32)
        r.n_valid = self.fill
        r.head = self.fill % self.C
        r.total = self.total
        r.next_pos = self.total
        r.calibrated = True
        return r
