"""Python binding of the kvring C ABI (``include/kvring.h``).

Argument marshalling only: every step of the cache's arithmetic runs in the
CUDA kernels of ``libkvring.so``.  PyTorch supplies device memory (one
``uint8`` buffer per ring, allocated once), streams and tensors.  There is
no CPU path: if the library is not built, or no sm_103a GPU is present,
calls raise.

The functions carry the C names (``kvring_create``, ``kvring_calibrate_scales``,
``kvring_write_frame``, ``kvring_delta_rotate``, ``kvring_attention``,
``kvring_export``); ``KvRing`` wraps them for one layer's cache.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

__all__ = [
    "KvRing", "KvRingError", "TO_OLDEST", "lib", "library_path", "header_functions",
    "kvring_required_bytes", "kvring_create", "kvring_destroy", "kvring_calibrate_scales",
    "kvring_write_frame", "kvring_delta_rotate", "kvring_attention", "kvring_attention_noalloc",
    "kvring_write_frames_many", "kvring_delta_rotate_many", "write_frames_many", "delta_rotate_many",
    "kvring_legacy_upkeep", "LegacyWindows", "kvring_project_write",
    "kvring_export",
    "kvring_status_string", "encode_e4m3", "STATE",
]

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
HEADER = os.path.join(ROOT, "include", "kvring.h")

TO_OLDEST = -1
OUT_F32, OUT_BF16 = 0, 1
STATE = dict(head=0, n_valid=1, total_lo=2, total_hi=3, next_pos=4, calibrated=5, error=6,
             last_delta=7)
STATE_WORDS = 8
DEVERR_POSITION, DEVERR_TIMEOUT, DEVERR_DELTA = 1, 2, 4
PROJECT_WRITE, PROJECT_STORE_KV = 1, 2


class KvringConfig(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32),
        ("max_position", ctypes.c_int32),
        ("max_kv_splits", ctypes.c_int32),
        ("attn_precision", ctypes.c_int32),
        ("pinned_prefix", ctypes.c_int32),
        ("rope_pairs_t", ctypes.c_int32),
        ("rope_pairs_y", ctypes.c_int32),
        ("rope_base", ctypes.c_double),
    ]


class KvRingError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {kvring_status_string(status)} (status {status})")


_LIB = None


def library_path() -> str:
    return os.path.join(HERE, "libkvring.so")


def lib():
    """Load libkvring.so (built in-tree by ``ring_kv_cache_gb300.build``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m ring_kv_cache_gb300.build`")
    L = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(KvringConfig)
    sig = {
        "kvring_required_bytes": (sz, [cfgp]),
        "kvring_create": (i32, [cfgp, vp, sz, vp, ctypes.POINTER(vp)]),
        "kvring_destroy": (i32, [vp]),
        "kvring_calibrate_scales": (i32, [vp, vp, vp, vp, i32, vp]),
        "kvring_write_frame": (i32, [vp, vp, vp, vp, i32, vp]),
        "kvring_delta_rotate": (i32, [vp, i32, vp]),
        "kvring_write_frames_many": (i32, [vp, i32, vp, vp, vp, i32, vp]),
        "kvring_legacy_upkeep": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, vp]),
        "kvring_delta_rotate_many": (i32, [vp, i32, i32, vp]),
        "kvring_attention": (i32, [vp, vp, vp, i32, vp, i32, vp]),
        "kvring_attention_noalloc": (i32, [vp, vp, vp, i32, vp, i32, vp]),
        "kvring_project_write": (i32, [vp, vp, vp, i32, vp, i32, vp, vp, i32, vp]),
        "kvring_export": (i32, [vp, vp, vp, vp, vp, vp, vp]),
        "kvring_debug_encode_e4m3": (i32, [vp, vp, i64, vp]),
        "kvring_debug_attention_levels": (i32, [vp, vp, vp]),
        "kvring_debug_set_attention_wait": (i32, [vp, i64, i32]),
        "kvring_debug_write_floor": (i32, [vp, i32, vp]),
        "kvring_debug_late_reads": (i64, []),
        "kvring_debug_attention_guess": (i32, [vp, i32]),
        "kvring_status_string": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _LIB = L
    return L


def header_functions() -> list[str]:
    """Names of the functions declared in include/kvring.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(kvring_\w+)\s*\(", text, re.M)))


def kvring_status_string(status: int) -> str:
    return lib().kvring_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise KvRingError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _tokens(x: torch.Tensor, heads: int, dim: int, name: str, device=None) -> int:
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and x.device != device:
        raise ValueError(f"{name} is on {x.device}, the ring on {device}")
    if x.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if x.dim() != 3 or x.shape[1] != heads or x.shape[2] != dim:
        raise ValueError(f"{name} must have shape [n, {heads}, {dim}], got {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x.shape[0]


def _positions(pos, n: int, name: str, three_d: bool = False, device=None):
    """Check a position tensor: int32 [n] (1-D RoPE) or [n, 3] = (t, y, x)."""
    if pos is None:
        if three_d:
            raise ValueError(f"{name}: 3-D RoPE needs explicit (t, y, x) positions")
        return None
    shape = (n, 3) if three_d else (n,)
    if not isinstance(pos, torch.Tensor) or not pos.is_cuda or pos.dtype != torch.int32 \
            or tuple(pos.shape) != shape or not pos.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor of shape {shape}")
    if device is not None and pos.device != device:
        raise ValueError(f"{name} is on {pos.device}, the ring on {device}")
    return pos


# ---------------------------------------------------------------------------
# C-named functions (marshalling only)
# ---------------------------------------------------------------------------
def make_config(heads, head_dim, capacity, max_tokens, max_position, rope_base=10000.0,
                max_kv_splits=16, attn_precision=0, pinned_prefix=0, rope3d=None) -> KvringConfig:
    pt, py = (0, 0) if rope3d is None else (int(rope3d[0]), int(rope3d[1]))
    return KvringConfig(int(heads), int(head_dim), int(capacity), int(max_tokens),
                        int(max_position), int(max_kv_splits), int(attn_precision),
                        int(pinned_prefix), pt, py, float(rope_base))


def kvring_required_bytes(cfg: KvringConfig) -> int:
    return int(lib().kvring_required_bytes(ctypes.byref(cfg)))


def kvring_create(cfg: KvringConfig, buf: torch.Tensor, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(lib().kvring_create(ctypes.byref(cfg), buf.data_ptr(), buf.numel() * buf.element_size(),
                               _stream_ptr(stream, buf.device), ctypes.byref(h)), "kvring_create")
    return h.value


def kvring_destroy(handle: int) -> None:
    _check(lib().kvring_destroy(handle), "kvring_destroy")


def kvring_calibrate_scales(handle, k, v, pos, n, stream_ptr) -> None:
    _check(lib().kvring_calibrate_scales(handle, _ptr(k), _ptr(v), _ptr(pos), int(n), stream_ptr),
           "kvring_calibrate_scales")


def kvring_write_frame(handle, k, v, pos, n, stream_ptr) -> None:
    _check(lib().kvring_write_frame(handle, _ptr(k), _ptr(v), _ptr(pos), int(n), stream_ptr),
           "kvring_write_frame")


def kvring_delta_rotate(handle, delta, stream_ptr) -> None:
    _check(lib().kvring_delta_rotate(handle, int(delta), stream_ptr), "kvring_delta_rotate")


def _ptr_array(values):
    arr = (ctypes.c_void_p * len(values))()
    for i, x in enumerate(values):
        arr[i] = x
    return arr


def kvring_write_frames_many(handles, ks, vs, poss, n, stream_ptr) -> None:
    """Batched write: host arrays of ring handles and device pointers."""
    m = len(handles)
    pos_arr = None if poss is None else _ptr_array([_ptr(p) for p in poss])
    _check(lib().kvring_write_frames_many(_ptr_array(handles), m, _ptr_array([_ptr(k) for k in ks]),
                                          _ptr_array([_ptr(v) for v in vs]), pos_arr, int(n), stream_ptr),
           "kvring_write_frames_many")


def kvring_delta_rotate_many(handles, delta, stream_ptr) -> None:
    _check(lib().kvring_delta_rotate_many(_ptr_array(handles), len(handles), int(delta), stream_ptr),
           "kvring_delta_rotate_many")


def write_frames_many(rings, ks, vs, poss=None, stream=None) -> None:
    """kvring_write_frame on several rings of one shape in one launch."""
    if not rings or len(ks) != len(rings) or len(vs) != len(rings) or (poss is not None and len(poss) != len(rings)):
        raise ValueError("one k, v (and pos) per ring")
    r0 = rings[0]
    n = _tokens(ks[0], r0.H, r0.d, "k", r0.device)
    for i, r in enumerate(rings):
        if r.device != r0.device:
            raise ValueError("every ring must be on one device")
        if _tokens(ks[i], r.H, r.d, "k", r.device) != n or _tokens(vs[i], r.H, r.d, "v", r.device) != n:
            raise ValueError("every k and v must hold the same number of tokens")
        if poss is not None:
            _positions(poss[i], n, "pos", r.three_d, r.device)
        elif r.three_d:
            raise ValueError("3-D RoPE needs explicit (t, y, x) positions")
    with torch.cuda.device(r0.device):
        kvring_write_frames_many([r.handle for r in rings], ks, vs, poss, n, r0._s(stream))


def delta_rotate_many(rings, delta: int = TO_OLDEST, stream=None) -> None:
    """kvring_delta_rotate on several rings of one shape in one launch."""
    if not rings:
        raise ValueError("no rings")
    if any(r.device != rings[0].device for r in rings):
        raise ValueError("every ring must be on one device")
    with torch.cuda.device(rings[0].device):
        kvring_delta_rotate_many([r.handle for r in rings], delta, rings[0]._s(stream))


def kvring_legacy_upkeep(handle, wk_in, wv_in, wk_out, wv_out, k, v, n, stream_ptr) -> None:
    _check(lib().kvring_legacy_upkeep(handle, _ptr(wk_in), _ptr(wv_in), _ptr(wk_out), _ptr(wv_out), _ptr(k),
                                      _ptr(v), int(n), stream_ptr), "kvring_legacy_upkeep")


class LegacyWindows:
    """The two bf16 window buffer pairs the legacy upkeep alternates between."""

    def __init__(self, ring: "KvRing"):
        shape = (ring.C, ring.H, ring.d)
        self.ring = ring
        self.k = [torch.zeros(shape, dtype=torch.bfloat16, device=ring.device) for _ in range(2)]
        self.v = [torch.zeros(shape, dtype=torch.bfloat16, device=ring.device) for _ in range(2)]
        self.cur = 0

    def upkeep(self, k, v, stream=None) -> None:
        """One call of the original upkeep on `ring` with the frame (k, v)."""
        r = self.ring
        n = _tokens(k, r.H, r.d, "k", r.device)
        if _tokens(v, r.H, r.d, "v", r.device) != n:
            raise ValueError("k and v must hold the same number of tokens")
        a, b = self.cur, 1 - self.cur
        with torch.cuda.device(r.device):
            kvring_legacy_upkeep(r.handle, self.k[a], self.v[a], self.k[b], self.v[b], k, v, n, r._s(stream))
        self.cur = b

    def window(self):
        """The current (k, v) bf16 windows [capacity, H, d]."""
        return self.k[self.cur], self.v[self.cur]


def kvring_attention(handle, q, qpos, n_q, out, out_dtype, stream_ptr) -> None:
    _check(lib().kvring_attention(handle, _ptr(q), _ptr(qpos), int(n_q), _ptr(out), int(out_dtype),
                                  stream_ptr), "kvring_attention")


def kvring_attention_noalloc(handle, q, qpos, n_q, out, out_dtype, stream_ptr) -> None:
    _check(lib().kvring_attention_noalloc(handle, _ptr(q), _ptr(qpos), int(n_q), _ptr(out),
                                          int(out_dtype), stream_ptr), "kvring_attention_noalloc")


def kvring_project_write(handle, x, w, d_model, pos, n, q_out, kv_out, flags, stream_ptr) -> None:
    _check(lib().kvring_project_write(handle, _ptr(x), _ptr(w), int(d_model), _ptr(pos), int(n), _ptr(q_out),
                                      _ptr(kv_out), int(flags), stream_ptr), "kvring_project_write")


def kvring_export(handle, k_out, v_out, scales, slot_pos, state, stream_ptr) -> None:
    _check(lib().kvring_export(handle, _ptr(k_out), _ptr(v_out), _ptr(scales), _ptr(slot_pos),
                               _ptr(state), stream_ptr), "kvring_export")


def late_reads() -> int:
    """How many write and attention calls so far read their frame or queries
    after waiting for the preceding kernel, because the library's previous
    kernel on their stream writes a buffer overlapping them."""
    return int(lib().kvring_debug_late_reads())


def encode_e4m3(x: torch.Tensor, stream=None) -> torch.Tensor:
    """E4M3 codes of a CUDA float32 tensor, with the kernels' conversion (test support)."""
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().kvring_debug_encode_e4m3(x.data_ptr(), out.data_ptr(), x.numel(),
                                          _stream_ptr(stream, x.device)), "kvring_debug_encode_e4m3")
    return out


# ---------------------------------------------------------------------------
class KvRing:
    """One layer's rolling FP8 attention cache on one CUDA device (the
    current one unless ``device`` names another).  Every call runs with that
    device current and takes tensors on it.  The ring's buffer is freed with
    the object: keep it alive until the work enqueued on it has completed."""

    def __init__(self, heads: int, head_dim: int, capacity: int, max_tokens: int,
                 max_position: int, rope_base: float = 10000.0, max_kv_splits: int = 16,
                 attn_precision: int = 0, device=None, stream=None, pinned_prefix: int = 0,
                 rope3d=None):
        if not torch.cuda.is_available():
            raise RuntimeError("KvRing needs a CUDA device")
        d = torch.device(device) if device is not None else torch.device("cuda")
        if d.type != "cuda":
            raise ValueError("KvRing needs a CUDA device")
        self.device = d if d.index is not None else torch.device("cuda", torch.cuda.current_device())
        self.H, self.d, self.C = int(heads), int(head_dim), int(capacity)
        self.max_tokens = int(max_tokens)
        self.P = int(pinned_prefix)
        self.three_d = rope3d is not None
        self.cfg = make_config(heads, head_dim, capacity, max_tokens, max_position, rope_base,
                               max_kv_splits, attn_precision, pinned_prefix, rope3d)
        n = kvring_required_bytes(self.cfg)
        if n == 0:
            raise ValueError("invalid kvring config")
        self.nbytes = n
        with torch.cuda.device(self.device):
            self.buf = torch.empty(n, dtype=torch.uint8, device=self.device)
            self.handle = kvring_create(self.cfg, self.buf, stream)

    def _s(self, stream) -> int:
        return _stream_ptr(stream, self.device)

    def calibrate(self, k, v, pos=None, stream=None) -> None:
        n = _tokens(k, self.H, self.d, "k", self.device)
        if _tokens(v, self.H, self.d, "v", self.device) != n:
            raise ValueError("k and v must hold the same number of tokens")
        pos = _positions(pos, n, "pos", self.three_d, self.device)
        with torch.cuda.device(self.device):
            kvring_calibrate_scales(self.handle, k, v, pos, n, self._s(stream))

    def write(self, k, v, pos=None, stream=None) -> None:
        n = _tokens(k, self.H, self.d, "k", self.device)
        if _tokens(v, self.H, self.d, "v", self.device) != n:
            raise ValueError("k and v must hold the same number of tokens")
        pos = _positions(pos, n, "pos", self.three_d, self.device)
        with torch.cuda.device(self.device):
            kvring_write_frame(self.handle, k, v, pos, n, self._s(stream))

    def delta_rotate(self, delta: int = TO_OLDEST, stream=None) -> None:
        with torch.cuda.device(self.device):
            kvring_delta_rotate(self.handle, delta, self._s(stream))

    def attention(self, q, qpos=None, out=None, out_dtype=torch.float32, stream=None) -> torch.Tensor:
        n = _tokens(q, self.H, self.d, "q", self.device)
        if out is None:
            out = torch.empty((n, self.H, self.d), dtype=out_dtype, device=self.device)
        if out.dtype not in (torch.float32, torch.bfloat16) or tuple(out.shape) != (n, self.H, self.d) \
                or not out.is_contiguous() or not out.is_cuda or out.device != self.device:
            raise ValueError("out must be a contiguous float32/bfloat16 tensor [n_q, H, d] on the ring's device")
        qpos = _positions(qpos, n, "qpos", self.three_d, self.device)
        with torch.cuda.device(self.device):
            kvring_attention(self.handle, q, qpos, n, out,
                             OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32, self._s(stream))
        return out

    def project_write(self, x, w, pos=None, write=True, store_kv=False, q_out=None, kv_out=None,
                      stream=None):
        """QKV projection of one frame with the cache write fused in
        (kvring_project_write): x bf16 [n, d_model], w bf16 [3 H d, d_model]
        (a linear layer's weight); returns (q_out bf16 [n, H, d], kv_out bf16
        [2, n, H, d] or None).  With ``write`` the keys and values enter the
        ring as kvring_write_frame would write them; ``store_kv`` also returns
        them (e.g. to calibrate a session from its first frame)."""
        for t, name in ((x, "x"), (w, "w")):
            if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 2 \
                    or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"{name} must be a contiguous 2-D bfloat16 tensor on {self.device}")
        n, dm = x.shape
        if dm < 64 or dm % 64:
            raise ValueError("d_model must be a positive multiple of 64")
        if tuple(w.shape) != (3 * self.H * self.d, dm):
            raise ValueError(f"w must have shape [{3 * self.H * self.d}, {dm}], got {tuple(w.shape)}")
        if pos is not None or (write and self.three_d):
            pos = _positions(pos, n, "pos", self.three_d, self.device)
        if q_out is None:
            q_out = torch.empty((n, self.H, self.d), dtype=torch.bfloat16, device=self.device)
        _tokens(q_out, self.H, self.d, "q_out", self.device)
        if store_kv:
            if kv_out is None:
                kv_out = torch.empty((2, n, self.H, self.d), dtype=torch.bfloat16, device=self.device)
            if kv_out.dtype != torch.bfloat16 or tuple(kv_out.shape) != (2, n, self.H, self.d) \
                    or not kv_out.is_contiguous() or kv_out.device != self.device:
                raise ValueError("kv_out must be a contiguous bfloat16 tensor [2, n, H, d] on the ring's device")
        flags = (PROJECT_WRITE if write else 0) | (PROJECT_STORE_KV if store_kv else 0)
        with torch.cuda.device(self.device):
            kvring_project_write(self.handle, x, w, dm, pos, n, q_out, kv_out if store_kv else None, flags,
                                 self._s(stream))
        return q_out, (kv_out if store_kv else None)

    def export(self, stream=None) -> dict:
        """Device copies of the cache, scales, positions and state (stream-ordered)."""
        dev = self.device
        k = torch.empty((self.H, self.C, self.d), dtype=torch.uint8, device=dev)
        v = torch.empty_like(k)
        scales = torch.empty(4 * self.H, dtype=torch.float32, device=dev)
        slot_pos = torch.empty(self.C, dtype=torch.int32, device=dev)
        state = torch.empty(STATE_WORDS, dtype=torch.int32, device=dev)
        with torch.cuda.device(dev):
            kvring_export(self.handle, k, v, scales, slot_pos, state, self._s(stream))
        return dict(k=k, v=v, scales=scales, slot_pos=slot_pos, state=state)

    def levels(self, stream=None) -> torch.Tensor:
        qt = (self.max_tokens + 127) // 128
        out = torch.empty((qt, self.H), dtype=torch.int32, device=self.device)
        with torch.cuda.device(self.device):
            _check(lib().kvring_debug_attention_levels(self.handle, out.data_ptr(), self._s(stream)),
                   "kvring_debug_attention_levels")
        return out

    def write_floor(self, n: int, stream=None) -> None:
        """Measurement support: the write's fixed cost for n tokens, no data
        (see the C header); the ring is left unchanged."""
        with torch.cuda.device(self.device):
            _check(lib().kvring_debug_write_floor(self.handle, int(n), self._s(stream)),
                   "kvring_debug_write_floor")

    def set_attention_guess(self, wrong: bool = False) -> None:
        """Test support: make the attention's early guess of the default
        query positions wrong on purpose (kvring_debug_attention_guess)."""
        _check(lib().kvring_debug_attention_guess(self.handle, int(bool(wrong))), "kvring_debug_attention_guess")

    def set_attention_wait(self, limit_ns: int = 1_000_000_000, stall: bool = False) -> None:
        """Test support: the attention kernel's wait limit, and a stall that
        makes its first wait give up on purpose (see the C header)."""
        _check(lib().kvring_debug_set_attention_wait(self.handle, int(limit_ns), int(bool(stall))),
               "kvring_debug_set_attention_wait")

    def close(self) -> None:
        if getattr(self, "handle", None):
            kvring_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
