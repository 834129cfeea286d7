"""Host-only checks of the C ABI: the library loads, exports every function
that include/kvring.h declares, sizes its buffer as documented and rejects
bad configs.  No GPU and no compute call is needed."""
import ctypes

import pytest

import ring_kv_cache_gb300 as kv


@pytest.fixture(scope="module")
def L():
    try:
        return kv.lib()
    except RuntimeError as e:  # not built yet in this checkout
        pytest.fail(str(e))


def test_header_declares_the_boundary():
    names = kv.header_functions()
    for want in ["kvring_create", "kvring_calibrate_scales", "kvring_write_frame",
                 "kvring_delta_rotate", "kvring_attention", "kvring_required_bytes",
                 "kvring_destroy", "kvring_export", "kvring_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in kv.header_functions():
        assert hasattr(L, name), name


def test_required_bytes_matches_layout(L):
    cfg = kv.make_config(10, 128, 5788, 757, 40960, max_kv_splits=8)
    n = kv.kvring_required_bytes(cfg)
    H, D, C, Q, S = 10, 128, 5788, 6, 8
    a = lambda x: (x + 255) // 256 * 256
    # up to 8 splits merge in a thread-block cluster: no split partials
    want = (a(H * C * D) * 2 + a(4 * C) + a(16 * H) + a(64) + a(8 * H) + a(40960 * D * 4)
            + a(Q * H * 4) * 2)
    assert n == want
    cfg = kv.make_config(10, 128, 5788, 757, 40960, max_kv_splits=16)
    S = 16
    want += a(S * Q * H * 128 * D * 4) + a(S * Q * H * 128 * 4)
    assert kv.kvring_required_bytes(cfg) == want


@pytest.mark.parametrize("field,value", [
    ("num_heads", 0), ("head_dim", 96), ("capacity", 0), ("max_tokens", 0),
    ("max_position", 0), ("max_kv_splits", 0), ("attn_precision", 5),
    ("pinned_prefix", -1), ("pinned_prefix", 48),
    ("rope_pairs_t", 4), ("rope_pairs_t", 40), ("rope_pairs_y", 8), ("rope_pairs_t", 12),
    ("rope_base", 0.0), ("rope_base", float("inf")),
])
def test_bad_configs_are_rejected(L, field, value):
    cfg = kv.make_config(2, 64, 48, 12, 256)
    assert kv.kvring_required_bytes(cfg) > 0
    setattr(cfg, field, value)
    assert kv.kvring_required_bytes(cfg) == 0


def test_3d_rope_sections_are_accepted_in_whole_chunks(L):
    for sec in [(8, 8), (16, 0), (8, 16), (32, 0)]:
        assert kv.kvring_required_bytes(kv.make_config(2, 64, 48, 12, 256, rope3d=sec)) > 0
    assert kv.kvring_required_bytes(kv.make_config(2, 128, 48, 12, 256, rope3d=(16, 24))) > 0
    assert kv.kvring_required_bytes(kv.make_config(2, 64, 48, 12, 256, rope3d=(8, 12))) == 0


def test_status_strings(L):
    assert kv.kvring_status_string(0) == "ok"
    assert "calibrated" in kv.kvring_status_string(2)
    assert kv.kvring_status_string(99) == "unknown status"


def test_create_rejects_null_arguments_without_touching_the_gpu(L):
    cfg = kv.make_config(2, 64, 48, 12, 256)
    out = ctypes.c_void_p()
    assert L.kvring_create(ctypes.byref(cfg), None, 1 << 20, None, ctypes.byref(out)) == 1
    assert L.kvring_create(ctypes.byref(cfg), 0x1001, 1 << 20, None, ctypes.byref(out)) == 1
    assert L.kvring_create(None, 0x1000, 1 << 20, None, ctypes.byref(out)) == 1
    assert L.kvring_write_frame(None, None, None, None, 1, None) == 1
    assert L.kvring_attention(None, None, None, 1, None, 0, None) == 1
    assert L.kvring_delta_rotate(None, 0, None) == 1
