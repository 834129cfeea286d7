"""The kernels' E4M3 conversion against the oracle codec (OCP OFP8 E4M3,
round to nearest even, saturating): all bf16 bit patterns, every fp32
exponent with every kept-mantissa / guard / sticky combination, and random
fp32 values."""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import e4m3

pytestmark = pytest.mark.gpu


def _gpu_codes(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).cuda()
    out = kv.encode_e4m3(t)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_all_finite_bf16_patterns():
    b = np.arange(65536, dtype=np.uint32)
    x = (b << 16).view(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(_gpu_codes(x), e4m3.encode(x))


def test_every_exponent_and_rounding_class():
    exps = np.arange(0, 255, dtype=np.uint32)                  # finite exponents incl. denormals
    top = np.arange(16, dtype=np.uint32)                        # 3 kept bits + guard bit
    sticky = np.array([0, 1, 0x40000, 0x7FFFF, 0x2AAAA], dtype=np.uint32)
    e, t, s = np.meshgrid(exps, top, sticky, indexing="ij")
    bits = (e << 23) | (t << 19) | s
    bits = np.concatenate([bits.ravel(), bits.ravel() | 0x80000000])
    x = bits.view(np.float32)
    assert np.array_equal(_gpu_codes(x), e4m3.encode(x))


def test_random_float32():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(4_000_000) * np.exp2(rng.integers(-20, 14, 4_000_000))).astype(np.float32)
    assert np.array_equal(_gpu_codes(x), e4m3.encode(x))


def test_odd_length_tail():
    x = np.array([1.0, -3.0, 500.0], dtype=np.float32)
    assert list(_gpu_codes(x)) == list(e4m3.encode(x))


def test_every_float32_pattern_against_the_library_cast():
    """All 2^32 fp32 bit patterns but NaNs, in chunks on the device, against
    torch's E4M3 cast after clamping to +-448 (the library routine the
    oracle codec agrees with on every bf16 pattern and on random fp32):
    saturation, infinities, subnormals and signed zeros included."""
    chunk = 1 << 28
    mismatches = 0
    for c in range(1 << 32 >> 28):
        bits = torch.arange(c * chunk, (c + 1) * chunk, dtype=torch.int64, device="cuda")
        bits = torch.where(bits >= 1 << 31, bits - (1 << 32), bits).to(torch.int32)
        x = bits.view(torch.float32)
        del bits
        ours = kv.encode_e4m3(x)
        ref = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        keep = ~torch.isnan(x)
        mismatches += int(((ours != ref) & keep).sum().item())
        del x, ours, ref, keep
    torch.cuda.synchronize()
    assert mismatches == 0
