"""Pins of the oracle's bf16 rounding against torch's CPU conversion (a
library routine) and hand-checked values."""
import numpy as np
import torch

import oracle


def _torch_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_matches_torch_random():
    rng = np.random.default_rng(5)
    f = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(1000) * 1e30).astype(np.float32),
        (rng.standard_normal(1000) * 1e-38).astype(np.float32),   # subnormals
        rng.integers(0, 2**32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    f = f[~np.isnan(f)]
    np.testing.assert_array_equal(oracle.f32_to_bf16(f), _torch_bits(f))


def test_bf16_ties_to_even_by_hand():
    # 1 + 2^-8 is halfway between bf16 1.0 (even) and 1 + 2^-7: stays 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even): up
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.0, 0.0, -0.0, 65504.0], np.float32)
    exp = np.array([0x3F80, 0x3F80, 0x3F82, 0xC000, 0x0000, 0x8000, 0x4780], np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16(vals), exp)


def test_bf16_nan_stays_nan_and_inf():
    bits = oracle.f32_to_bf16(np.array([np.nan, np.inf, -np.inf], np.float32))
    back = oracle.bf16_to_f64(bits)
    assert np.isnan(back[0]) and back[1] == np.inf and back[2] == -np.inf


def test_bf16_decode_exact():
    b = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(b)
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(got[m], ref[m])
    assert np.isnan(got[~m]).all()
