"""Pins for the oracle's binary16 / bfloat16 conversions.

The oracle converts with its own code written from the IEEE-754 format
definition; these tests pin it to numpy's float16 and torch's bfloat16 (library
routines) over every binary16 value, every rounding tie and boundary, and
random binary32 bit patterns across the whole exponent range.
"""
import numpy as np
import pytest

import oracle


def test_f16_to_f32_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f32_near_f16_boundaries():
    # every finite binary16 value, the midpoints between neighbours, and one
    # binary32 ulp either side of each midpoint
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    mids32 = mids.astype(np.float32)  # exact: a midpoint needs 12 bits
    assert np.array_equal(mids32.astype(np.float64), mids)
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(0))
    extra = np.array([65504, 65519.996, 65520, 65536, 1e6, 2.0 ** -24, 2.0 ** -25,
                      2.0 ** -25 * 1.0000001, 2.0 ** -26, 1e-30, 0.0], dtype=np.float32)
    v = np.concatenate([h.astype(np.float32), mids32, up, dn, extra])
    return np.concatenate([v, -v])


def test_f32_to_f16_ties_and_boundaries():
    x = _f32_near_f16_boundaries()
    got = oracle.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_f16_random_bit_patterns():
    rng = np.random.default_rng(12345)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f32_to_f16_nan_and_inf():
    x = np.array([np.nan, np.inf, -np.inf], dtype=np.float32)
    got = oracle.f32_to_f16(x)
    assert got[0] & 0x7C00 == 0x7C00 and got[0] & 0x3FF
    assert got[1] == 0x7C00 and got[2] == 0xFC00


def test_bf16_to_f32_matches_torch():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
