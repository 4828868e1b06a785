"""Pins for the oracle's per-token, per-head asymmetric quantizer.

LMDeploy article (devpress.csdn.net), §2.4 "KV Cache 在线量化": INT8/INT4,
min/max computed online, asymmetric. The oracle's rule is pinned by
* hand-derived rows (tests/golden/quant_rows.json),
* brute force: each stored code is the code whose dequantized value is
  nearest to the input (checked over all 2^b codes), away from exact ties,
* the error bound |x - (c S + Z)| <= S/2 (+ the fp16 rounding of zero),
* the ends: the minimum maps to code 0 and the maximum to 2^b - 1,
* scale and zero equal numpy's float16 rounding of the fp32 range / (2^b-1)
  and of the minimum,
* monotonicity in x.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_rows.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_golden_rows(case):
    D = _golden()["head_dim"]
    x = np.full(D, case["x_fill"], dtype=np.float32)
    x[: len(case["x_prefix"])] = case["x_prefix"]
    codes, sb, zb = oracle.quantize_rows(x[None], case["bits"])
    assert int(sb[0]) == int(case["scale_bits"], 16)
    assert int(zb[0]) == int(case["zero_bits"], 16)
    want = np.full(D, case["code_fill"], dtype=np.int64)
    pref = case.get("codes_prefix_clamped", case["codes_prefix"])
    want[: len(pref)] = pref
    assert np.array_equal(codes[0].astype(np.int64), want)


def _rows(n_rows, seed=11, scale=1.0, dtype="f16"):
    bits = synthetic.normal(seed, 99, 0, n_rows * 128, scale, None, dtype)
    return oracle.to_f32(bits, dtype).reshape(n_rows, 128)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype,scale", [("f16", 1.0), ("f16", 8.0), ("bf16", 0.5),
                                         ("f16", 1e-3)])
def test_nearest_code_brute_force(bits, dtype, scale):
    x = _rows(2000, scale=scale, dtype=dtype)
    codes, sb, zb = oracle.quantize_rows(x, bits)
    S = oracle.f16_to_f32(sb).astype(np.float64)[:, None]
    Z = oracle.f16_to_f32(zb).astype(np.float64)[:, None]
    qmax = (1 << bits) - 1
    allc = np.arange(qmax + 1, dtype=np.float64)
    x64 = x.astype(np.float64)
    # distance from every input to every dequantized code value
    dist = np.abs(x64[:, :, None] - (allc[None, None, :] * S[:, :, None] + Z[:, :, None]))
    best = dist.argmin(axis=2)
    srt = np.sort(dist, axis=2)
    clear = (srt[:, :, 1] - srt[:, :, 0]) > 1e-6 * S  # not within a hair of a tie
    assert clear.mean() > 0.99
    assert np.array_equal(codes.astype(np.int64)[clear], best[clear])


@pytest.mark.parametrize("bits", [8, 4])
def test_error_bound_and_ends(bits):
    x = _rows(4000, seed=12)
    codes, sb, zb = oracle.quantize_rows(x, bits)
    S = oracle.f16_to_f32(sb).astype(np.float64)
    Z = oracle.f16_to_f32(zb).astype(np.float64)
    mn = x.min(axis=1).astype(np.float64)
    xhat = codes * S[:, None] + Z[:, None]
    err = np.abs(x - xhat)
    bound = S[:, None] / 2 + np.abs(mn - Z)[:, None] + 1e-6 * np.abs(x)
    assert (err <= bound).all()
    qmax = (1 << bits) - 1
    rows = np.arange(x.shape[0])
    assert (codes[rows, x.argmin(axis=1)] == 0).all()
    assert (codes[rows, x.argmax(axis=1)] == qmax).all()
    assert codes.max() <= qmax


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_scale_zero_are_fp16_roundings(bits, dtype):
    x = _rows(3000, seed=13, dtype=dtype)
    _, sb, zb = oracle.quantize_rows(x, bits)
    mn = x.min(axis=1)
    mx = x.max(axis=1)
    qmax = np.float32((1 << bits) - 1)
    s32 = (mx - mn) / qmax  # numpy float32 arithmetic (IEEE)
    assert np.array_equal(sb, s32.astype(np.float16).view(np.uint16))
    assert np.array_equal(zb, (mn + np.float32(0)).astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("bits", [8, 4])
def test_monotone_in_x(bits):
    x = _rows(1000, seed=14)
    codes, _, _ = oracle.quantize_rows(x, bits)
    order = np.argsort(x, axis=1, kind="stable")
    c_sorted = np.take_along_axis(codes, order, axis=1).astype(np.int64)
    assert (np.diff(c_sorted, axis=1) >= 0).all()


def test_every_fp16_value_in_a_fixed_row():
    """Each finite fp16 value in [-8, 8] placed in a row whose min/max are -8 and 8."""
    h = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    vals = h[np.isfinite(h) & (np.abs(h) <= 8)]
    n = vals.size
    rows = np.zeros((n, 128), dtype=np.float32)
    rows[:, 0] = -8
    rows[:, 1] = 8
    rows[:, 2] = vals
    for bits in (8, 4):
        codes, sb, zb = oracle.quantize_rows(rows, bits)
        S = float(oracle.f16_to_f32(sb[:1])[0])
        assert (zb == 0xC800).all()  # -8
        # the exact quotient, in fp64, away from half-way points
        qt = (vals.astype(np.float64) + 8) / S
        frac = qt - np.floor(qt)
        clear = np.abs(frac - 0.5) > 1e-5
        want = np.clip(np.rint(qt), 0, (1 << bits) - 1)
        assert np.array_equal(codes[clear, 2].astype(np.float64), want[clear])
