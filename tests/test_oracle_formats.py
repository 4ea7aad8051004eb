"""Pins for the oracle's number-format converters (CPU only).

The E4M3 / E2M1 / BF16 converters are checked against (1) hand-derived points and ties from the
format definitions (tests/golden/closed_forms.json), (2) the independent library converters of
torch and ml_dtypes on every one of the 65 536 BF16 bit patterns.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


def all_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    return x[np.isfinite(x)]


def test_e4m3_golden_points():
    for value, code in GOLD["e4m3_points"]["cases"]:
        assert oracle.e4m3_encode(np.array([value]))[0] == code, value
        assert oracle.e4m3_decode_table()[code] == value


def test_e4m3_golden_rounding():
    for value, code in GOLD["e4m3_rounding"]["cases"]:
        assert oracle.e4m3_encode(np.array([value], np.float32))[0] == code, value


def test_e4m3_decode_table_closed_form():
    t = oracle.e4m3_decode_table()
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    finite = t[:127]
    assert finite.max() == 448.0
    assert np.all(np.diff(finite) > 0)          # strictly increasing magnitudes
    assert finite[1] == 2.0 ** -9               # smallest subnormal
    assert np.array_equal(t[128:255], -finite)  # sign bit
    # subnormal spacing 2^-9 up to the first normal 2^-6
    assert np.allclose(np.diff(finite[:9]), 2.0 ** -9)


@pytest.mark.parametrize("lib", ["torch", "ml_dtypes"])
def test_e4m3_encode_exhaustive_bf16(lib):
    x = all_bf16_as_f32()
    ours = oracle.e4m3_encode(x)
    inrange = np.abs(x) < 464.0  # library converters give NaN above 464 (no saturation)
    if lib == "torch":
        ref = torch.from_numpy(x[inrange]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    else:
        md = pytest.importorskip("ml_dtypes")
        ref = x[inrange].astype(md.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ours[inrange], ref)
    sat = ~inrange
    assert np.all((ours[sat] & 0x7F) == 126)
    assert np.array_equal(ours[sat] >> 7, (np.signbit(x[sat])).astype(np.uint8))


def test_e4m3_encode_ties_dense():
    """Every midpoint between adjacent finite magnitudes, and one fp32 ulp either side."""
    t = oracle.e4m3_decode_table()[:127]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)
    lo = np.nextafter(mids, np.float32(0))
    hi = np.nextafter(mids, np.float32(np.inf))
    for arr in (mids, lo, hi, -mids):
        ours = oracle.e4m3_encode(arr)
        ref = torch.from_numpy(arr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours, ref)


def test_e2m1_golden():
    for value, code in GOLD["e2m1_rounding"]["cases"]:
        assert oracle.e2m1_encode(np.array([value], np.float32))[0] == code, value
    assert list(oracle.e2m1_decode_table()[:8]) == [0, .5, 1, 1.5, 2, 3, 4, 6]


def test_e2m1_encode_exhaustive_bf16():
    md = pytest.importorskip("ml_dtypes")
    x = all_bf16_as_f32()
    ours = oracle.e2m1_encode(x)
    ref = x.astype(md.float4_e2m1fn).view(np.uint8) & 0xF  # the library saturates at 6
    assert np.array_equal(ours, ref)


def test_f64_to_bf16_against_torch():
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(4000), g.standard_normal(1000) * 1e-30,
                        g.standard_normal(1000) * 1e30]).astype(np.float32).astype(np.float64)
    ours = oracle.f64_to_bf16(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # halfway cases between two BF16 neighbours go to the even mantissa
    assert oracle.f64_to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert oracle.f64_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
