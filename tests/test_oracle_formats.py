"""Pins of the oracle's format codecs against things other than itself.

- E4M3fn, E5M2, E8M0 and bfloat16 decode/encode are compared with PyTorch's
  own float8 / bfloat16 conversions (an independent library routine).
- E2M1 is compared with the OCP MX v1.0 value table (tests/golden).
- Format maxima are compared with the values printed on the pages.
- Ties-to-even, saturation, round trip and monotonicity are checked as
  properties of round-to-nearest-even.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden


def _torch_dec(dtype):
    return torch.arange(256, dtype=torch.uint8).view(dtype).to(torch.float64).numpy()


@pytest.mark.parametrize("name,dtype", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_decode_exhaustive_matches_torch(orc, name, dtype):
    ref = _torch_dec(dtype)
    dec = getattr(orc, f"dec_{name}")
    for c in range(256):
        got = dec(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), hex(c)


def test_e8m0_decode_exhaustive_matches_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for c in range(256):
        got = orc.dec_e8m0(c)
        assert (math.isnan(got) and math.isnan(ref[c])) or got == ref[c], hex(c)


def test_e2m1_decode_matches_ocp_table(orc):
    for code, val in read_golden("e2m1_values.txt"):
        c, v = int(code, 16), float(val)
        got = orc.dec_e2m1(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), code


def test_bf16_decode_matches_torch(orc):
    bits = np.arange(0, 65536, 97, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, r in zip(bits, ref):
        got = orc.dec_bf16(int(b))
        assert (math.isnan(got) and math.isnan(r)) or got == r


def test_format_maxima_match_pages(orc):
    g = {(r[0], r[1]): float(r[2]) for r in read_golden("format_constants.txt")}
    assert orc.dec_e5m2(0x7B) == g[("max", "fp8_e5m2")]
    assert orc.dec_e4m3(0x7E) == g[("max", "fp8_e4m3")]
    # the page's +-240 is the largest E4M3 value below the all-ones exponent field
    assert orc.dec_e4m3(0x77) == g[("max_ieee_style", "fp8_e4m3")]
    assert orc.dec_e2m1(0x7) == g[("max", "e2m1")]
    assert all(orc.dec_e4m3(c) < orc.dec_e4m3(0x7E) for c in range(0x7E))


def test_anchor_values(orc):
    assert orc.dec_e4m3(0x08) == 2.0 ** -6
    assert orc.dec_e4m3(0x01) == 2.0 ** -9
    assert orc.dec_e5m2(0x01) == 2.0 ** -16
    assert orc.dec_e2m1(0x1) == 0.5
    assert orc.dec_e8m0(127) == 1.0 and orc.dec_e8m0(0) == 2.0 ** -127


def _random_fp32(n, lo_exp, hi_exp, seed):
    rng = np.random.default_rng(seed)
    mag = 2.0 ** rng.uniform(lo_exp, hi_exp, n)
    sign = rng.choice([-1.0, 1.0], n)
    return (mag * sign).astype(np.float32)


def _midpoints(orc, dec, max_code):
    vals = sorted({dec(c) for c in range(max_code + 1)})
    return np.array([(a + b) / 2 for a, b in zip(vals, vals[1:])], np.float32)


@pytest.mark.parametrize("name,dtype,maxv,max_code", [
    ("e4m3", torch.float8_e4m3fn, 448.0, 0x7E), ("e5m2", torch.float8_e5m2, 57344.0, 0x7B)])
def test_fp8_encode_matches_torch_in_range(orc, name, dtype, maxv, max_code):
    dec = getattr(orc, f"dec_{name}")
    enc = getattr(orc, f"enc_{name}")
    x = np.concatenate([
        _random_fp32(20000, -30, math.log2(maxv), 1),
        _midpoints(orc, dec, max_code), -_midpoints(orc, dec, max_code),
        np.array([0.0, -0.0, maxv, -maxv, 1e-30, -1e-30], np.float32)])
    x = x[np.abs(x) <= maxv]
    ref = torch.from_numpy(x).to(dtype).view(torch.uint8).numpy()
    got = np.array([enc(float(v)) for v in x], np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(x[i]), hex(ref[i]), hex(got[i])) for i in bad[:5]]


@pytest.mark.parametrize("name,max_code,sign", [("e4m3", 0x7E, 0x80), ("e5m2", 0x7B, 0x80),
                                                ("e2m1", 0x7, 0x8)])
def test_encode_round_trip_saturation_monotone(orc, name, max_code, sign):
    dec = getattr(orc, f"dec_{name}")
    enc = getattr(orc, f"enc_{name}")
    for c in list(range(max_code + 1)) + [sign | c for c in range(max_code + 1)]:
        assert enc(dec(c)) == c, hex(c)
    maxv = dec(max_code)
    assert enc(1e30) == max_code and enc(-1e30) == (sign | max_code)
    assert enc(maxv * 1.01) == max_code
    assert enc(float("inf")) == max_code and enc(float("-inf")) == (sign | max_code)
    xs = np.sort(_random_fp32(4000, -20, math.log2(maxv) + 1, 7))
    vals = [dec(enc(float(v))) for v in xs]
    assert all(a <= b for a, b in zip(vals, vals[1:]))


def test_e2m1_ties_to_even(orc):
    # midpoints between neighbouring E2M1 values round to the even code
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, v in expect.items():
        assert orc.dec_e2m1(orc.enc_e2m1(x)) == v
        assert orc.dec_e2m1(orc.enc_e2m1(-x)) == -v
    # just off the midpoints rounds to the nearer value
    assert orc.dec_e2m1(orc.enc_e2m1(np.nextafter(np.float32(2.5), np.float32(9)))) == 3.0
    assert orc.dec_e2m1(orc.enc_e2m1(np.nextafter(np.float32(0.25), np.float32(0)))) == 0.0


def test_signed_zero_and_nan(orc):
    assert orc.enc_e4m3(-0.0) == 0x80 and orc.enc_e5m2(-0.0) == 0x80 and orc.enc_e2m1(-0.0) == 0x8
    assert orc.enc_e4m3(-1e-30) == 0x80 and orc.enc_e2m1(-0.1) == 0x8
    assert orc.enc_e4m3(float("nan")) == 0x7F
    assert orc.enc_e5m2(float("-nan")) in (0x7F, 0xFF)


def test_quantization_error_within_half_gap(orc):
    """For in-range inputs the decoded value is a nearest code: the error is at
    most half the gap between the two codes that bracket the input."""
    for name, max_code in (("e4m3", 0x7E), ("e5m2", 0x7B), ("e2m1", 0x7)):
        dec = getattr(orc, f"dec_{name}")
        enc = getattr(orc, f"enc_{name}")
        vals = np.array(sorted({dec(c) for c in range(max_code + 1)}))
        for x in _random_fp32(3000, -12, math.log2(vals[-1]), 11):
            a = abs(float(x))
            i = np.searchsorted(vals, a)
            lo, hi = vals[max(i - 1, 0)], vals[min(i, len(vals) - 1)]
            assert abs(abs(dec(enc(float(x)))) - a) <= (hi - lo) / 2 + 0.0


def test_bf16_round_matches_torch(orc):
    x = np.concatenate([_random_fp32(20000, -140, 127.9, 3),
                        np.array([3.3961e38, 3.4e38, -3.39e38, 1e-45, -0.0, 0.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.enc_bf16(float(v)) for v in x], np.uint16)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(x[i]), hex(ref[i]), hex(got[i])) for i in bad[:5]]
