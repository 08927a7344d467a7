"""Pins for oracle.formats: E4M3 decode/encode and BF16 conversions.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/e4m3_points.txt), PyTorch's independent float8 and
bfloat16 casts, or exact rational arithmetic.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from oracle import formats as F


def _golden_points():
    pts = []
    for line in (GOLDEN / "e4m3_points.txt").read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val, src = line.split(maxsplit=2)
        pts.append((int(code, 16), float(val), src))
    return pts


@pytest.mark.parametrize("code,val,src", _golden_points())
def test_lut_printed_points(code, val, src):
    got = F.e4m3_decode_lut()[code]
    if math.isnan(val):
        assert math.isnan(got), src
    else:
        assert got == val and math.copysign(1, got) == math.copysign(1, val), src


def test_lut_matches_torch_float8_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    lut = F.e4m3_decode_lut()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(lut))
    assert np.array_equal(ref[~nan], lut[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(lut[~nan]))


def test_lut_no_infinity_and_range():
    lut = F.e4m3_decode_lut()
    assert not np.isinf(lut).any()
    assert sorted(np.nonzero(np.isnan(lut))[0].tolist()) == [0x7F, 0xFF]
    finite = lut[~np.isnan(lut)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    pos = lut[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must be strictly increasing"


def _structured_f32_sample():
    # every sign/exponent/high-mantissa pattern with low bits set to values that
    # sit exactly on, just below and just above the E4M3 rounding points
    hi = np.arange(0, 1 << 12, dtype=np.uint32) << np.uint32(20)       # sign, exp, top 3 mantissa
    lows = np.array([0, 1, 0x7FFFF, 0x80000, 0x80001, 0xFFFFF, 0x40000, 0xC0000], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    rng = np.random.default_rng(0)
    bits = np.concatenate([bits, rng.integers(0, 1 << 32, 200000, dtype=np.uint64).astype(np.uint32)])
    v = bits.view(np.float32)
    return v[np.isfinite(v) & (np.abs(v) <= 448.0)]


def test_encode_matches_torch_cast_in_range():
    v = _structured_f32_sample()
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode_rne_sat(v)
    assert np.array_equal(ref, got)


@pytest.mark.parametrize("value,code", [
    (1.0625, 0x38),             # midpoint 1.0 | 1.125 -> even mantissa 0
    (1.1875, 0x3A),             # midpoint 1.125 | 1.25 -> even mantissa 2
    (2.0 ** -10, 0x00),         # midpoint 0 | 2^-9 -> even (zero)
    (3 * 2.0 ** -10, 0x02),     # midpoint 2^-9 | 2^-8 -> even code 2
    (440.0, 0x7E),              # midpoint 416 | 448 -> even mantissa 6 (448)
    (464.0, 0x7E),              # beyond the top: saturates
    (1e30, 0x7E),
    (math.inf, 0x7E),
    (-math.inf, 0xFE),
    (-449.0, 0xFE),
])
def test_encode_ties_and_saturation(value, code):
    assert int(F.e4m3_encode_rne_sat(np.float32(value))) == code


def test_encode_nan():
    assert int(F.e4m3_encode_rne_sat(np.float32(np.nan))) == 0x7F


def test_encode_decode_roundtrip_all_finite_codes():
    lut = F.e4m3_decode_lut()
    codes = np.array([c for c in range(256) if not np.isnan(lut[c])], dtype=np.uint8)
    back = F.e4m3_encode_rne_sat(lut[codes].astype(np.float32))
    assert np.array_equal(back, codes)


def test_bf16_widening_is_exact_all_patterns():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = F.bf16_bits_to_f32(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])
    # expansion is exact: narrowing back gives the same pattern
    assert np.array_equal(F.f32_to_bf16_bits(f[~nan]), b[~nan])


def test_f32_to_bf16_matches_torch():
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    v = bits.view(np.float32)
    v = v[~np.isnan(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.f32_to_bf16_bits(v), ref)


def _bf16_rne_exact(x: float) -> float:
    """Round a double to BF16 (8 significant bits) with exact rationals."""
    if x == 0 or math.isinf(x):
        return x
    fx = Fraction(x)
    a = abs(fx)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    m = a / q
    n = math.floor(m)
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * q
    if r >= Fraction(2) ** 128:
        return math.copysign(math.inf, x)
    return math.copysign(float(r), x)


def test_f64_to_bf16_exact_rounding():
    rng = np.random.default_rng(1)
    xs = list(rng.normal(0, 1, 3000)) + list(rng.normal(0, 1, 1000) * 1e-38) + \
        list(rng.normal(0, 1, 500) * 1e38) + [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8),
                                               2 ** -133, 2 ** -134, 3 * 2 ** -135]
    xs = np.array(xs, dtype=np.float64)
    got = F.bf16_bits_to_f32(F.f64_to_bf16_bits(xs)).astype(np.float64)
    ref = np.array([_bf16_rne_exact(float(x)) for x in xs])
    assert np.array_equal(got, ref)
