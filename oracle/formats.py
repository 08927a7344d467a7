"""Number formats: OCP FP8 E4M3 ("fn" flavour) and BF16.

Test infrastructure (CPU oracle); see the package docstring for who may use it.

Everything here is written from the format definitions, not from any library:

* E4M3 is 1 sign bit, 4 exponent bits with bias 7 and 3 mantissa bits.
  The finite range is [-448, +448]. There is no infinity. Codes 0x7F and 0xFF
  are NaN. [FP8 Native Serving, "FP8 E4M3: range and quirks"]
* A 256-entry decode table is the CPU-side decoder. [FP8 Native Serving,
  "FP8 E4M3: range and quirks": a 256-entry E4M3 table kept for CPU sanity
  checks]
* BF16 -> F32 is exact (a 16-bit left shift). [Qwen checkpoints with block FP8
  weights, first paragraph: BF16 block scales expand exactly to F32]
* F32 -> BF16 is round-to-nearest-even and byte-exact against PyTorch's cast.
  [FP8 Native Serving, "FP8 E4M3: range and quirks": the f32_to_bf16 RNE cast]
"""

from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_BIAS = 7
_E4M3_MIN_NORMAL_EXP = 1 - E4M3_BIAS          # -6
_E4M3_SUBNORMAL_QUANTUM = 2.0 ** (_E4M3_MIN_NORMAL_EXP - 3)   # 2^-9


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code as a Python float (exact), NaN for 0x7F/0xFF.

    sign * 2^(e-7) * (1 + m/8) for e > 0; sign * 2^-6 * (m/8) for e == 0.
    The all-ones exponent with mantissa 7 is NaN. With mantissa < 7 it is an
    ordinary finite value, because the format has no infinity.
    """
    code = int(code) & 0xFF
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, _E4M3_MIN_NORMAL_EXP)
    return s * math.ldexp(1.0 + m / 8.0, e - E4M3_BIAS)


_LUT: np.ndarray | None = None


def e4m3_decode_lut() -> np.ndarray:
    """The 256-entry decode table (float64, exact), built code by code."""
    global _LUT
    if _LUT is None:
        _LUT = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
        _LUT.setflags(write=False)
    return _LUT


def e4m3_encode_rne_sat(v) -> np.ndarray:
    """Round each value to the nearest E4M3 code, ties to even, saturating.

    |v| >= 448 gives +-448 (code 0x7E/0xFE). Values between 448 and the
    midpoint 464 round to 448 anyway, and larger ones saturate. NaN gives
    0x7F, or 0xFF when the sign bit is set. The input is taken at its own
    precision: float32 values widen exactly to float64, and every step below
    is exact in float64 except the final rint, which is the rounding itself.
    """
    a64 = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(a64).astype(np.uint8) << 7).astype(np.uint8)
    a = np.abs(a64)
    with np.errstate(invalid="ignore", over="ignore"):
        # subnormal range: multiples of 2^-9; rint(8) lands on code 0x08 = 2^-6
        m_sub = np.rint(a / _E4M3_SUBNORMAL_QUANTUM)
        # normal range: a = f * 2^E with f in [0.5, 1), so the unbiased exponent is E-1
        _, E = np.frexp(a)
        e_unb = E.astype(np.int64) - 1
        mant = np.rint(np.ldexp(a, -(e_unb - 3)))            # in [8, 16]
        code_norm = ((e_unb + E4M3_BIAS) << 3) + (mant.astype(np.int64) - 8)
    out = np.where(a < 2.0 ** _E4M3_MIN_NORMAL_EXP, m_sub, code_norm)
    out = np.where(a >= E4M3_MAX, 0x7E, out)
    out = np.where(np.isnan(a), 0x7F, out)
    return (out.astype(np.int64).astype(np.uint8) | sign).astype(np.uint8)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float32, exactly: shift into the high half."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 -> BF16 bits, round to nearest even on the 16 dropped bits.

    NaN maps to the quiet pattern 0x7FC0 and loses its sign, as PyTorch's
    cast does. Overflow rounds to +-inf, as RNE must.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    return np.where(nan, np.uint16(0x7FC0), r).astype(np.uint16)


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> BF16 bits with one correct RNE rounding (no float32 detour).

    BF16 keeps 8 significant bits. Normal quantum is 2^(e-7), the subnormal
    quantum is 2^-133, and the top finite value is (2 - 2^-7) * 2^127.
    """
    a64 = np.asarray(x, dtype=np.float64)
    sign = np.signbit(a64)
    a = np.abs(a64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, E = np.frexp(a)
        e_unb = np.maximum(E.astype(np.int64) - 1, -126)
        quantum_exp = e_unb - 7
        r = np.ldexp(np.rint(np.ldexp(a, -quantum_exp)), quantum_exp)
        r = np.where(r >= 2.0 ** 128, np.inf, r)
        bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(sign, bits | np.uint16(0x8000), bits)
    return np.where(np.isnan(a), np.uint16(0x7FC0), bits).astype(np.uint16)
