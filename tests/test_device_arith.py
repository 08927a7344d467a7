"""Host checks of the device quantizers' division-free arithmetic.

The GPU forms the 1x128 scale max(amax, 1e-10f) / 448 without a division:
with y = RN(1/448), q0 = RN(a*y), r = RN(a - q0*448) (one FMA) and
q = RN(q0 + r*y) (one FMA), Markstein's theorem makes q the correctly
rounded quotient. The group maximum is always a BF16 value (the inputs are
BF16, and h is rounded to BF16 before it is quantized), so checking every
positive finite BF16 value and the 1e-10f floor covers every scale the
kernels can produce. Each rounding is emulated exactly with rationals.
"""

from fractions import Fraction

import numpy as np


def _rn_f32(x: Fraction) -> np.float32:
    """Round a rational to the nearest float32, ties to even (exactly)."""
    c = np.float32(float(x))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best, best_d = None, None
    for v in cands:
        d = abs(Fraction(float(v)) - x)
        if best is None or d < best_d or (d == best_d and int(np.float32(v).view(np.uint32)) % 2 == 0):
            best, best_d = np.float32(v), d
    return best


def _markstein_scale(a: np.float32) -> np.float32:
    y = np.float32(1.0) / np.float32(448.0)
    fa, fy = Fraction(float(a)), Fraction(float(y))
    q0 = _rn_f32(fa * fy)
    r_exact = fa - Fraction(float(q0)) * 448
    r = _rn_f32(r_exact)
    assert Fraction(float(r)) == r_exact            # the remainder is exact, as the theorem says
    return _rn_f32(Fraction(float(r)) * fy + Fraction(float(q0)))


def test_division_free_scale_is_the_ieee_quotient_for_every_bf16_max():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32) << 16          # positive finite BF16
    amax = bits.view(np.float32)
    a = np.maximum(amax, np.float32(1e-10))
    a = np.unique(np.append(a, np.float32(1e-10)))
    want = a / np.float32(448.0)                                      # IEEE float32 division
    got = np.array([_markstein_scale(v) for v in a], dtype=np.float32)
    bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert bad.size == 0, [(float(a[i]), float(got[i]), float(want[i])) for i in bad[:5]]
