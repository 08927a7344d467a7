"""Pins for the dense-FFN decode step (oracle/chain.py decode_ffn), checked
against values recomputed by hand in scalar Python.

Weights are one-hot E4M3 1.0 codes with power-of-two block scales: gate row i
picks column pi(i) of x with scale 2, up row i picks column sigma(i) with
scale 1/2, down row j picks column tau(j) of h with scale 4, the three maps
being different permutations. Every product is then exact, so the gate/up
output is 2x and x/2, h is BF16(silu(g) * u) with math.exp, and y is 4h
(W8A16) or 4 times h's dequantized E4M3 code (W8A8, codes by exhaustive
nearest-code search). For the W8A8 arm each 128-column group of x is built
with max |x| = 448 * 2^-4 and every entry a multiple of an E4M3 value by
2^-4, so the activation quantization is exact. A swapped permutation, a
transposed weight or the wrong member's scale changes y."""

import math

import numpy as np
import pytest

from oracle import chain as CH
from oracle import formats as F
from test_oracle_chain import _bf16, _e4m3_brute

H, I, M = 256, 192, 3
ONE = 0x38                                       # E4M3 1.0


def _perms(seed=11):
    """pi, sigma: distinct columns of x for the gate and up rows; tau: the
    column of h that each down row picks."""
    rng = np.random.default_rng(seed)
    return rng.permutation(H)[:I], rng.permutation(H)[:I], rng.integers(0, I, size=H)


def _weights(pi, sigma, tau):
    q_gu = np.zeros((2 * I, H), np.uint8)
    for i in range(I):
        q_gu[i, pi[i]] = ONE
        q_gu[I + i, sigma[i]] = ONE
    ib, hb = -(-I // 128), H // 128
    s_gu = np.zeros((2 * ib, hb), np.uint16)
    s_gu[:ib] = F.f64_to_bf16_bits(np.array(2.0))
    s_gu[ib:] = F.f64_to_bf16_bits(np.array(0.5))
    q_d = np.zeros((H, I), np.uint8)
    for j in range(H):
        q_d[j, tau[j]] = ONE
    s_d = np.full((H // 128, ib), F.f64_to_bf16_bits(np.array(4.0)), np.uint16)
    return q_gu, s_gu, q_d, s_d


def _h_by_hand(x, pi, sigma):
    h = np.zeros((M, I))
    for m in range(M):
        for i in range(I):
            g, u = _bf16(2.0 * x[m, pi[i]]), _bf16(0.5 * x[m, sigma[i]])
            h[m, i] = _bf16(g / (1.0 + math.exp(-g)) * u)
    return h


def test_w8a16_decode_step_by_hand():
    pi, sigma, tau = _perms()
    rng = np.random.default_rng(1)
    xb = F.f64_to_bf16_bits(rng.normal(size=(M, H)) * 2.0)
    x = F.bf16_bits_to_f32(xb).astype(np.float64)
    y = CH.decode_ffn(xb, *_weights(pi, sigma, tau), arith="w8a16")
    h = _h_by_hand(x, pi, sigma)
    assert np.array_equal(y, 4.0 * h[:, tau])


def test_w8a8_decode_step_by_hand():
    pi, sigma, tau = _perms(seed=12)
    rng = np.random.default_rng(2)
    lut = F.e4m3_decode_lut().astype(np.float64)
    finite = lut[np.isfinite(lut) & (np.abs(lut) <= 448)]
    x = rng.choice(finite, size=(M, H)) * 2.0 ** -4
    for m in range(M):
        for g in range(H // 128):
            x[m, g * 128 + rng.integers(0, 128)] = 448.0 * 2.0 ** -4 * rng.choice([-1, 1])
    xb = F.f64_to_bf16_bits(x)
    assert np.array_equal(F.bf16_bits_to_f32(xb).astype(np.float64), x)   # x is exact in BF16
    y = CH.decode_ffn(xb, *_weights(pi, sigma, tau), arith="w8a8")
    h = _h_by_hand(x, pi, sigma)
    want = np.zeros((M, H))
    for m in range(M):
        hq = np.zeros(I)
        for grp in range(-(-I // 128)):
            cols = range(grp * 128, min(grp * 128 + 128, I))
            s = np.float32(max(max(abs(h[m, c]) for c in cols), 1e-10)) / np.float32(448.0)
            for c in cols:
                hq[c] = float(lut[_e4m3_brute(float(np.float32(np.float32(h[m, c]) / s)))]) * float(s)
        want[m] = 4.0 * hq[tau]
    assert np.array_equal(y, want)


def test_decode_step_rejects_unknown_arithmetic():
    pi, sigma, tau = _perms()
    with pytest.raises(ValueError):
        CH.decode_ffn(np.zeros((1, H), np.uint16), *_weights(pi, sigma, tau), arith="fp4")
