"""Pins for the fused dense-FFN glue step (oracle/chain.py), checked against
values built by hand rather than by the oracle's own routines.

With one-hot weights the projection is the identity on the dequantized
activations, times the member's block scale. Gate and up get different
scales (2 and 1/2), so swapping the halves, or reading the up member's scale
rows from the gate's origin, changes h. h is recomputed in scalar Python
(math.exp), and each code is found by brute force over all 256 E4M3 codes
(nearest value, ties to the even code)."""

import math

import numpy as np

from oracle import chain as CH
from oracle import formats as F
from oracle import quant as Q


def _bf16(v: float) -> float:
    return float(F.bf16_bits_to_f32(F.f64_to_bf16_bits(np.array([v])))[0])


def _e4m3_brute(v: float) -> int:
    """Nearest finite E4M3 code of the same sign as v (ties to the even code),
    saturating at +-448: an exhaustive search, not the oracle's encoder."""
    vals = F.e4m3_decode_lut().astype(np.float64)
    neg = math.copysign(1.0, v) < 0
    if abs(v) >= 448.0:
        return 0xFE if neg else 0x7E
    codes = [c for c in (range(0x80, 0xFF) if neg else range(0x00, 0x7F))]
    dist = [abs(vals[c] - v) for c in codes]
    best = min(dist)
    ties = [c for c, d in zip(codes, dist) if d == best]
    return ties[0] if len(ties) == 1 else next(c for c in ties if c % 2 == 0)


def _one_hot_problem(M=5, I=200, K=256, seed=3):
    rng = np.random.default_rng(seed)
    xb = F.f64_to_bf16_bits(rng.normal(size=(M, K)) * 2.0)
    qa, sa = Q.act_quant_group(xb)
    qw = np.zeros((2 * I, K), np.uint8)
    one = 0x38                                   # E4M3 1.0
    for j in range(I):
        qw[j, j] = one                            # gate row j picks column j
        qw[I + j, j] = one                        # up row j picks column j
    ib, kb = -(-I // 128), K // 128
    sw = np.zeros((2 * ib, kb), np.uint16)
    sw[:ib] = F.f64_to_bf16_bits(np.array(2.0))   # gate member grid
    sw[ib:] = F.f64_to_bf16_bits(np.array(0.5))   # up member grid (member-local origin)
    return qa, sa, qw, sw, I


def test_gate_up_silu_quant_one_hot_by_hand():
    qa, sa, qw, sw, I = _one_hot_problem()
    q_h, s_h = CH.gate_up_silu_quant(qa, sa, qw, sw)
    lut = F.e4m3_decode_lut().astype(np.float64)
    M = qa.shape[0]
    for m in range(M):
        xq = [float(lut[qa[m, j]]) * float(sa[m, j // 128]) for j in range(I)]
        h = []
        for j in range(I):
            g, u = _bf16(2.0 * xq[j]), _bf16(0.5 * xq[j])
            h.append(_bf16(g / (1.0 + math.exp(-g)) * u))
        for grp in range(-(-I // 128)):
            hs = h[grp * 128:(grp + 1) * 128]
            s = np.float32(max(max(abs(v) for v in hs), 1e-10)) / np.float32(448.0)
            assert s_h[m, grp] == s
            for t, v in enumerate(hs):
                want = _e4m3_brute(float(np.float32(np.float32(v) / s)))
                assert q_h[m, grp * 128 + t] == want, (m, grp, t, v)


def test_gate_up_halves_are_not_interchangeable():
    qa, sa, qw, sw, I = _one_hot_problem(seed=4)
    q1, _ = CH.gate_up_silu_quant(qa, sa, qw, sw)
    swapped = np.concatenate([qw[I:], qw[:I]])
    sw_swapped = np.concatenate([sw[sw.shape[0] // 2:], sw[:sw.shape[0] // 2]])
    q2, _ = CH.gate_up_silu_quant(qa, sa, swapped, sw_swapped)
    assert np.mean(q1 != q2) > 0.5


def test_grouped_form_matches_per_expert_dense_form():
    rng = np.random.default_rng(7)
    G, I, K = 3, 130, 256
    offsets = [0, 4, 4, 9]
    T = offsets[-1]
    qa, sa = Q.act_quant_group(F.f64_to_bf16_bits(rng.normal(size=(T, K))))
    qw = np.stack([_one_hot_problem(M=1, I=I, K=K)[2] for _ in range(G)])
    ib = -(-I // 128)
    sw = np.stack([np.full((2 * ib, K // 128), F.f64_to_bf16_bits(np.array(0.25 * (e + 1))),
                           np.uint16) for e in range(G)])
    qg, sg = CH.grouped_gate_up_silu_quant(qa, sa, qw, sw, offsets)
    for e in range(G):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            qd, sd = CH.gate_up_silu_quant(qa[lo:hi], sa[lo:hi], qw[e], sw[e])
            assert np.array_equal(qg[lo:hi], qd) and np.array_equal(sg[lo:hi], sd)
