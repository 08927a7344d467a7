"""Pins for the MoE gather + quantization, the weighted combine and the MoE
layer (oracle/moe.py), against values fixed by hand, closed forms and special
cases that reduce to the dense chain.

* gather: each token row carries one marker entry, so the codes and the scale
  of a routed row name the token it came from; the scale is marker / 448 and
  the marker's code is 448's (0x7E), everything else zero.
* combine: hand-summed rows, BF16 rounding of a sum that is not
  representable, skipped invalid rows, and the inverse relation of row_token
  and row_of (combining copies of each token's own row gives the token back).
* layer: with every expert identical, the layer is the dense chain; with the
  experts' down scales multiplied by 2^(e mod 4), each routed row is the dense
  row times that power of two, so the layer is the dense row times the sum of
  w_j 2^(e_j mod 4), with the top-k and the weights recomputed here in scalar
  Python from the logits.
"""

import math

import numpy as np
import pytest

from oracle import chain as CH
from oracle import formats as F
from oracle import linear as L
from oracle import moe as MOE
from oracle import quant as Q


def _bits(vals):
    return F.f64_to_bf16_bits(np.asarray(vals, dtype=np.float64))


def _marker_tokens(T, H):
    """Token t: value (t + 1) * 0.75 at column (37 t) mod H, zero elsewhere."""
    x = np.zeros((T, H))
    for t in range(T):
        x[t, (37 * t) % H] = (t + 1) * 0.75
    return _bits(x)


def test_gather_markers_name_their_tokens():
    T, H = 9, 200                          # two groups; the second is a 72-column tail
    xb = _marker_tokens(T, H)
    row_token = [3, 0, -1, 8, T, 3, 5]
    q, s = MOE.gather_act_quant(xb, row_token)
    assert q.shape == (7, H) and s.shape == (7, 2)
    floor = np.float32(1e-10) / np.float32(448.0)
    for r, t in enumerate(row_token):
        if not 0 <= t < T:
            assert not q[r].any()
            assert np.all(s[r] == floor)
            continue
        col = (37 * t) % H
        nz = np.nonzero(q[r])[0]
        assert list(nz) == [col] and q[r, col] == 0x7E
        g = col // 128
        assert s[r, g] == np.float32((t + 1) * 0.75) / np.float32(448.0)
        assert s[r, 1 - g] == floor


def test_gather_of_repeated_token_repeats_bytes():
    rng = np.random.default_rng(0)
    xb = _bits(rng.normal(size=(4, 256)))
    q, s = MOE.gather_act_quant(xb, [2, 2, 1])
    assert np.array_equal(q[0], q[1]) and np.array_equal(s[0], s[1])
    assert not np.array_equal(q[0], q[2])


def test_combine_hand_example():
    y = _bits([[1.0, 2.0], [3.0, -4.0], [8.0, 8.0]])
    rows = np.array([[0, 1], [2, 0], [1, -1]])
    w = np.array([[0.25, 0.75], [0.5, 0.5], [2.0, 1.0]])
    out = F.bf16_bits_to_f32(MOE.combine(y, rows, w))
    # [0.25*1 + 0.75*3, 0.25*2 - 0.75*4], [0.5*8 + 0.5*1, 0.5*8 + 0.5*2], [2*3, 2*(-4)]
    assert np.array_equal(out, np.float32([[2.5, -2.5], [4.5, 5.0], [6.0, -8.0]]))


def test_combine_rounds_once_to_bf16():
    # 1 + 2^-9 is a quarter BF16 ulp above 1 (rounds down); 1 + 3*2^-9 is
    # three quarters (rounds up to 1 + 2^-7); 1 + 2^-8 is the tie (to even: 1)
    y = _bits([[1.0], [2.0 ** -9], [1.0]])
    rows = np.array([[0, 1], [0, 1], [0, 1], [2, 1]])
    w = np.array([[1.0, 1.0], [1.0, 3.0], [1.0, 2.0], [1.0, 2.0 + 2.0 ** -20]])
    out = F.bf16_bits_to_f32(MOE.combine(y, rows, w))[:, 0]
    assert list(out) == [1.0, 1.0 + 2.0 ** -7, 1.0, 1.0 + 2.0 ** -7]


def test_combine_skips_rows_outside_the_buffer():
    y = _bits([[5.0, -1.0]])
    out = F.bf16_bits_to_f32(MOE.combine(y, np.array([[0, -1, 1, 7]]), np.ones((1, 4))))
    assert np.array_equal(out, np.float32([[5.0, -1.0]]))


@pytest.mark.parametrize("T,E,k", [(40, 16, 4), (7, 128, 8)])
def test_combine_inverts_the_permutation(T, E, k):
    rng = np.random.default_rng(T + E)
    route = L.route_topk(rng.normal(size=(T, E)).astype(np.float32), k)
    xb = _bits(rng.normal(size=(T, 64)))
    y = xb[route["row_token"]]              # each routed row is a copy of its token
    w32 = route["weights"].astype(np.float32)
    out = MOE.combine(y, route["row_of"], w32 / w32.sum(axis=1, keepdims=True))
    assert np.array_equal(out, xb)


def _layer_problem(T=24, E=6, k=3, H=256, I=192, seed=5, distinct_down=False):
    rng = np.random.default_rng(seed)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    xb = _bits(rng.normal(size=(T, H)))
    q_gu, s_gu = zip(*[Q.quantize_weight_blocks(w) for w in
                       [rng.normal(size=(I, H)) * 0.05, rng.normal(size=(I, H)) * 0.05]])
    q_gu, s_gu = np.concatenate(q_gu), np.concatenate(s_gu)
    q_d, s_d = Q.quantize_weight_blocks(rng.normal(size=(H, I)) * 0.05)
    sd = np.repeat(s_d[None], E, axis=0)
    if distinct_down:
        mult = np.array([2.0 ** (e % 4) for e in range(E)])
        sd = F.f64_to_bf16_bits(F.bf16_bits_to_f32(sd).astype(np.float64) * mult[:, None, None])
    stack = lambda a: np.repeat(a[None], E, axis=0)
    return (logits, xb, stack(q_gu), stack(s_gu), stack(q_d), sd, q_gu, s_gu, q_d, s_d)


def _dense(xb, q_gu, s_gu, q_d, s_d):
    qa, sa = Q.act_quant_group(xb)
    qh, sh = CH.gate_up_silu_quant(qa, sa, q_gu, s_gu)
    return F.bf16_bits_to_f32(F.f64_to_bf16_bits(L.linear_w8a8(qh, sh, q_d, s_d)))


def test_layer_with_identical_experts_is_the_dense_chain():
    logits, xb, Qgu, Sgu, Qd, Sd, q_gu, s_gu, q_d, s_d = _layer_problem()
    route = L.route_topk(logits, 3)
    out = MOE.moe_layer(xb, route, Qgu, Sgu, Qd, Sd)
    dense = _dense(xb, q_gu, s_gu, q_d, s_d).astype(np.float64)
    assert np.allclose(out, dense, rtol=1e-12, atol=0)
    sub = [0, 5, 23]
    assert np.array_equal(MOE.moe_layer(xb, route, Qgu, Sgu, Qd, Sd, tokens=sub), out[sub])


def test_layer_weights_each_expert_by_its_own_down_scale():
    T, E, k = 24, 6, 3
    logits, xb, Qgu, Sgu, Qd, Sd, q_gu, s_gu, q_d, s_d = _layer_problem(distinct_down=True)
    out = MOE.moe_layer(xb, L.route_topk(logits, k), Qgu, Sgu, Qd, Sd)
    dense = _dense(xb, q_gu, s_gu, q_d, s_d).astype(np.float64)
    for t in range(T):
        top = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        ex = [math.exp(float(logits[t, e]) - float(logits[t].max())) for e in top]
        factor = sum(p / sum(ex) * 2.0 ** (e % 4) for p, e in zip(ex, top))
        assert np.allclose(out[t], dense[t] * factor, rtol=1e-12, atol=0), t
