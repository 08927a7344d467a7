"""Pins for oracle.linear: W8A8 / W8A16 / grouped projections, scale rows, routing.

The main pin is exact rational brute force on tiny inputs with tails on both
axes, unequal K blocks and member-local origins (the fixture properties the
block-FP8 GPU test distinguishes [Qwen checkpoints with block FP8 weights, last
paragraph]). Further pins: the one-block special case against torch.matmul,
the page's W8A8-versus-W8A16 accuracy gate, and hand-computed scale-row tables.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from oracle import formats as F
from oracle import linear as L
from oracle import quant as Q


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _frac_lut():
    lut = F.e4m3_decode_lut()
    return [Fraction(float(v)) if np.isfinite(v) else None for v in lut]


def _tiny_problem(seed, M, N, K, members):
    g = synth.generator(seed)
    w = synth.weight_f32(g, N, K).numpy()
    x = synth.activations_bf16(g, M, K, outlier="entries", frac=0.05, factor=20.0)
    rows = members or [N]
    q_parts, s_parts, r0 = [], [], 0
    for n in rows:
        qi, si = Q.quantize_weight_blocks(w[r0:r0 + n])
        q_parts.append(qi)
        s_parts.append(si)
        r0 += n
    return _bits(x), np.concatenate(q_parts), np.concatenate(s_parts)


def _brute_w8a8(qa, sa, qw, sw_f32, rmap, K):
    lut = _frac_lut()
    M, N = qa.shape[0], qw.shape[0]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for kb in range(-(-K // 128)):
                part = Fraction(0)
                for k in range(128 * kb, min(128 * kb + 128, K)):
                    part += lut[qa[m, k]] * lut[qw[n, k]]
                tot += Fraction(float(sa[m, kb])) * Fraction(float(sw_f32[rmap[n], kb])) * part
            y[m, n] = float(tot)
    return y


def _brute_w8a16(xb, qw, sw_f32, rmap, K):
    lut = _frac_lut()
    x = F.bf16_bits_to_f32(xb)
    M, N = x.shape[0], qw.shape[0]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for kb in range(-(-K // 128)):
                part = Fraction(0)
                for k in range(128 * kb, min(128 * kb + 128, K)):
                    part += Fraction(float(x[m, k])) * lut[qw[n, k]]
                tot += Fraction(float(sw_f32[rmap[n], kb])) * part
            y[m, n] = float(tot)
    return y


def test_scale_rows_hand_tables():
    r = L.scale_rows(10240, [8192, 1024, 1024])
    assert r[0] == 0 and r[8191] == 63 and r[8192] == 64 and r[9215] == 71
    assert r[9216] == 72 and r[10239] == 79
    r = L.scale_rows(300, [100, 200])
    assert r[:100].tolist() == [0] * 100
    assert r[100:228].tolist() == [1] * 128 and r[228:300].tolist() == [2] * 72
    r = L.scale_rows(192)
    assert r[:128].tolist() == [0] * 128 and r[128:].tolist() == [1] * 64


@pytest.mark.parametrize("members", [None, [70, 60]])
def test_w8a8_brute_force_tails(members):
    M, N, K = 3, 130, 260
    xb, qw, sw = _tiny_problem(21, M, N, K, members)
    qa, sa = Q.act_quant_group(xb)
    swf = F.bf16_bits_to_f32(sw)
    rmap = L.scale_rows(N, members)
    got = L.linear_w8a8(qa, sa, qw, sw, members)
    ref = _brute_w8a8(qa, sa, qw, swf, rmap, K)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14 * np.abs(ref).max())


@pytest.mark.parametrize("members", [None, [70, 60]])
def test_w8a16_brute_force_tails(members):
    M, N, K = 2, 130, 260
    xb, qw, sw = _tiny_problem(22, M, N, K, members)
    swf = F.bf16_bits_to_f32(sw)
    rmap = L.scale_rows(N, members)
    got = L.linear_w8a16(xb, qw, sw, members)
    ref = _brute_w8a16(xb, qw, swf, rmap, K)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14 * np.abs(ref).max())


def test_row_col_subsets_match_full():
    xb, qw, sw = _tiny_problem(23, 9, 300, 384, [100, 200])
    qa, sa = Q.act_quant_group(xb)
    full = L.linear_w8a8(qa, sa, qw, sw, [100, 200])
    rows, cols = [0, 4, 8], [0, 99, 100, 227, 228, 299]
    sub = L.linear_w8a8(qa, sa, qw, sw, [100, 200], rows=rows, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])


def test_single_block_unit_scales_is_plain_matmul():
    rng = np.random.default_rng(5)
    qa = rng.integers(0, 256, (8, 128), dtype=np.uint8)
    qw = rng.integers(0, 256, (64, 128), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0     # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0
    ones_a = np.ones((8, 1), np.float32)
    ones_w = np.ones((1, 1), np.float32)
    got = L.linear_w8a8(qa, ones_a, qw, ones_w)
    A = torch.from_numpy(qa).view(torch.float8_e4m3fn).double()
    W = torch.from_numpy(qw).view(torch.float8_e4m3fn).double()
    assert np.array_equal(got, torch.matmul(A, W.T).numpy())


def test_w8a8_vs_w8a16_accuracy_gate_config0():
    """[Module w8a8_prefill, "ACCURACY"]: cosine >= 0.999, relative RMS <= 2%."""
    d = synth.single_tails(0)
    qw, sw = Q.quantize_weight_blocks(d["w"].numpy())
    xb = _bits(d["x"])
    qa, sa = Q.act_quant_group(xb)
    y8 = L.linear_w8a8(qa, sa, qw, sw)
    y16 = L.linear_w8a16(xb, qw, sw)
    cos = float((y8 * y16).sum() / np.sqrt((y8 ** 2).sum() * (y16 ** 2).sum()))
    rrms = float(np.sqrt(((y8 - y16) ** 2).mean() / (y16 ** 2).mean()))
    assert cos >= 0.999 and rrms <= 0.02


def test_reciprocal_scale_is_orders_off():
    xb, qw, sw = _tiny_problem(24, 4, 192, 320, None)
    good = L.linear_w8a16(xb, qw, sw)
    inv = (1.0 / F.bf16_bits_to_f32(sw)).astype(np.float32)
    bad = L.linear_w8a16(xb, qw, inv)
    assert np.linalg.norm(bad - good) > 1e3 * np.linalg.norm(good)


def test_grouped_brute_force_with_empty_expert():
    K, N = 256, 136
    offsets = np.array([0, 2, 2, 5])
    g = synth.generator(31)
    w = synth.weight_stack_f32(g, 3, N, K).numpy()
    x = synth.activations_bf16(g, 5, K)
    qa, sa = Q.act_quant_group(_bits(x))
    qw = np.zeros((3, N, K), np.uint8)
    sw = np.zeros((3, 2, 2), np.uint16)
    for e in range(3):
        qw[e], sw[e] = Q.quantize_weight_blocks(w[e])
    got = L.grouped_linear_w8a8(qa, sa, qw, sw, offsets)
    rmap = L.scale_rows(N)
    for e in range(3):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        ref = _brute_w8a8(qa[r0:r1], sa[r0:r1], qw[e], F.bf16_bits_to_f32(sw[e]), rmap, K)
        assert np.allclose(got[r0:r1], ref, rtol=1e-12, atol=1e-14 * np.abs(ref).max())


def test_route_topk_brute_force():
    logits = np.array([[0.1, 2.0, 2.0, -1.0, 0.5, 0.0],
                       [3.0, 1.0, 1.0, 1.0, 1.0, 1.0],
                       [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],
                       [-5.0, 4.0, 0.3, 0.2, 1.0, 2.5],
                       [1.0, 1.5, 2.0, 2.5, 3.0, 3.5]], dtype=np.float32)
    k = 2
    out = L.route_topk(logits, k)
    T, E = logits.shape
    for t in range(T):
        z = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-z[e], e))   # softmax is monotone in z
        assert out["experts"][t].tolist() == order[:k]
        p = np.exp(np.array(z) - max(z))
        p = p / p.sum()
        w = p[order[:k]] / p[order[:k]].sum()
        assert np.allclose(out["weights"][t], w, rtol=1e-15)
    counts = np.bincount(out["experts"].reshape(-1), minlength=E)
    assert out["offsets"].tolist() == [0] + np.cumsum(counts).tolist()
    assert np.all(np.diff(out["row_expert"]) >= 0)
    for e in range(E):
        sl = slice(out["offsets"][e], out["offsets"][e + 1])
        assert np.all(out["row_expert"][sl] == e)
        assert np.all(np.diff(out["row_token"][sl]) > 0)
    for t in range(T):
        for j in range(k):
            r = out["row_of"][t, j]
            assert out["row_token"][r] == t and out["row_expert"][r] == out["experts"][t, j]
