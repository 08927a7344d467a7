"""GPU parity: the steps on either side of the grouped MoE projection
(bfp8_moe_gather_act_quant, bfp8_moe_combine) and the MoE FFN layer they
close, against oracle/moe.py.

Gather + quantization is integer/byte work decided in float32 on both sides:
bit-exact. The combine sums top-k products in float32 fused multiply-adds
(slot order) and rounds once to BF16; against the exact sum S the error is
at most 2^-8 |S| (the BF16 rounding: an 8-bit significand) plus 2 * k * 2^-24 * sum_j |w_j y_j|
(the k roundings of the float32 chain, and the BF16 rounding of that error),
and the rounding flips that float32 error can cause are rare, so at least
99.9% of the outputs must also equal the oracle's BF16 bits.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import (assert_close, bits16, cos_rrms, quantize_members, scale_to_dev, to_dev_bf16,
                      to_dev_u8)
from oracle import chain as CH
from oracle import formats as F
from oracle import linear as L
from oracle import moe as MOE

pytestmark = pytest.mark.gpu


def _i32(a, dev):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev)


def _gather(bfp8, dev, xb, row_token, ldx=None, ldq=None):
    T, H = xb.shape
    ldx = ldx or H
    ldq = ldq or H
    xpad = np.zeros((T, ldx), dtype=np.uint16)
    xpad[:, :H] = xb
    x = to_dev_bf16(xpad, dev)[:, :H]
    R = len(row_token)
    qbuf = torch.full((R, ldq), 0xAA, dtype=torch.uint8, device=dev)
    s = torch.full((R, -(-H // 128)), -1.0, dtype=torch.float32, device=dev)
    bfp8.bfp8_moe_gather_act_quant(x, _i32(row_token, dev), qbuf[:, :H], s)
    torch.cuda.synchronize()
    qb = qbuf.cpu().numpy()
    assert (qb[:, H:] == 0xAA).all(), "wrote past the row"
    return qb[:, :H], s.cpu().numpy()


@pytest.mark.parametrize("ldx,ldq", [(None, None), (336, 336), (325, 333)],
                         ids=["packed", "aligned_pitch", "odd_pitch"])
def test_gather_small(bfp8, cuda_device, ldx, ldq):
    T, H = 37, 320                                    # a 64-column tail group
    g = synth.generator(77)
    xb = bits16(synth.activations_bf16(g, T, H, outlier="entries", frac=0.02, factor=30.0))
    rng = np.random.default_rng(3)
    row_token = np.concatenate([rng.integers(0, T, 45), [-1, T, 0, T - 1, 2 ** 30]])
    q, s = _gather(bfp8, cuda_device, xb, row_token, ldx, ldq)
    q_ref, s_ref = MOE.gather_act_quant(xb, row_token)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))


def test_gather_empty_is_a_no_op(bfp8, cuda_device):
    dev = cuda_device
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device=dev)
    q = torch.full((0, 256), 1, dtype=torch.uint8, device=dev)
    s = torch.empty(0, 2, dtype=torch.float32, device=dev)
    bfp8.bfp8_moe_gather_act_quant(x, torch.empty(0, dtype=torch.int32, device=dev), q, s)
    torch.cuda.synchronize()


def test_gather_moe_workload(bfp8, cuda_device):
    """8192 tokens x top-8 of 128 experts, hidden 2048: every routed row."""
    d = synth.moe(0)
    route = L.route_topk(d["logits"].numpy(), synth.MOE_PREFILL["top_k"])
    xb = bits16(d["x"])
    q, s = _gather(bfp8, cuda_device, xb, route["row_token"])
    q_ref, s_ref = MOE.gather_act_quant(xb, route["row_token"])
    assert np.array_equal(q, q_ref)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))


def _combine(bfp8, dev, yb, rows, w, ldy=None, ldo=None):
    R, H = yb.shape
    T = rows.shape[0]
    ldy = ldy or H
    ldo = ldo or H
    ypad = np.zeros((R, ldy), dtype=np.uint16)
    ypad[:, :H] = yb
    y = to_dev_bf16(ypad, dev)[:, :H]
    obuf = torch.full((T, ldo), 7.0, dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_moe_combine(y, _i32(rows, dev), torch.from_numpy(np.float32(w)).to(dev),
                          obuf[:, :H])
    torch.cuda.synchronize()
    ob = bits16(obuf)
    assert (ob[:, H:] == bits16(torch.tensor([7.0], dtype=torch.bfloat16))[0]).all()
    return ob[:, :H]


def _check_combine(out_bits, yb, rows, w, what):
    w = np.float32(w)
    S = MOE.combine_f64(yb, rows, w)
    y = F.bf16_bits_to_f32(yb).astype(np.float64)
    R = y.shape[0]
    mag = np.zeros_like(S)
    for j in range(rows.shape[1]):
        r = rows[:, j]
        ok = (r >= 0) & (r < R)
        mag[ok] += np.abs(w[ok, j, None].astype(np.float64) * y[r[ok]])
    got = F.bf16_bits_to_f32(out_bits).astype(np.float64)
    bound = 2.0 ** -8 * np.abs(S) + 2 * rows.shape[1] * 2.0 ** -24 * mag + 1e-38
    bad = np.abs(got - S) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} outside the float32 bound"
    agree = float(np.mean(out_bits == F.f64_to_bf16_bits(S)))
    assert agree >= 0.999, f"{what}: BF16 bits agree on {agree:.5f}"


@pytest.mark.parametrize("ldy,ldo", [(None, None), (208, 216), (203, 201)],
                         ids=["packed", "aligned_pitch", "odd_pitch"])
def test_combine_small(bfp8, cuda_device, ldy, ldo):
    R, H, T, k = 90, 200, 50, 3                        # 200 = 25 eight-column chunks
    rng = np.random.default_rng(9)
    yb = F.f64_to_bf16_bits(rng.normal(size=(R, H)) * 3.0)
    rows = rng.integers(0, R, size=(T, k))
    rows[0, 1], rows[1, 0], rows[2, 2], rows[3, :] = -1, R, 2 ** 30, -5   # skipped slots
    w = rng.normal(size=(T, k))                        # signed, not normalized
    out = _combine(bfp8, cuda_device, yb, rows, w, ldy, ldo)
    _check_combine(out, yb, rows, w, "combine small")
    assert (F.bf16_bits_to_f32(out[3]) == 0).all()


def test_combine_moe_workload(bfp8, cuda_device):
    """65,536 routed rows of hidden 2048 back onto 8192 tokens, top-8."""
    d = synth.moe(0)
    route = L.route_topk(d["logits"].numpy(), synth.MOE_PREFILL["top_k"])
    g = synth.generator(5)
    yb = bits16(synth.activations_bf16(g, len(route["row_token"]), synth.MOE_PREFILL["hidden"]))
    out = _combine(bfp8, cuda_device, yb, route["row_of"], route["weights"])
    _check_combine(out, yb, route["row_of"], route["weights"], "combine moe")


def _stack(w, members=None):
    qs, ss = zip(*[quantize_members(w[e], members) for e in range(w.shape[0])])
    return np.stack(qs), np.stack(ss)


def test_moe_layer_end_to_end(bfp8, cuda_device):
    """The MoE FFN at 8192 tokens x top-8 of 128 experts, hidden 2048, expert
    intermediate 768, on the GPU path gather+quant -> grouped gate/up with
    SiLU*up+quant -> grouped down -> combine. On the routed rows of sampled
    tokens, each stage is checked on the bytes both sides share, at that
    stage's own bar: gather bit-exact; gate/up+quant codes as the fused
    tests; down (fed the GPU's h bytes) and combine (fed the GPU's down
    output) as GEMM outputs and the combine bound. End to end, a rare h code
    that rounds the other way is a quantization-level difference, so each
    token meets the W8A8 accuracy gate against the oracle's layer: cosine >=
    0.999 and relative RMS <= 2%."""
    dev = cuda_device
    c = synth.MOE_PREFILL
    d = synth.moe(0)
    T, H, I, E = c["tokens"], c["hidden"], c["inter"], c["experts"]
    route = L.route_topk(d["logits"].numpy(), c["top_k"])
    R = len(route["row_token"])
    xb = bits16(d["x"])
    q_gu, s_gu = _stack(d["w_gate_up"].numpy(), [I, I])
    q_d, s_d = _stack(d["w_down"].numpy())
    offsets = route["offsets"]
    off = _i32(offsets, dev)
    qa = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sa = torch.empty(R, H // 128, dtype=torch.float32, device=dev)
    qh = torch.empty(R, I, dtype=torch.uint8, device=dev)
    sh = torch.empty(R, I // 128, dtype=torch.float32, device=dev)
    y = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws1 = torch.empty(bfp8.bfp8_grouped_linear_silu_quant_workspace(R, E, I, H),
                      dtype=torch.uint8, device=dev)
    ws2 = torch.empty(bfp8.bfp8_grouped_linear_workspace(R, E, H, I), dtype=torch.uint8,
                      device=dev)
    w32 = np.float32(route["weights"])
    bfp8.bfp8_moe_gather_act_quant(to_dev_bf16(xb, dev), _i32(route["row_token"], dev), qa, sa)
    bfp8.bfp8_grouped_linear_silu_quant(qa, sa, to_dev_u8(q_gu, dev), scale_to_dev(s_gu, dev), off,
                                        qh, sh, workspace=ws1)
    bfp8.bfp8_grouped_linear(qh, sh, to_dev_u8(q_d, dev), scale_to_dev(s_d, dev), off, y,
                             workspace=ws2)
    bfp8.bfp8_moe_combine(y, _i32(route["row_of"], dev), torch.from_numpy(w32).to(dev), out)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0

    tokens = np.sort(np.random.default_rng(4).choice(T, 16, replace=False))
    rows = np.unique(route["row_of"][tokens].reshape(-1))
    # gather + quantization
    qa_g, sa_g = qa.cpu().numpy(), sa.cpu().numpy()
    qa_r, sa_r = MOE.gather_act_quant(xb, route["row_token"][rows])
    assert np.array_equal(qa_g[rows], qa_r) and np.array_equal(sa_g[rows], sa_r)
    # gate/up + SiLU*up + quantization of h
    qh_g, sh_g = qh.cpu().numpy(), sh.cpu().numpy()
    qh_r, sh_r = CH.grouped_gate_up_silu_quant(qa_g, sa_g, q_gu, s_gu, offsets, rows=rows)
    assert float(np.mean(qh_g[rows] == qh_r)) >= 0.995
    assert np.allclose(sh_g[rows], sh_r, rtol=2 ** -6, atol=0)
    # down, fed the GPU's own h bytes
    y_bits = bits16(y)
    y_r = L.grouped_linear_w8a8(qh_g, sh_g, q_d, s_d, offsets, rows=rows)
    assert_close(F.bf16_bits_to_f32(y_bits[rows]), y_r, "moe down stage")
    # combine, fed the GPU's own down output
    out_bits = bits16(out)
    _check_combine(out_bits[tokens], y_bits, route["row_of"][tokens], w32[tokens], "moe combine")
    # end to end against the oracle's layer
    route32 = dict(route, weights=w32.astype(np.float64))
    ref = MOE.moe_layer(xb, route32, q_gu, s_gu, q_d, s_d, tokens=tokens)
    got = F.bf16_bits_to_f32(out_bits[tokens]).astype(np.float64)
    for i, t in enumerate(tokens):
        cos, rrms = cos_rrms(got[i], ref[i])
        assert cos >= 0.999 and rrms <= 0.02, (int(t), cos, rrms)
