"""GPU parity: per-tensor scaled FP8 weights (BFP8_SCALE_PER_TENSOR), the
degenerate block grid whose single block covers the tensor.

For every projection kind the per-tensor call must give exactly the bytes of
the same call on the explicit grid that repeats the multiplier in every block
(tensor_scale_grid), which the block-scaled parity tests already cover; and
it must meet the same acceptance bounds against the oracle on that grid.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import (assert_close, bits16, gpu_bf16_to_f64, sample_indices, scale_to_dev,
                      to_dev_bf16, to_dev_u8)
from oracle import chain as CH
from oracle import formats as F
from oracle import linear as L
from oracle import quant as Q

pytestmark = pytest.mark.gpu


def _scalar_dev(s, dev):
    """The per-tensor multiplier as a 0-d tensor (BF16 bits or float32)."""
    return scale_to_dev(np.asarray(s).reshape(()), dev)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_w8a8_and_w8a16_gemm(bfp8, cuda_device, sd):
    dev = cuda_device
    M, N, K = 200, 300, 320
    g = synth.generator(61)
    q, s = Q.quantize_weight_tensor(synth.weight_f32(g, N, K).numpy(), sd)
    grid = Q.tensor_scale_grid(s, N, K)
    xb = bits16(synth.activations_bf16(g, M, K, outlier="entries", frac=0.01, factor=20.0))
    qa, sa = Q.act_quant_group(xb)
    w = to_dev_u8(q, dev)
    outs = {}
    for kind, sc in (("tensor", _scalar_dev(s, dev)), ("grid", scale_to_dev(grid, dev))):
        y8 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_linear_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), w, sc, y8)
        y16 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_linear_w8a16(to_dev_bf16(xb, dev), w, sc, y16)
        torch.cuda.synchronize()
        assert bfp8.bfp8_device_status() == 0
        outs[kind] = (y8, y16)
    assert _same(outs["tensor"][0], outs["grid"][0]) and _same(outs["tensor"][1], outs["grid"][1])
    assert_close(gpu_bf16_to_f64(outs["tensor"][0]), L.linear_w8a8(qa, sa, q, grid), "w8a8 per-tensor")
    assert_close(gpu_bf16_to_f64(outs["tensor"][1]), L.linear_w8a16(xb, q, grid), "w8a16 per-tensor")


def test_fused_gate_up_with_one_multiplier(bfp8, cuda_device):
    dev = cuda_device
    M, I, K = 129, 200, 256
    g = synth.generator(62)
    q, s = Q.quantize_weight_tensor(synth.weight_f32(g, 2 * I, K).numpy(), "f32")
    grid = Q.tensor_scale_grid(s, 2 * I, K, [I, I])
    qa, sa = Q.act_quant_group(bits16(synth.activations_bf16(g, M, K)))
    res = []
    for sc in (_scalar_dev(s, dev), scale_to_dev(grid, dev)):
        qh = torch.empty(M, I, dtype=torch.uint8, device=dev)
        sh = torch.empty(M, -(-I // 128), dtype=torch.float32, device=dev)
        bfp8.bfp8_linear_w8a8_silu_quant(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev),
                                         to_dev_u8(q, dev), sc, qh, sh)
        torch.cuda.synchronize()
        res.append((qh.cpu().numpy(), sh.cpu().numpy()))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
    q_ref, s_ref = CH.gate_up_silu_quant(qa, sa, q, grid)
    assert np.mean(res[0][0] == q_ref) >= 0.995
    assert np.allclose(res[0][1], s_ref, rtol=2 ** -6, atol=0)


def test_grouped_per_expert_multipliers(bfp8, cuda_device):
    dev = cuda_device
    G, N, K = 5, 256, 384
    offsets = [0, 40, 40, 170, 300, 301]
    g = synth.generator(63)
    ws = synth.weight_stack_f32(g, G, N, K).numpy()
    ws *= (np.arange(1, G + 1, dtype=np.float32) ** 2)[:, None, None]   # distinct multipliers
    qs, ss = zip(*[Q.quantize_weight_tensor(ws[e], "f32") for e in range(G)])
    q, s = np.stack(qs), np.stack([np.asarray(v).reshape(()) for v in ss]).astype(np.float32)
    grid = np.stack([Q.tensor_scale_grid(s[e], N, K) for e in range(G)])
    qa, sa = Q.act_quant_group(bits16(synth.activations_bf16(g, offsets[-1], K)))
    off = torch.tensor(offsets, dtype=torch.int32, device=dev)
    outs = []
    for sc in (torch.from_numpy(s).to(dev), torch.from_numpy(grid).to(dev)):
        y = torch.empty(offsets[-1], N, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_grouped_linear(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(q, dev),
                                 sc, off, y)
        torch.cuda.synchronize()
        outs.append(y)
    assert _same(outs[0], outs[1])
    assert_close(gpu_bf16_to_f64(outs[0]), L.grouped_linear_w8a8(qa, sa, q, grid, offsets),
                 "grouped per-tensor")


@pytest.mark.parametrize("M", [1, 16])
def test_decode_gemv_both_arms(bfp8, cuda_device, M):
    dev = cuda_device
    N, K = 34816, 5120
    members = [17408, 17408]
    g = synth.generator(64)
    q, s = Q.quantize_weight_tensor(synth.weight_f32(g, N, K).numpy(), "bf16")
    grid = Q.tensor_scale_grid(s, N, K, members)
    xb = bits16(synth.decode_tokens(70 + M, M, K))
    qa, sa = Q.act_quant_group(xb)
    w = to_dev_u8(q, dev)
    wsz = bfp8.bfp8_gemv_decode_workspace(M, N, K)
    res = []
    for sc in (_scalar_dev(s, dev), scale_to_dev(grid, dev)):
        ws = torch.empty(wsz, dtype=torch.uint8, device=dev)
        y16 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        y8 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_gemv_decode(to_dev_bf16(xb, dev), w, sc, y16, ws, member_rows=members)
        bfp8.bfp8_gemv_decode_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), w, sc, y8, ws,
                                   member_rows=members)
        torch.cuda.synchronize()
        assert bfp8.bfp8_device_status() == 0
        res.append((y16, y8))
    assert _same(res[0][0], res[1][0]) and _same(res[0][1], res[1][1])
    cols = sample_indices(N, 800, seed=M)
    assert_close(gpu_bf16_to_f64(res[0][0])[:, cols], L.linear_w8a16(xb, q, grid, members, cols=cols),
                 "gemv w8a16 per-tensor")
    assert_close(gpu_bf16_to_f64(res[0][1])[:, cols],
                 L.linear_w8a8(qa, sa, q, grid, members, cols=cols), "gemv w8a8 per-tensor")


@pytest.mark.parametrize("sd", ["f32", "bf16"])
def test_decode_step_with_one_multiplier_per_weight(bfp8, cuda_device, sd):
    """The dense-FFN decode step with a per-tensor multiplier for each of its
    two weights gives the bytes of the same step on the expanded grids, in
    both arithmetics."""
    dev = cuda_device
    M, H, I = 5, 1024, 1536
    g = synth.generator(65)
    qgu, sgu = Q.quantize_weight_tensor(synth.weight_f32(g, 2 * I, H).numpy(), sd)
    qd, sdn = Q.quantize_weight_tensor(synth.weight_f32(g, H, I).numpy(), sd)
    ggu = Q.tensor_scale_grid(sgu, 2 * I, H, [I, I])
    gd = Q.tensor_scale_grid(sdn, H, I)
    x = to_dev_bf16(bits16(synth.decode_tokens(75, M, H)), dev)
    wgu, wd = to_dev_u8(qgu, dev), to_dev_u8(qd, dev)
    for arith in (bfp8.BFP8_DECODE_W8A16, bfp8.BFP8_DECODE_W8A8):
        ys = []
        for scales in ((_scalar_dev(sgu, dev), _scalar_dev(sdn, dev)),
                       (scale_to_dev(ggu, dev), scale_to_dev(gd, dev))):
            ws = torch.empty(bfp8.bfp8_decode_ffn_workspace(M, H, I, arith), dtype=torch.uint8,
                             device=dev)
            y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
            bfp8.bfp8_decode_ffn(x, wgu, scales[0], wd, scales[1], y, ws, arith=arith)
            torch.cuda.synchronize()
            assert bfp8.bfp8_device_status() == 0
            ys.append(y)
        assert _same(ys[0], ys[1]), arith


def test_library_refuses_a_per_tensor_flag_on_an_unknown_dtype(bfp8, cuda_device):
    dev = cuda_device
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(128, 128, dtype=torch.uint8, device=dev)
    s = torch.ones((), dtype=torch.float16, device=dev)
    y = torch.empty(4, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(bfp8.Bfp8Error) as e:
        bfp8.bfp8_linear_w8a16(x, w, s, y)
    assert e.value.status == 8     # SCALE_DTYPE
