"""GPU parity: quantizers against the CPU oracle.

bfp8_act_quant_group and bfp8_quantize_weight_block must be bit-exact: codes
and scales. bfp8_silu_mul_act_quant computes SiLU with the GPU's expf and the
oracle in float64, so the two can differ by one BF16 ulp of h near a rounding
point. It is checked by the E4M3 error bound and near-total byte equality.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import bits16, dec_e4m3, to_dev_bf16
from oracle import formats as F
from oracle import quant as Q

pytestmark = pytest.mark.gpu


def _run_act_quant(bfp8, dev, xb, mn_major=False):
    M, K = xb.shape
    Kb = -(-K // 128)
    x = to_dev_bf16(xb, dev)
    q = torch.zeros(M, K, dtype=torch.uint8, device=dev)
    if mn_major:
        s = torch.zeros(Kb, M, dtype=torch.float32, device=dev)
        bfp8.bfp8_act_quant_group(x, q, s, s_stride_m=1, s_stride_kb=M)
        s = s.t()
    else:
        s = torch.zeros(M, Kb, dtype=torch.float32, device=dev)
        bfp8.bfp8_act_quant_group(x, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.contiguous().cpu().numpy()


@pytest.mark.parametrize("M,K,outlier", [
    (8, 320, "entries"),      # the single-linear workload: 1% x20 entry outliers, tail group of 64
    (5, 198, "entries"),      # K not a multiple of 4: scalar tail path
    (3, 128, None),
    (949, 5120, "channels"),  # dense-FFN prefill activations with 0.5% x30 channels
    (1, 17408, None),
    (257, 1000, "entries"),
])
def test_act_quant_bit_exact(bfp8, cuda_device, M, K, outlier):
    xb = bits16(synth.activations_bf16(synth.generator(M * 7 + K), M, K, outlier=outlier,
                                       frac=0.01 if outlier == "entries" else 0.005,
                                       factor=20.0 if outlier == "entries" else 30.0))
    q, s = _run_act_quant(bfp8, cuda_device, xb)
    qr, sr = Q.act_quant_group(xb)
    assert np.array_equal(q, qr)
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))


def test_act_quant_mn_major_scales(bfp8, cuda_device):
    xb = bits16(synth.activations_bf16(synth.generator(3), 40, 640))
    q, s = _run_act_quant(bfp8, cuda_device, xb, mn_major=True)
    qr, sr = Q.act_quant_group(xb)
    assert np.array_equal(q, qr) and np.array_equal(s, sr)


def test_act_quant_zero_rows_and_empty(bfp8, cuda_device):
    xb = np.zeros((4, 256), np.uint16)
    xb[2, 7] = F.f32_to_bf16_bits(np.float32(-3.5))
    q, s = _run_act_quant(bfp8, cuda_device, xb)
    qr, sr = Q.act_quant_group(xb)
    assert np.array_equal(q, qr) and np.array_equal(s, sr)
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device=cuda_device)
    bfp8.bfp8_act_quant_group(x, torch.zeros(0, 256, dtype=torch.uint8, device=cuda_device),
                              torch.zeros(0, 2, device=cuda_device))


@pytest.mark.parametrize("N,K,dtype", [(192, 320, "bf16"), (130, 200, "f32"), (257, 515, "bf16"),
                                       (128, 256, "f32")])
def test_weight_quant_bit_exact(bfp8, cuda_device, N, K, dtype):
    w = synth.weight_f32(synth.generator(N + K), N, K)
    q = torch.zeros(N, K, dtype=torch.uint8, device=cuda_device)
    Nb, Kb = -(-N // 128), -(-K // 128)
    s = torch.zeros(Nb, Kb, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32,
                    device=cuda_device)
    bfp8.bfp8_quantize_weight_block(w.to(cuda_device), q, s)
    torch.cuda.synchronize()
    qr, sr = Q.quantize_weight_blocks(w.numpy(), dtype)
    assert np.array_equal(q.cpu().numpy(), qr)
    got_s = bits16(s) if dtype == "bf16" else s.cpu().numpy()
    assert np.array_equal(got_s, sr)


@pytest.mark.parametrize("M,I", [(8, 256), (949, 17408), (33, 768), (3, 100)])
def test_silu_mul_act_quant(bfp8, cuda_device, M, I):
    gu = bits16(synth.activations_bf16(synth.generator(M + I), M, 2 * I))
    x = to_dev_bf16(gu, cuda_device)
    Kb = -(-I // 128)
    q = torch.zeros(M, I, dtype=torch.uint8, device=cuda_device)
    s = torch.zeros(M, Kb, dtype=torch.float32, device=cuda_device)
    bfp8.bfp8_silu_mul_act_quant(x, q, s)
    torch.cuda.synchronize()
    q, s = q.cpu().numpy(), s.cpu().numpy()
    h = F.bf16_bits_to_f32(Q.silu_mul_bf16(gu)).astype(np.float64)
    qr, sr = Q.act_quant_group(Q.silu_mul_bf16(gu))
    assert np.mean(q == qr) >= 0.999
    assert np.allclose(s, sr, rtol=2 ** -7, atol=0)
    sfull = np.repeat(s.astype(np.float64), 128, axis=1)[:, :I]
    deq = dec_e4m3(q) * sfull
    bound = 2 ** -4 * np.abs(h) * (1 + 2 ** -6) + sfull * 2 ** -9
    assert np.all(np.abs(deq - h) <= bound)
