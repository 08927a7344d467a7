"""GPU parity: the dense-FFN prefill chain (M = 949, gate/up [34816, 5120] ->
SiLU(gate)*up + 1x128 quant -> down [5120, 17408]), stage by stage (each GPU
stage fed the oracle's own input bytes) and end to end, on sampled rows."""

import numpy as np
import pytest
import torch

from gpu_util import (assert_close, bits16, dense_ffn_weights, gpu_bf16_to_f64, sample_indices,
                      scale_to_dev, to_dev_bf16, to_dev_u8)
from oracle import formats as F
from oracle import linear as L
from oracle import quant as Q

pytestmark = pytest.mark.gpu


def test_dense_ffn_chain(bfp8, cuda_device):
    dev = cuda_device
    qgu, sgu, qd, sd, xb = dense_ffn_weights(0)
    M, H = xb.shape
    I = 17408
    x = to_dev_bf16(xb, dev)
    wgu, swgu = to_dev_u8(qgu, dev), scale_to_dev(sgu, dev)
    wd, swd = to_dev_u8(qd, dev), scale_to_dev(sd, dev)
    qa = torch.empty(M, H, dtype=torch.uint8, device=dev)
    sa = torch.empty(M, H // 128, dtype=torch.float32, device=dev)
    gu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev)
    qh = torch.empty(M, I, dtype=torch.uint8, device=dev)
    sh = torch.empty(M, I // 128, dtype=torch.float32, device=dev)
    y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    ws1 = torch.empty(bfp8.bfp8_linear_w8a8_workspace(M, 2 * I, H, [I, I]), dtype=torch.uint8, device=dev)
    ws2 = torch.empty(bfp8.bfp8_linear_w8a8_workspace(M, H, I), dtype=torch.uint8, device=dev)
    bfp8.bfp8_act_quant_group(x, qa, sa)
    bfp8.bfp8_linear_w8a8(qa, sa, wgu, swgu, gu, member_rows=[I, I], workspace=ws1)
    bfp8.bfp8_silu_mul_act_quant(gu, qh, sh)
    bfp8.bfp8_linear_w8a8(qh, sh, wd, swd, y, workspace=ws2)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0

    rows = sample_indices(M, 24, seed=11)
    # stage 1: act quant, bit-exact
    qa_r, sa_r = Q.act_quant_group(xb)
    assert np.array_equal(qa.cpu().numpy(), qa_r)
    assert np.array_equal(sa.cpu().numpy(), sa_r)
    # stage 2: gate/up on the sampled rows, every column
    gu_r = L.linear_w8a8(qa_r, sa_r, qgu, sgu, [I, I], rows=rows)
    gu_g = gpu_bf16_to_f64(gu)[rows]
    assert_close(gu_g, gu_r, "gate/up")
    # stage 3: SiLU*up + quant of the GPU's own gate/up bytes vs the oracle on the same bytes
    gu_bits = bits16(gu)[rows]
    qh_r, sh_r = Q.silu_mul_act_quant(gu_bits)
    assert np.array_equal(qh.cpu().numpy()[rows], qh_r)
    assert np.array_equal(sh.cpu().numpy()[rows].view(np.uint32), sh_r.view(np.uint32))
    # stage 4: down fed the oracle's quantized h for those rows
    qh_full = qh.cpu().numpy()
    sh_full = sh.cpu().numpy()
    qh_full[rows], sh_full[rows] = qh_r, sh_r
    y2 = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_linear_w8a8(to_dev_u8(qh_full, dev), torch.from_numpy(sh_full).to(dev), wd, swd, y2)
    torch.cuda.synchronize()
    assert_close(gpu_bf16_to_f64(y2)[rows], L.linear_w8a8(qh_r, sh_r, qd, sd), "down stage")
    # end to end: oracle chain on the sampled rows from x
    gu_bits_r = F.f64_to_bf16_bits(gu_r)
    qh_e, sh_e = Q.silu_mul_act_quant(gu_bits_r)
    y_ref = L.linear_w8a8(qh_e, sh_e, qd, sd)
    assert_close(gpu_bf16_to_f64(y)[rows], y_ref, "chain end to end")


def test_two_chains_on_two_streams_at_once(bfp8, cuda_device):
    """Two dense-FFN chains (act quant -> fused gate/up -> down, stream-K
    workspaces) in flight at once on two streams, each with its own buffers,
    give the bytes of the same chains run one after the other."""
    dev = cuda_device
    qgu, sgu, qd, sd, xb = dense_ffn_weights(0)
    H, I, M = xb.shape[1], 17408, 300
    wgu, swgu = to_dev_u8(qgu, dev), scale_to_dev(sgu, dev)
    wd, swd = to_dev_u8(qd, dev), scale_to_dev(sd, dev)
    xs = [to_dev_bf16(xb[:M], dev), to_dev_bf16(xb[M:2 * M], dev)]

    def buffers():
        return dict(qa=torch.empty(M, H, dtype=torch.uint8, device=dev),
                    sa=torch.empty(M, H // 128, dtype=torch.float32, device=dev),
                    qh=torch.empty(M, I, dtype=torch.uint8, device=dev),
                    sh=torch.empty(M, I // 128, dtype=torch.float32, device=dev),
                    y=torch.empty(M, H, dtype=torch.bfloat16, device=dev),
                    ws1=torch.empty(bfp8.bfp8_linear_w8a8_silu_quant_workspace(M, I, H),
                                    dtype=torch.uint8, device=dev),
                    ws2=torch.empty(bfp8.bfp8_linear_w8a8_workspace(M, H, I), dtype=torch.uint8,
                                    device=dev))

    def chain(x, b, stream=None):
        bfp8.bfp8_act_quant_group(x, b["qa"], b["sa"], stream=stream)
        bfp8.bfp8_linear_w8a8_silu_quant(b["qa"], b["sa"], wgu, swgu, b["qh"], b["sh"],
                                         workspace=b["ws1"], stream=stream)
        bfp8.bfp8_linear_w8a8(b["qh"], b["sh"], wd, swd, b["y"], workspace=b["ws2"],
                              stream=stream)

    want = []
    for x in xs:
        b = buffers()
        chain(x, b)
        torch.cuda.synchronize()
        want.append(b["y"])
    streams = [torch.cuda.Stream(device=dev) for _ in xs]
    bufs = [buffers() for _ in xs]
    torch.cuda.synchronize()
    for _ in range(3):
        for x, s, b in zip(xs, streams, bufs):
            chain(x, b, stream=s)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    for b, ref in zip(bufs, want):
        assert torch.equal(b["y"].view(torch.int16), ref.view(torch.int16))
