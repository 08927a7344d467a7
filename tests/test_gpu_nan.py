"""GPU parity on E4M3 NaN weight codes.

The format has no infinity and two NaN codes, 0x7F and 0xFF [FP8 Native
Serving, "FP8 E4M3: range and quirks"]; the oracle's decode table maps both
to NaN, and a NaN propagates through every sum it enters. A weight row that
holds a NaN code therefore makes its whole output column NaN (0 * NaN is NaN
too), in every arithmetic: W8A8, W8A16, the per-expert projection, both
decode GEMV arms and the decode step.

Each case checks that the GPU's set of NaN outputs equals the oracle's,
element by element, and that every other output is within the GEMM tolerance.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import (assert_close, bits16, gpu_bf16_to_f64, quantize_members, scale_to_dev,
                      to_dev_bf16, to_dev_u8)
from oracle import chain as CH
from oracle import linear as L
from oracle import quant as Q

pytestmark = pytest.mark.gpu

# (row, column, code): rows in three different 128-row tiles, codes in the
# first, a middle and the last K-block, both NaN codes
NAN_AT = [(5, 0, 0x7F), (130, 300, 0xFF), (383, 639, 0x7F), (200, 128, 0xFF)]


def _plant(q, at=NAN_AT):
    q = q.copy()
    for n, k, code in at:
        q[n, k] = code
    return q


def _check(got, ref, what):
    got_nan, ref_nan = np.isnan(got), np.isnan(ref)
    assert ref_nan.any(), what
    assert np.array_equal(got_nan, ref_nan), (
        what, np.argwhere(got_nan != ref_nan)[:5].tolist())
    fin = ~ref_nan
    assert_close(got[fin], ref[fin], what)


def _weights(N=384, K=640, seed=7):
    g = synth.generator(seed)
    q, s = quantize_members(synth.weight_f32(g, N, K).numpy())
    return g, _plant(q), s


def test_nan_codes_w8a8_and_w8a16(bfp8, cuda_device):
    dev = cuda_device
    g, q, s = _weights()
    M, K = 20, q.shape[1]
    xb = bits16(synth.activations_bf16(g, M, K))
    qa, sa = Q.act_quant_group(xb)
    w, sw = to_dev_u8(q, dev), scale_to_dev(s, dev)
    y8 = torch.empty(M, q.shape[0], dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_linear_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), w, sw, y8)
    y16 = torch.empty_like(y8)
    bfp8.bfp8_linear_w8a16(to_dev_bf16(xb, dev), w, sw, y16)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    _check(gpu_bf16_to_f64(y8), L.linear_w8a8(qa, sa, q, s), "w8a8")
    _check(gpu_bf16_to_f64(y16), L.linear_w8a16(xb, q, s), "w8a16")


def test_nan_codes_gemv_both_arms(bfp8, cuda_device):
    dev = cuda_device
    g, q, s = _weights(seed=8)
    M, N, K = 4, q.shape[0], q.shape[1]
    xb = bits16(synth.activations_bf16(g, M, K))
    qa, sa = Q.act_quant_group(xb)
    w, sw = to_dev_u8(q, dev), scale_to_dev(s, dev)
    ws = torch.empty(bfp8.bfp8_gemv_decode_workspace(M, N, K), dtype=torch.uint8, device=dev)
    y16 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_gemv_decode(to_dev_bf16(xb, dev), w, sw, y16, ws)
    y8 = torch.empty_like(y16)
    bfp8.bfp8_gemv_decode_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), w, sw, y8, ws)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    _check(gpu_bf16_to_f64(y16), L.linear_w8a16(xb, q, s), "gemv w8a16")
    _check(gpu_bf16_to_f64(y8), L.linear_w8a8(qa, sa, q, s), "gemv w8a8")


def test_nan_codes_grouped(bfp8, cuda_device):
    dev = cuda_device
    offsets = [0, 40, 40, 300, 333]
    G, N, K = 4, 384, 256
    g = synth.generator(9)
    wst = synth.weight_stack_f32(g, G, N, K).numpy()
    qs, ss = zip(*[Q.quantize_weight_blocks(wst[e]) for e in range(G)])
    qw, sw = np.stack(qs), np.stack(ss)
    qw[2] = _plant(qw[2], [(7, 3, 0x7F), (260, 255, 0xFF)])     # expert 2: rows 40..299
    qw[1] = _plant(qw[1], [(9, 9, 0x7F)])                        # expert 1 has no rows
    xb = bits16(synth.activations_bf16(g, offsets[-1], K))
    qa, sa = Q.act_quant_group(xb)
    y = torch.empty(offsets[-1], N, dtype=torch.bfloat16, device=dev)
    off = torch.tensor(offsets, dtype=torch.int32, device=dev)
    bfp8.bfp8_grouped_linear(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(qw, dev),
                             scale_to_dev(sw, dev), off, y)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    _check(gpu_bf16_to_f64(y), L.grouped_linear_w8a8(qa, sa, qw, sw, np.array(offsets)), "grouped")


@pytest.mark.parametrize("arith", ["w8a16", "w8a8"])
def test_nan_codes_decode_step(bfp8, cuda_device, arith):
    """A NaN code in the down weight makes its output column NaN; one in the
    gate/up weight poisons h and with it every output of the step."""
    dev = cuda_device
    M, H, I = 2, 256, 384
    g = synth.generator(10)
    qgu, sgu = quantize_members(synth.weight_f32(g, 2 * I, H).numpy(), [I, I])
    qd, sd = quantize_members(synth.weight_f32(g, H, I).numpy())
    xb = bits16(synth.activations_bf16(g, M, H))
    code = bfp8.BFP8_DECODE_W8A16 if arith == "w8a16" else bfp8.BFP8_DECODE_W8A8
    ws = torch.empty(bfp8.bfp8_decode_ffn_workspace(M, H, I, code), dtype=torch.uint8, device=dev)
    for what, qgu_, qd_ in [("down", qgu, _plant(qd, [(17, 5, 0xFF), (200, 383, 0x7F)])),
                            ("gate/up", _plant(qgu, [(3, 100, 0x7F)]), qd)]:
        y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_decode_ffn(to_dev_bf16(xb, dev), to_dev_u8(qgu_, dev), scale_to_dev(sgu, dev),
                             to_dev_u8(qd_, dev), scale_to_dev(sd, dev), y, ws, arith=code)
        torch.cuda.synchronize()
        assert bfp8.bfp8_device_status() == 0
        ref = CH.decode_ffn(xb, qgu_, sgu, qd_, sd, arith=arith)
        got = gpu_bf16_to_f64(y)
        if what == "gate/up":
            assert np.isnan(ref).all() and np.isnan(got).all(), (arith, what)
        else:
            _check(got, ref, f"decode step {arith} ({what})")
