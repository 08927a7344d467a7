"""GPU parity: the gate/up projection with SiLU(gate)*up and the 1x128
quantization of h fused into its epilogue (bfp8_linear_w8a8_silu_quant,
bfp8_grouped_linear_silu_quant), against the oracle's composition of the
steps it fuses.

The GPU accumulates in FP32 and the oracle in float64, so an element of the
BF16 gate/up product can round to the neighbouring BF16 value, and an h
byte or a group scale then moves with it. Acceptance, per case:
  * codes equal to the oracle's for >= 99.5% of elements;
  * scales within 2^-6 relative of the oracle's;
  * every dequantized h within 2^-3 |h| + 4 * s * 2^-9 of the oracle's h.
The last bound catches swapped gate/up halves, wrong scale rows and wrong
columns; the first two catch anything that is not rare rounding.
The fused result must also be byte-identical to the unfused GPU path (the
W8A8 GEMM writing BF16, then the SiLU*up quantizer), both of which are
parity-tested on their own.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import (bits16, dec_e4m3, dense_ffn_weights, quantize_members, sample_indices,
                      scale_to_dev, to_dev_u8)
from oracle import chain as CH
from oracle import formats as F
from oracle import linear as L
from oracle import quant as Q

pytestmark = pytest.mark.gpu


def _check(q, s, q_ref, s_ref, h_ref_bits, what):
    assert q.shape == q_ref.shape and s.shape == s_ref.shape, what
    agree = float(np.mean(q == q_ref))
    assert agree >= 0.995, f"{what}: codes agree on {agree:.5f}"
    assert np.allclose(s, s_ref, rtol=2 ** -6, atol=0), f"{what}: scales"
    h = F.bf16_bits_to_f32(h_ref_bits).astype(np.float64)
    I = q.shape[1]
    sfull = np.repeat(s_ref.astype(np.float64), 128, axis=1)[:, :I]
    deq = dec_e4m3(q) * np.repeat(s.astype(np.float64), 128, axis=1)[:, :I]
    bad = np.abs(deq - h) > 2 ** -3 * np.abs(h) + 4 * sfull * 2 ** -9
    assert not bad.any(), f"{what}: {int(bad.sum())} dequantized values off"


def _h_ref(qa, sa, qw, sw, rows=None):
    I = qw.shape[0] // 2
    gu = L.linear_w8a8(qa, sa, qw, sw, [I, I], rows=rows)
    return Q.silu_mul_bf16(F.f64_to_bf16_bits(gu))


def _fused(bfp8, dev, qa, sa, qw, sw, stream_k=True):
    M, K = qa.shape
    I = qw.shape[0] // 2
    q = torch.full((M, I), 0xAA, dtype=torch.uint8, device=dev)
    s = torch.full((M, -(-I // 128)), -1.0, dtype=torch.float32, device=dev)
    ws = None
    if stream_k:
        ws = torch.empty(bfp8.bfp8_linear_w8a8_silu_quant_workspace(M, I, K), dtype=torch.uint8,
                         device=dev)
    bfp8.bfp8_linear_w8a8_silu_quant(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev),
                                     to_dev_u8(qw, dev), scale_to_dev(sw, dev), q, s, workspace=ws)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    return q, s


def _unfused(bfp8, dev, qa, sa, qw, sw):
    M, K = qa.shape
    I = qw.shape[0] // 2
    gu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_linear_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(qw, dev),
                          scale_to_dev(sw, dev), gu, member_rows=[I, I])
    q = torch.empty(M, I, dtype=torch.uint8, device=dev)
    s = torch.empty(M, -(-I // 128), dtype=torch.float32, device=dev)
    bfp8.bfp8_silu_mul_act_quant(gu, q, s)
    torch.cuda.synchronize()
    return q, s


SMALL = [
    # M, I, K
    (8, 192, 320),      # tails: a 64-column last group of h, K tail
    (200, 200, 256),    # member-local grids with I off the 128 grid
    (129, 384, 640),
    (1, 128, 128),
    (300, 1000, 512),
]


@pytest.mark.parametrize("stream_k", [True, False], ids=["stream_k", "whole_tiles"])
@pytest.mark.parametrize("M,I,K", SMALL)
def test_fused_small(bfp8, cuda_device, M, I, K, stream_k):
    g = synth.generator(M * 13 + I * 5 + K)
    w = synth.weight_f32(g, 2 * I, K).numpy()
    xb = bits16(synth.activations_bf16(g, M, K, outlier="entries", frac=0.01, factor=20.0))
    qw, sw = quantize_members(w, [I, I])
    qa, sa = Q.act_quant_group(xb)
    q, s = _fused(bfp8, cuda_device, qa, sa, qw, sw, stream_k)
    q_np, s_np = q.cpu().numpy(), s.cpu().numpy()
    q_ref, s_ref = CH.gate_up_silu_quant(qa, sa, qw, sw)
    _check(q_np, s_np, q_ref, s_ref, _h_ref(qa, sa, qw, sw), f"fused {M}x{I}x{K}")
    if not stream_k:  # byte identity needs the same (whole-tile) accumulation order
        qu, su = _unfused(bfp8, cuda_device, qa, sa, qw, sw)
        assert torch.equal(q, qu) and torch.equal(s.view(torch.int32), su.view(torch.int32))


def test_fused_dense_ffn_full_size(bfp8, cuda_device):
    """M=949, I=17408, K=5120: sampled rows against the oracle, every byte
    against the unfused GPU path."""
    qgu, sgu, _, _, xb = dense_ffn_weights(0)
    qa, sa = Q.act_quant_group(xb)
    q, s = _fused(bfp8, cuda_device, qa, sa, qgu, sgu)
    rows = sample_indices(949, 16, seed=21)
    q_ref, s_ref = CH.gate_up_silu_quant(qa, sa, qgu, sgu, rows=rows)
    _check(q.cpu().numpy()[rows], s.cpu().numpy()[rows], q_ref, s_ref,
           _h_ref(qa, sa, qgu, sgu, rows=rows), "fused dense-ffn")
    q, s = _fused(bfp8, cuda_device, qa, sa, qgu, sgu, stream_k=False)
    qu, su = _unfused(bfp8, cuda_device, qa, sa, qgu, sgu)
    assert torch.equal(q, qu) and torch.equal(s.view(torch.int32), su.view(torch.int32))


def _grouped_fused(bfp8, dev, qa, sa, qw, sw, offsets, stream_k=True):
    T, K = qa.shape
    G, I = qw.shape[0], qw.shape[1] // 2
    q = torch.full((T, I), 0xAA, dtype=torch.uint8, device=dev)
    s = torch.full((T, -(-I // 128)), -1.0, dtype=torch.float32, device=dev)
    ws = None
    if stream_k:
        ws = torch.empty(bfp8.bfp8_grouped_linear_silu_quant_workspace(T, G, I, K),
                         dtype=torch.uint8, device=dev)
    off = torch.from_numpy(np.asarray(offsets, dtype=np.int32)).to(dev)
    bfp8.bfp8_grouped_linear_silu_quant(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev),
                                        to_dev_u8(qw, dev), scale_to_dev(sw, dev), off, q, s,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    return q, s


def _stack_members(w, I):
    qs, ss = zip(*[quantize_members(w[e], [I, I]) for e in range(w.shape[0])])
    return np.stack(qs), np.stack(ss)


def _grouped_h_ref(qa, sa, qw, sw, offsets, rows):
    I = qw.shape[1] // 2
    eor = np.searchsorted(np.asarray(offsets), rows, side="right") - 1
    gu = np.zeros((len(rows), 2 * I))
    for e in range(qw.shape[0]):
        sel = np.nonzero(eor == e)[0]
        if sel.size:
            gu[sel] = L.linear_w8a8(qa, sa, qw[e], sw[e], [I, I], rows=rows[sel])
    return Q.silu_mul_bf16(F.f64_to_bf16_bits(gu))


@pytest.mark.parametrize("I", [200, 256])
def test_grouped_fused_small_with_empty_experts(bfp8, cuda_device, I):
    offsets = [0, 3, 3, 200, 330, 331, 331]
    G, K = 6, 256
    g = synth.generator(43 + I)
    qw, sw = _stack_members(synth.weight_stack_f32(g, G, 2 * I, K).numpy(), I)
    xb = bits16(synth.activations_bf16(g, offsets[-1], K, outlier="entries", frac=0.01,
                                       factor=20.0))
    qa, sa = Q.act_quant_group(xb)
    q, s = _grouped_fused(bfp8, cuda_device, qa, sa, qw, sw, offsets)
    rows = np.arange(offsets[-1])
    q_ref, s_ref = CH.grouped_gate_up_silu_quant(qa, sa, qw, sw, offsets)
    _check(q.cpu().numpy(), s.cpu().numpy(), q_ref, s_ref,
           _grouped_h_ref(qa, sa, qw, sw, offsets, rows), f"grouped fused I={I}")


def test_grouped_fused_sparse_experts(bfp8, cuda_device):
    """200 experts, most of them empty: the SiLU warps and the epilogue find
    each tile's expert more than 32 experts past the previous one's."""
    from test_gpu_grouped import sparse_offsets
    offsets = sparse_offsets()
    G, I, K = 200, 128, 256
    g = synth.generator(47)
    qw, sw = _stack_members(synth.weight_stack_f32(g, G, 2 * I, K).numpy(), I)
    xb = bits16(synth.activations_bf16(g, offsets[-1], K))
    qa, sa = Q.act_quant_group(xb)
    q, s = _grouped_fused(bfp8, cuda_device, qa, sa, qw, sw, offsets)
    rows = np.arange(offsets[-1])
    q_ref, s_ref = CH.grouped_gate_up_silu_quant(qa, sa, qw, sw, offsets)
    _check(q.cpu().numpy(), s.cpu().numpy(), q_ref, s_ref,
           _grouped_h_ref(qa, sa, qw, sw, offsets, rows), "grouped fused sparse experts")


def test_grouped_fused_moe_workload(bfp8, cuda_device):
    """8192 tokens x top-8 of 128 experts (65,536 routed rows), hidden 2048,
    expert gate/up [1536, 2048]: sampled rows of every expert against the
    oracle, every byte against the unfused GPU path."""
    d = synth.moe(0)
    c = synth.MOE_PREFILL
    route = L.route_topk(d["logits"].numpy(), c["top_k"])
    offsets = route["offsets"]
    qa, sa = Q.act_quant_group(bits16(d["x"])[route["row_token"]])
    I = c["inter"]
    qw, sw = _stack_members(d["w_gate_up"].numpy(), I)
    q, s = _grouped_fused(bfp8, cuda_device, qa, sa, qw, sw, offsets)
    rng = np.random.default_rng(1)
    rows = []
    for e in range(c["experts"]):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            rows += sorted({lo, hi - 1, int(rng.integers(lo, hi))})
    rows = np.array(rows)
    q_ref, s_ref = CH.grouped_gate_up_silu_quant(qa, sa, qw, sw, offsets, rows=rows)
    _check(q.cpu().numpy()[rows], s.cpu().numpy()[rows], q_ref, s_ref,
           _grouped_h_ref(qa, sa, qw, sw, offsets, rows), "grouped fused moe")
    # unfused GPU path: grouped GEMM to BF16 (I = 768 is on the 128 grid, so the
    # member-local grid is the plain one), then the SiLU*up quantizer; both in
    # whole tiles, so that the accumulation order is the same
    dev = cuda_device
    q, s = _grouped_fused(bfp8, dev, qa, sa, qw, sw, offsets, stream_k=False)
    T, K = qa.shape
    gu = torch.empty(T, 2 * I, dtype=torch.bfloat16, device=dev)
    off = torch.from_numpy(np.asarray(offsets, dtype=np.int32)).to(dev)
    bfp8.bfp8_grouped_linear(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(qw, dev),
                             scale_to_dev(sw, dev), off, gu)
    qu = torch.empty(T, I, dtype=torch.uint8, device=dev)
    su = torch.empty(T, I // 128, dtype=torch.float32, device=dev)
    bfp8.bfp8_silu_mul_act_quant(gu, qu, su)
    torch.cuda.synchronize()
    assert torch.equal(q, qu) and torch.equal(s.view(torch.int32), su.view(torch.int32))
