"""GPU parity: bfp8_grouped_linear (per-expert W8A8 over a token-offset table).

A small case with empty and ragged experts is checked in full. The MoE
workload (8192 tokens, top-8 of 128 experts from a softmax over seeded N(0,1)
router logits, hidden 2048, expert gate/up [1536, 2048], down [2048, 768]) is
checked on sampled rows from every expert, with the oracle's own routing
table as input.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import assert_close, bits16, gpu_bf16_to_f64, scale_to_dev, to_dev_u8
from oracle import linear as L
from oracle import quant as Q

pytestmark = pytest.mark.gpu


def _grouped(bfp8, dev, qa, sa, qw, sw, offsets, stream_k=True):
    T, K = qa.shape
    G, N = qw.shape[0], qw.shape[1]
    y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device=dev)
    off = torch.from_numpy(np.asarray(offsets, dtype=np.int32)).to(dev)
    ws = None
    if stream_k:
        ws = torch.empty(bfp8.bfp8_grouped_linear_workspace(T, G, N, K), dtype=torch.uint8,
                         device=dev)
    bfp8.bfp8_grouped_linear(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(qw, dev),
                             scale_to_dev(sw, dev), off, y, workspace=ws)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    return y


def _stack_quant(w):
    G = w.shape[0]
    qs, ss = zip(*[Q.quantize_weight_blocks(w[e]) for e in range(G)])
    return np.stack(qs), np.stack(ss)


@pytest.mark.parametrize("stream_k", [True, False], ids=["stream_k", "whole_tiles"])
def test_grouped_small_with_empty_experts(bfp8, cuda_device, stream_k):
    offsets = [0, 3, 3, 200, 330, 331, 331]
    G, N, K = 6, 384, 256
    g = synth.generator(41)
    qw, sw = _stack_quant(synth.weight_stack_f32(g, G, N, K).numpy())
    xb = bits16(synth.activations_bf16(g, offsets[-1], K, outlier="entries", frac=0.01, factor=20.0))
    qa, sa = Q.act_quant_group(xb)
    y = gpu_bf16_to_f64(_grouped(bfp8, cuda_device, qa, sa, qw, sw, offsets, stream_k))
    assert_close(y, L.grouped_linear_w8a8(qa, sa, qw, sw, offsets), "grouped small")


# 200 experts, a few with rows, the others empty: a tile's expert can lie more
# than 32 experts past the previous tile's, so every walker's expert lookup
# (a warp-wide ballot over 32 expert boundaries at a time) takes several steps.
SPARSE_ROWS = {0: 130, 37: 60, 75: 200, 76: 5, 150: 129, 199: 70}


def sparse_offsets(G=200):
    offsets = [0]
    for e in range(G):
        offsets.append(offsets[-1] + SPARSE_ROWS.get(e, 0))
    return offsets


@pytest.mark.parametrize("stream_k", [True, False], ids=["stream_k", "whole_tiles"])
def test_grouped_sparse_experts(bfp8, cuda_device, stream_k):
    offsets = sparse_offsets()
    G, N, K = 200, 256, 256
    g = synth.generator(45)
    qw, sw = _stack_quant(synth.weight_stack_f32(g, G, N, K).numpy())
    xb = bits16(synth.activations_bf16(g, offsets[-1], K))
    qa, sa = Q.act_quant_group(xb)
    y = gpu_bf16_to_f64(_grouped(bfp8, cuda_device, qa, sa, qw, sw, offsets, stream_k))
    assert_close(y, L.grouped_linear_w8a8(qa, sa, qw, sw, offsets), "grouped sparse experts")


def test_grouped_moe_workload(bfp8, cuda_device):
    d = synth.moe(0)
    c = synth.MOE_PREFILL
    route = L.route_topk(d["logits"].numpy(), c["top_k"])
    offsets = route["offsets"]
    assert offsets[-1] == c["tokens"] * c["top_k"]
    xs = bits16(d["x"])[route["row_token"]]          # expert-sorted rows
    qa, sa = Q.act_quant_group(xs)
    qgu, sgu = _stack_quant(d["w_gate_up"].numpy())
    assert sgu.shape == (128, 12, 16)
    y = gpu_bf16_to_f64(_grouped(bfp8, cuda_device, qa, sa, qgu, sgu, offsets))
    rng = np.random.default_rng(0)
    rows = []
    for e in range(128):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            rows += sorted({lo, hi - 1, int(rng.integers(lo, hi))})
    rows = np.array(rows)
    cols = np.unique(np.concatenate([rng.choice(1536, 64, replace=False), [0, 767, 768, 1535]]))
    ref = L.grouped_linear_w8a8(qa, sa, qgu, sgu, offsets, rows=rows, cols=cols)
    assert_close(y[np.ix_(rows, cols)], ref, "moe gate/up")
    # down projection on quantized SiLU(gate)*up of the oracle's own rows
    h = bits16(synth.activations_bf16(synth.generator(9), qa.shape[0], c["inter"]))
    qh, sh = Q.act_quant_group(h)
    qd, sd = _stack_quant(d["w_down"].numpy())
    yd = gpu_bf16_to_f64(_grouped(bfp8, cuda_device, qh, sh, qd, sd, offsets))
    cols = np.unique(np.concatenate([rng.choice(2048, 64, replace=False), [0, 2047]]))
    assert_close(yd[np.ix_(rows, cols)],
                 L.grouped_linear_w8a8(qh, sh, qd, sd, offsets, rows=rows, cols=cols), "moe down")


@pytest.mark.parametrize("pad", [8, 3], ids=["ldy_aligned", "ldy_unaligned"])
def test_grouped_strided_output_keeps_padding(bfp8, cuda_device, pad):
    """y as a row-strided view: with a 16-byte aligned row pitch, whole
    32-row warp tiles go out by TMA tensor stores (clipped at column N), the
    rows of an expert's last partial group by the masked warp stores; with an
    unaligned pitch every store is a masked warp store. Either way the
    padding columns and nothing else stay untouched. Expert sizes put tile
    and 32-row boundaries on both sides of the split."""
    dev = cuda_device
    offsets = [0, 32, 96, 96, 224, 385, 386, 514]
    G, N, K = 7, 320, 384
    g = synth.generator(43)
    qw, sw = _stack_quant(synth.weight_stack_f32(g, G, N, K).numpy())
    xb = bits16(synth.activations_bf16(g, offsets[-1], K))
    qa, sa = Q.act_quant_group(xb)
    T = offsets[-1]
    yb = torch.full((T, N + pad), float("nan"), dtype=torch.bfloat16, device=dev)
    y = yb[:, :N]
    off = torch.from_numpy(np.asarray(offsets, dtype=np.int32)).to(dev)
    bfp8.bfp8_grouped_linear(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(qw, dev),
                             scale_to_dev(sw, dev), off, y)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    assert torch.isnan(yb[:, N:].float()).all()
    assert_close(gpu_bf16_to_f64(y), L.grouped_linear_w8a8(qa, sa, qw, sw, offsets), f"grouped pad {pad}")


def test_grouped_on_two_streams_at_once(bfp8, cuda_device):
    """Two per-expert projections with different offset tables in flight at
    once on two streams, each with its own stream-K workspace, give the bytes
    of the same calls run one after the other (each CTA builds its tile
    schedule from its own call's table)."""
    dev = cuda_device
    G, N, K = 6, 384, 256
    tables = ([0, 3, 3, 200, 330, 331, 331], [0, 0, 129, 129, 129, 250, 331])
    g = synth.generator(42)
    qw, sw = _stack_quant(synth.weight_stack_f32(g, G, N, K).numpy())
    xb = bits16(synth.activations_bf16(g, 331, K, outlier="entries", frac=0.01, factor=20.0))
    qa, sa = Q.act_quant_group(xb)
    want = [_grouped(bfp8, dev, qa, sa, qw, sw, t) for t in tables]
    a, sad = to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev)
    w, swd = to_dev_u8(qw, dev), scale_to_dev(sw, dev)
    offs = [torch.tensor(t, dtype=torch.int32, device=dev) for t in tables]
    wss = [torch.empty(bfp8.bfp8_grouped_linear_workspace(331, G, N, K), dtype=torch.uint8,
                       device=dev) for _ in tables]
    ys = [torch.empty(331, N, dtype=torch.bfloat16, device=dev) for _ in tables]
    streams = [torch.cuda.Stream(device=dev) for _ in tables]
    torch.cuda.synchronize()
    for _ in range(3):
        for off, ws, y, s in zip(offs, wss, ys, streams):
            bfp8.bfp8_grouped_linear(a, sad, w, swd, off, y, workspace=ws, stream=s)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    for y, ref in zip(ys, want):
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
