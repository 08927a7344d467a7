"""GPU parity: bfp8_linear_w8a8 and bfp8_linear_w8a16 (tcgen05 / TMEM) against
the oracle.

Small cases cover every output element: tails on both axes, several tiles,
M = 1, member-local grids with members that are not multiples of 128, F32
scales, the token-contiguous activation-scale layout and a padded output
stride. Full-size cases (dense-FFN gate/up and down at M = 949, attention
QKV with its three member grids and O at M = 4096) compare sampled rows and
columns that span every tile type and the ragged ends.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import (assert_close, bits16, cos_rrms, dense_ffn_weights, gpu_bf16_to_f64,
                      quantize_members, sample_indices, scale_to_dev, to_dev_bf16, to_dev_u8)
from oracle import linear as L
from oracle import quant as Q

pytestmark = pytest.mark.gpu


def _w8a8(bfp8, dev, qa, sa, q, s, members=None, mn_major=False, ldy_pad=0, stream_k=True):
    M, K = qa.shape
    N = q.shape[0]
    ws = None
    if stream_k:
        ws = torch.empty(bfp8.bfp8_linear_w8a8_workspace(M, N, K, members), dtype=torch.uint8,
                         device=dev)
    a = to_dev_u8(qa, dev)
    if mn_major:
        sa_d = torch.from_numpy(np.ascontiguousarray(sa.T)).to(dev)
        sa_kw = dict(s_stride_m=1, s_stride_kb=M)
    else:
        sa_d = torch.from_numpy(np.ascontiguousarray(sa)).to(dev)
        sa_kw = {}
    ybuf = torch.full((M, N + ldy_pad), -7.0, dtype=torch.bfloat16, device=dev)
    y = ybuf[:, :N]
    bfp8.bfp8_linear_w8a8(a, sa_d, to_dev_u8(q, dev), scale_to_dev(s, dev), y,
                          member_rows=members, workspace=ws, **sa_kw)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    if ldy_pad:
        assert torch.all(ybuf[:, N:] == -7.0), "padding columns were written"
    return y


def _w8a16(bfp8, dev, xb, q, s, members=None):
    M, K = xb.shape
    N = q.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_linear_w8a16(to_dev_bf16(xb, dev), to_dev_u8(q, dev), scale_to_dev(s, dev), y,
                           member_rows=members)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    return y


def _problem(seed, M, N, K, members=None, scale_dtype="bf16", outlier="entries"):
    g = synth.generator(seed)
    w = synth.weight_f32(g, N, K).numpy()
    xb = bits16(synth.activations_bf16(g, M, K, outlier=outlier, frac=0.01, factor=20.0))
    q, s = quantize_members(w, members, scale_dtype)
    return xb, q, s


SMALL = [
    # M, N, K, members, scale dtype
    (8, 192, 320, None, "bf16"),            # the single-linear workload (tails on both axes)
    (1, 128, 128, None, "bf16"),
    (200, 448, 256, [70, 250, 128], "bf16"),  # member-local origins off the 128 grid
    (300, 600, 640, None, "f32"),
    (129, 256, 384, None, "bf16"),
    (64, 520, 1152, [8, 512], "bf16"),
]


@pytest.mark.parametrize("stream_k", [True, False], ids=["stream_k", "whole_tiles"])
@pytest.mark.parametrize("M,N,K,members,sdt", SMALL)
def test_w8a8_small(bfp8, cuda_device, M, N, K, members, sdt, stream_k):
    xb, q, s = _problem(M * 31 + N * 7 + K, M, N, K, members, sdt)
    qa, sa = Q.act_quant_group(xb)
    y = _w8a8(bfp8, cuda_device, qa, sa, q, s, members, stream_k=stream_k)
    ref = L.linear_w8a8(qa, sa, q, s, members)
    assert_close(gpu_bf16_to_f64(y), ref, f"w8a8 {M}x{N}x{K}")


def test_w8a8_stream_k_deterministic(bfp8, cuda_device):
    """Split tiles are summed in a fixed order: repeated calls give identical bytes,
    and the workspace counters come back clean for the next call."""
    xb, q, s = _problem(77, 300, 1024, 4096)
    qa, sa = Q.act_quant_group(xb)
    dev = cuda_device
    a, sad = to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev)
    w, swd = to_dev_u8(q, dev), scale_to_dev(s, dev)
    ws = torch.empty(bfp8.bfp8_linear_w8a8_workspace(300, 1024, 4096), dtype=torch.uint8, device=dev)
    ys = []
    for _ in range(3):
        y = torch.empty(300, 1024, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_linear_w8a8(a, sad, w, swd, y, workspace=ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    assert torch.equal(ys[0].view(torch.int16), ys[2].view(torch.int16))
    assert_close(gpu_bf16_to_f64(ys[0]), L.linear_w8a8(qa, sa, q, s), "stream-K")


def test_stream_k_workspaces_full_of_stale_bytes(bfp8, cuda_device):
    """Every call clears its stream-K tile counters on its stream before the
    kernel runs, and each partial tile is written before it is read, so a
    workspace full of stale bytes gives the bytes of a zeroed one: the dense
    projection, the fused gate/up and the per-expert projection, each at a
    size whose tail wave is split."""
    dev = cuda_device
    xb, q, s = _problem(78, 300, 1024, 4096)
    qa, sa = Q.act_quant_group(xb)
    a, sad = to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev)
    w, swd = to_dev_u8(q, dev), scale_to_dev(s, dev)
    I = 512                                                # fused: [gate; up] = the first 1024 rows

    def dense(ws):
        y = torch.full((300, 1024), float("nan"), dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_linear_w8a8(a, sad, w, swd, y, workspace=ws)
        return [y.view(torch.int16)]

    def fused(ws):
        qh = torch.full((300, I), 0xAA, dtype=torch.uint8, device=dev)
        sh = torch.full((300, I // 128), -1.0, dtype=torch.float32, device=dev)
        bfp8.bfp8_linear_w8a8_silu_quant(a, sad, w, swd, qh, sh, workspace=ws)
        return [qh, sh.view(torch.int32)]

    G, T = 3, 300
    off = torch.tensor([0, 7, 7, T], dtype=torch.int32, device=dev)
    wg = w[:768].reshape(1, 768, 4096).expand(G, 768, 4096).contiguous()
    sg = swd[:6].reshape(1, 6, 32).expand(G, 6, 32).contiguous()

    def grouped(ws):
        y = torch.full((T, 768), float("nan"), dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_grouped_linear(a, sad, wg, sg, off, y, workspace=ws)
        return [y.view(torch.int16)]

    for name, call, n_ws in (
            ("dense", dense, bfp8.bfp8_linear_w8a8_workspace(300, 1024, 4096)),
            ("fused", fused, bfp8.bfp8_linear_w8a8_silu_quant_workspace(300, I, 4096)),
            ("grouped", grouped, bfp8.bfp8_grouped_linear_workspace(T, G, 768, 4096))):
        assert n_ws > 0, name
        outs = []
        for fill in (0x00, 0xA5):
            outs.append(call(torch.full((n_ws,), fill, dtype=torch.uint8, device=dev)))
        torch.cuda.synchronize()
        assert bfp8.bfp8_device_status() == 0
        for u, v in zip(*outs):
            assert torch.equal(u, v), name
    ref = L.linear_w8a8(qa, sa, q, s)
    y = torch.empty(300, 1024, dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_linear_w8a8(a, sad, w, swd, y,
                          workspace=torch.full((bfp8.bfp8_linear_w8a8_workspace(300, 1024, 4096),),
                                               0xA5, dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    assert_close(gpu_bf16_to_f64(y), ref, "stream-K on a stale workspace")


def test_w8a8_mn_major_scales_and_padded_output(bfp8, cuda_device):
    xb, q, s = _problem(5, 150, 320, 512)
    qa, sa = Q.act_quant_group(xb)
    y = _w8a8(bfp8, cuda_device, qa, sa, q, s, mn_major=True, ldy_pad=24)
    assert_close(gpu_bf16_to_f64(y), L.linear_w8a8(qa, sa, q, s), "w8a8 mn-major")


@pytest.mark.parametrize("M,N,K,members,sdt", SMALL)
def test_w8a16_small(bfp8, cuda_device, M, N, K, members, sdt):
    xb, q, s = _problem(M * 17 + N * 3 + K, M, N, K, members, sdt)
    y = _w8a16(bfp8, cuda_device, xb, q, s, members)
    ref = L.linear_w8a16(xb, q, s, members)
    assert_close(gpu_bf16_to_f64(y), ref, f"w8a16 {M}x{N}x{K}")


def test_w8a8_vs_w8a16_accuracy_gate(bfp8, cuda_device):
    """GPU W8A8 against the W8A16 oracle: cosine >= 0.999, relative RMS <= 2%
    [Module w8a8_prefill, "ACCURACY"], on the single-linear workload."""
    d = synth.single_tails(0)
    q, s = Q.quantize_weight_blocks(d["w"].numpy())
    xb = bits16(d["x"])
    qa, sa = Q.act_quant_group(xb)
    y = gpu_bf16_to_f64(_w8a8(bfp8, cuda_device, qa, sa, q, s))
    cos, rrms = cos_rrms(y, L.linear_w8a16(xb, q, s))
    assert cos >= 0.999 and rrms <= 0.02


@pytest.mark.parametrize("stream_k", [True, False], ids=["stream_k", "whole_tiles"])
@pytest.mark.parametrize("which", ["gate_up", "down"])
def test_w8a8_dense_ffn_full_size(bfp8, cuda_device, which, stream_k):
    qgu, sgu, qd, sd, xb = dense_ffn_weights(0)
    if which == "gate_up":
        q, s, members = qgu, sgu, [17408, 17408]
        qa, sa = Q.act_quant_group(xb)
    else:
        q, s, members = qd, sd, None
        h = bits16(synth.activations_bf16(synth.generator(77), 949, 17408))
        qa, sa = Q.act_quant_group(h)
    y = gpu_bf16_to_f64(_w8a8(bfp8, cuda_device, qa, sa, q, s, members, stream_k=stream_k))
    rows = sample_indices(qa.shape[0], 48, seed=1)
    cols = sample_indices(q.shape[0], 700, seed=2)
    ref = L.linear_w8a8(qa, sa, q, s, members, rows=rows, cols=cols)
    assert_close(y[np.ix_(rows, cols)], ref, f"dense-ffn {which}")


def test_w8a8_attention_full_size(bfp8, cuda_device):
    d = synth.attention(0)
    members = [8192, 1024, 1024]
    wqkv = np.concatenate([d["w_q"].numpy(), d["w_k"].numpy(), d["w_v"].numpy()])
    q, s = quantize_members(wqkv, members)
    assert s.shape == (80, 40)
    qo, so = Q.quantize_weight_blocks(d["w_o"].numpy())
    xb = bits16(d["x"])
    qa, sa = Q.act_quant_group(xb)
    y = gpu_bf16_to_f64(_w8a8(bfp8, cuda_device, qa, sa, q, s, members))
    rows = sample_indices(4096, 40, seed=3)
    cols = np.unique(np.concatenate([sample_indices(10240, 600, seed=4),
                                     [8191, 8192, 9215, 9216, 10239]]))
    assert_close(y[np.ix_(rows, cols)], L.linear_w8a8(qa, sa, q, s, members, rows=rows, cols=cols),
                 "qkv")
    ctx = bits16(synth.activations_bf16(synth.generator(5), 4096, 8192))
    qc, sc = Q.act_quant_group(ctx)
    yo = gpu_bf16_to_f64(_w8a8(bfp8, cuda_device, qc, sc, qo, so))
    cols = sample_indices(5120, 500, seed=6)
    assert_close(yo[np.ix_(rows, cols)], L.linear_w8a8(qc, sc, qo, so, rows=rows, cols=cols), "o")


def test_w8a16_dense_ffn_gate_up_full_size(bfp8, cuda_device):
    qgu, sgu, _, _, xb = dense_ffn_weights(0)
    y = gpu_bf16_to_f64(_w8a16(bfp8, cuda_device, xb, qgu, sgu, [17408, 17408]))
    rows = sample_indices(949, 24, seed=8)
    cols = sample_indices(34816, 400, seed=9)
    assert_close(y[np.ix_(rows, cols)],
                 L.linear_w8a16(xb, qgu, sgu, [17408, 17408], rows=rows, cols=cols), "w8a16 gu")


@pytest.mark.parametrize("M,N,K,members", [
    (949, 10240, 5120, [8192, 1024, 1024]),   # 320 tiles: 152 whole, then 168 split in 19 groups of 8
    (1064, 5120, 2048, None),                 # 180 tiles, all split: 16 groups of 9, 8 CTAs idle
])
def test_w8a8_stream_k_lockstep_geometries(bfp8, cuda_device, M, N, K, members):
    """Split tiles in lockstep groups (one CTA per M tile of an (N tile,
    K-block) range): against the oracle on sampled rows and columns, within
    two BF16 roundings of the whole-tile result everywhere, and
    byte-identical from call to call."""
    dev = cuda_device
    xb, q, s = _problem(91 + M, M, N, K, members)
    qa, sa = Q.act_quant_group(xb)
    y1 = _w8a8(bfp8, dev, qa, sa, q, s, members)
    y2 = _w8a8(bfp8, dev, qa, sa, q, s, members)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    yw = gpu_bf16_to_f64(_w8a8(bfp8, dev, qa, sa, q, s, members, stream_k=False))
    y = gpu_bf16_to_f64(y1)
    rows = sample_indices(M, 40, seed=M)
    cols = sample_indices(N, 500, seed=N)
    assert_close(y[np.ix_(rows, cols)], L.linear_w8a8(qa, sa, q, s, members, rows=rows, cols=cols),
                 f"lockstep stream-K {M}x{N}x{K}")
    # both results are BF16 roundings (unit roundoff 2^-8 each) of FP32 sums
    # that differ only in summation order: at most 2^-7 apart, relatively
    rms = float(np.sqrt(np.mean(yw ** 2)))
    assert np.all(np.abs(y - yw) <= 2.0 ** -7 * np.abs(yw) + 1e-4 * rms), "stream-K vs whole tiles"
