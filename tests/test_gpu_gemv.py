"""GPU parity: bfp8_gemv_decode (M <= 16) against the oracle's W8A16 definition.

Cases: a one-hot probe with unit scales whose outputs are exact E4M3 values
(it pins the in-register decode, the K permutation and the row mapping);
small ragged shapes; member-local grids; the decode workload's full shapes
(gate/up [34816, 5120], down [5120, 17408], M in {1, 4, 16}) on sampled output
columns, with plain N(0, 1) tokens and with the activation workloads' outlier
patterns (1% of entries x20, 0.5% of channels x30); and bitwise determinism
across calls that share one workspace.
"""

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import (assert_close, bits16, dense_ffn_weights, gpu_bf16_to_f64, quantize_members,
                      sample_indices, scale_to_dev, to_dev_bf16, to_dev_u8)
from oracle import formats as F
from oracle import linear as L

pytestmark = pytest.mark.gpu


def _gemv(bfp8, dev, xb, q, s, members=None):
    M, K = xb.shape
    N = q.shape[0]
    x = to_dev_bf16(xb, dev)
    w = to_dev_u8(q, dev)
    sw = scale_to_dev(s, dev)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(bfp8.bfp8_gemv_decode_workspace(M, N, K), dtype=torch.uint8, device=dev)
    bfp8.bfp8_gemv_decode(x, w, sw, y, ws, member_rows=members)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    return y


def test_gemv_one_hot_exact_decode(bfp8, cuda_device):
    rng = np.random.default_rng(0)
    N, K, M = 256, 512, 16
    q = rng.integers(0, 256, (N, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38                      # no NaN codes
    s = F.f32_to_bf16_bits(np.ones((2, 4), np.float32))
    ks = rng.choice(K, M, replace=False)
    x = np.zeros((M, K), np.float32)
    x[np.arange(M), ks] = 1.0
    y = _gemv(bfp8, cuda_device, F.f32_to_bf16_bits(x), q, s)
    got = gpu_bf16_to_f64(y)
    want = F.e4m3_decode_lut()[q[:, ks].T]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K,members", [
    (1, 192, 320, None), (3, 200, 320, None), (8, 130, 256, None), (9, 384, 640, None),
    (16, 300, 1024, [100, 200]), (5, 1000, 2048, [500, 500]), (16, 256, 128, None),
])
def test_gemv_small(bfp8, cuda_device, M, N, K, members):
    g = synth.generator(M * 1000 + N + K)
    w = synth.weight_f32(g, N, K).numpy()
    xb = bits16(synth.activations_bf16(g, M, K))
    q, s = quantize_members(w, members)
    y = _gemv(bfp8, cuda_device, xb, q, s, members)
    ref = L.linear_w8a16(xb, q, s, members)
    assert_close(gpu_bf16_to_f64(y), ref, f"gemv M={M} N={N} K={K}")


# Token outliers stretch a block's max |x|: the hi/lo E4M3 split carries the
# block's other entries only to within max|x| * 2^-18, so these are its worst
# case at the decode shapes.
DECODE_TOKENS = [(1, None), (4, None), (16, None), (1, "entries"), (16, "entries"),
                 (1, "channels"), (16, "channels")]


@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("M,outlier", DECODE_TOKENS)
def test_gemv_decode_workload(bfp8, cuda_device, which, M, outlier):
    qgu, sgu, qd, sd, _ = dense_ffn_weights(0)
    q, s = (qgu, sgu) if which == "gate_up" else (qd, sd)
    members = [17408, 17408] if which == "gate_up" else None
    N, K = q.shape
    xb = bits16(synth.decode_tokens(100 + M, M, K, outlier))
    y = _gemv(bfp8, cuda_device, xb, q, s, members)
    cols = sample_indices(N, 1500, seed=M)
    ref = L.linear_w8a16(xb, q, s, members, cols=cols)
    assert_close(gpu_bf16_to_f64(y)[:, cols], ref, f"decode {which} M={M} outlier={outlier}")


def test_gemv_deterministic_workspace_reuse(bfp8, cuda_device):
    qgu, sgu, qd, sd, _ = dense_ffn_weights(0)
    dev = cuda_device
    M, K = 16, qd.shape[1]
    N = qd.shape[0]
    x = to_dev_bf16(bits16(synth.decode_tokens(7, M, K)), dev)
    w = to_dev_u8(qd, dev)
    sw = scale_to_dev(sd, dev)
    ws = torch.empty(bfp8.bfp8_gemv_decode_workspace(M, N, K), dtype=torch.uint8, device=dev)
    ys = []
    for _ in range(3):
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_gemv_decode(x, w, sw, y, ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    assert torch.equal(ys[0].view(torch.int16), ys[2].view(torch.int16))


# ---- the W8A8 arm: E4M3 tokens with 1x128 scales (bfp8_gemv_decode_w8a8)

def _gemv_w8a8(bfp8, dev, qa, sa, q, s, members=None):
    M, K = qa.shape
    N = q.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(bfp8.bfp8_gemv_decode_workspace(M, N, K), dtype=torch.uint8, device=dev)
    bfp8.bfp8_gemv_decode_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), to_dev_u8(q, dev),
                               scale_to_dev(s, dev), y, ws, member_rows=members)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    return y


@pytest.mark.parametrize("M,N,K,members", [
    (1, 192, 320, None), (3, 200, 320, None), (8, 130, 256, None), (9, 384, 640, None),
    (16, 300, 1024, [100, 200]), (5, 1000, 2048, [500, 500]), (16, 256, 128, None),
])
def test_gemv_w8a8_small(bfp8, cuda_device, M, N, K, members):
    g = synth.generator(M * 2000 + N + K)
    w = synth.weight_f32(g, N, K).numpy()
    xb = bits16(synth.activations_bf16(g, M, K, outlier="entries", frac=0.01, factor=20.0))
    q, s = quantize_members(w, members)
    from oracle import quant as Q
    qa, sa = Q.act_quant_group(xb)
    y = _gemv_w8a8(bfp8, cuda_device, qa, sa, q, s, members)
    assert_close(gpu_bf16_to_f64(y), L.linear_w8a8(qa, sa, q, s, members), f"gemv w8a8 M={M} N={N} K={K}")


@pytest.mark.parametrize("which", ["gate_up", "down"])
@pytest.mark.parametrize("M,outlier", DECODE_TOKENS)
def test_gemv_w8a8_decode_workload(bfp8, cuda_device, which, M, outlier):
    from oracle import quant as Q
    qgu, sgu, qd, sd, _ = dense_ffn_weights(0)
    q, s = (qgu, sgu) if which == "gate_up" else (qd, sd)
    members = [17408, 17408] if which == "gate_up" else None
    N, K = q.shape
    qa, sa = Q.act_quant_group(bits16(synth.decode_tokens(200 + M, M, K, outlier)))
    y = _gemv_w8a8(bfp8, cuda_device, qa, sa, q, s, members)
    cols = sample_indices(N, 1500, seed=M + 7)
    assert_close(gpu_bf16_to_f64(y)[:, cols], L.linear_w8a8(qa, sa, q, s, members, cols=cols),
                 f"decode w8a8 {which} M={M}")


@pytest.mark.parametrize("arm", ["w8a16", "w8a8"])
def test_gemv_on_a_dirty_workspace(bfp8, cuda_device, arm):
    """Each call zeroes its split-tile counters before the GEMV counts on them
    (the token split, or the W8A8 arm's clearing kernel): a workspace full of
    stale bytes gives the bytes of a zeroed one. At [1000, 2048] every
    128-row tile is split over 16 CTAs, so every output goes through a
    counter."""
    dev = cuda_device
    M, N, K = 5, 1000, 2048
    g = synth.generator(77)
    q, s = quantize_members(synth.weight_f32(g, N, K).numpy(), None)
    xb = bits16(synth.activations_bf16(g, M, K))
    w, sw = to_dev_u8(q, dev), scale_to_dev(s, dev)
    n_ws = bfp8.bfp8_gemv_decode_workspace(M, N, K)
    ys = []
    for fill in (0x00, 0xA5):
        ws = torch.full((n_ws,), fill, dtype=torch.uint8, device=dev)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        if arm == "w8a16":
            bfp8.bfp8_gemv_decode(to_dev_bf16(xb, dev), w, sw, y, ws)
        else:
            from oracle import quant as Q
            qa, sa = Q.act_quant_group(xb)
            bfp8.bfp8_gemv_decode_w8a8(to_dev_u8(qa, dev), torch.from_numpy(sa).to(dev), w, sw,
                                       y, ws)
        torch.cuda.synchronize()
        assert bfp8.bfp8_device_status() == 0
        assert not torch.isnan(y).any()
        ys.append(y)
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
