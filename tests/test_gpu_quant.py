"""GPU parity: quantizers against the CPU oracle.

bfp8_act_quant_group, bfp8_quantize_weight_block and bfp8_silu_mul_act_quant
must be bit-exact: codes and scale bits. So must bfp8_silu_mul's BF16 h: the
oracle evaluates silu(g) * u in float64 and rounds once, and the GPU must give
the same bits on every finite input, including the products that fall next to
a BF16 rounding midpoint (where a float32 evaluation alone could round the
other way).
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


def _silu_quant(bfp8, dev, gu):
    M, I = gu.shape[0], gu.shape[1] // 2
    x = to_dev_bf16(gu, dev)
    q = torch.zeros(M, I, dtype=torch.uint8, device=dev)
    s = torch.zeros(M, -(-I // 128), dtype=torch.float32, device=dev)
    bfp8.bfp8_silu_mul_act_quant(x, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("M,I", [(8, 256), (949, 17408), (33, 768), (3, 100), (65536, 768)])
def test_silu_mul_act_quant(bfp8, cuda_device, M, I):
    """The dense-FFN glue (949 x 17408) and the MoE glue over all routed rows
    (65,536 x 768), bit-exact on codes and scale bits."""
    gu = bits16(synth.activations_bf16(synth.generator(M + I), M, 2 * I))
    q, s = _silu_quant(bfp8, cuda_device, gu)
    qr, sr = Q.act_quant_group(Q.silu_mul_bf16(gu))
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(q, qr)


def _silu_hard_pairs(limit: int, rel: float = 2.0 ** -19):
    """(g, u) BF16 bit pairs whose product silu(g) * u lies within `rel` of a
    BF16 rounding midpoint: the inputs where a float32 evaluation with a few
    ulps of error could round to the wrong neighbour. Found by brute force over
    every finite BF16 g in [-64, 64) and every u in [1, 2)."""
    gb = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        g = F.bf16_bits_to_f32(gb).astype(np.float64)
    keep = np.isfinite(g) & (np.abs(g) < 64) & (g != 0)
    gb, g = gb[keep], g[keep]
    ub = np.arange(0x3F80, 0x4000, dtype=np.uint16)           # every u in [1, 2)
    u = F.bf16_bits_to_f32(ub).astype(np.float64)
    p = (g / (1.0 + np.exp(-g)))[:, None] * u[None, :]
    a = np.abs(p)
    e = np.floor(np.log2(a))
    step = 2.0 ** (np.maximum(e, -126) - 7)                    # BF16 spacing at p
    frac = a / step - np.floor(a / step)                       # position between neighbours
    hard = np.abs(frac - 0.5) * step <= rel * a
    gi, ui = np.nonzero(hard)
    order = np.random.default_rng(11).permutation(gi.size)[:limit]
    return gb[gi[order]], ub[ui[order]]


def test_silu_mul_near_bf16_midpoints(bfp8, cuda_device):
    """Rows built from the hardest (g, u) pairs, with random signs on u: both
    bfp8_silu_mul's h and bfp8_silu_mul_act_quant's codes and scales must be
    exact."""
    g, u = _silu_hard_pairs(64 * 1024)
    assert g.size >= 20000, g.size
    n = (g.size // 1024) * 1024
    signs = (np.random.default_rng(3).integers(0, 2, n).astype(np.uint16) << 15)
    gu = np.concatenate([g[:n].reshape(-1, 1024), (u[:n] | signs).reshape(-1, 1024)], axis=1)
    h = torch.empty(gu.shape[0], 1024, dtype=torch.bfloat16, device=cuda_device)
    bfp8.bfp8_silu_mul(to_dev_bf16(gu, cuda_device), h)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(h), Q.silu_mul_bf16(gu))
    q, s = _silu_quant(bfp8, cuda_device, gu)
    qr, sr = Q.act_quant_group(Q.silu_mul_bf16(gu))
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(q, qr)


def test_silu_mul_every_bf16_gate(bfp8, cuda_device):
    """Every finite BF16 gate value g (all 65,536 patterns but inf and NaN,
    subnormals and the largest magnitudes included) against every up value u
    in [1, 2) and their negatives: 16.7 million products, each h bit-exact."""
    gb = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    gb = gb[np.isfinite(F.bf16_bits_to_f32(gb))]
    I = gb.size
    ub = np.arange(0x3F80, 0x4000, dtype=np.uint16)
    ub = np.concatenate([ub, ub | np.uint16(0x8000)])
    gu = np.empty((ub.size, 2 * I), np.uint16)
    gu[:, :I] = gb[None, :]
    gu[:, I:] = ub[:, None]
    h = torch.empty(ub.size, I, dtype=torch.bfloat16, device=cuda_device)
    bfp8.bfp8_silu_mul(to_dev_bf16(gu, cuda_device), h)
    torch.cuda.synchronize()
    got, ref = bits16(h), Q.silu_mul_bf16(gu)
    bad = got != ref
    assert not bad.any(), (int(bad.sum()), [(hex(gu[r, c]), hex(gu[r, I + c]), hex(got[r, c]),
                                            hex(ref[r, c])) for r, c in np.argwhere(bad)[:5]])


def _near_midpoint_groups(seed=5, n_amax=3000, rel=2.0 ** -22, limit_rows=256):
    """BF16 groups whose quotients x / s sit within ~2 FP32 ulps of an E4M3
    rounding midpoint: the only inputs where a quotient off by one FP32 ulp
    would change a code. Column 0 of each row holds the group maximum."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(n_amax):
        a_bits = np.uint16(rng.integers(0x3F00, 0x4480))     # amax in [0.5, 1024)
        A = F.bf16_bits_to_f32(np.array([a_bits], np.uint16))[0]
        s = np.float32(A) / np.float32(448.0)
        xb = np.arange(1, int(a_bits) + 1, dtype=np.uint16)
        q = F.bf16_bits_to_f32(xb).astype(np.float64) / np.float64(s)
        e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
        unit = np.where(q >= 2.0 ** -6, 2.0 ** e / 16.0, 2.0 ** -10)   # half the E4M3 step
        odd = np.floor(q / unit / 2.0) * 2.0 + 1.0                      # nearest odd multiple
        odd = np.where(np.abs(q / unit - odd) > 1.0, odd + 2.0, odd)
        mid = odd * unit
        hit = np.abs(q - mid) <= rel * mid
        cand = xb[hit]
        if cand.size:
            row = np.zeros(128, np.uint16)
            row[0] = a_bits
            take = cand[:127]
            signs = rng.integers(0, 2, take.size).astype(np.uint16) << 15
            row[1:1 + take.size] = take | signs
            rows.append(row)
        if len(rows) >= limit_rows:
            break
    return np.stack(rows)


def test_act_quant_near_rounding_midpoints(bfp8, cuda_device):
    """The per-group reciprocal + remainder-correction quotient must round
    exactly like IEEE x / s on the inputs where that is hardest."""
    xb = _near_midpoint_groups()
    n_hard = int(np.count_nonzero(xb[:, 1:]))
    assert n_hard >= 100, n_hard
    q, s = _run_act_quant(bfp8, cuda_device, xb)
    qr, sr = Q.act_quant_group(xb)
    assert np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    assert np.array_equal(q, qr)
