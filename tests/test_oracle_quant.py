"""Pins for oracle.quant: activation quantizer, weight quantizer, dequant, SiLU glue.

The checks use what the pages and the mathematics fix: the multiply (not
divide) convention and its error gap, the [128,256] -> [1,2] grid, exact BF16
scale expansion, E4M3 rounding bounds, PyTorch's independent float8 cast, and
closed forms of SiLU.
"""

import math

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from conftest import GOLDEN
from oracle import formats as F
from oracle import linear as L
from oracle import quant as Q
from oracle.linear import scale_grid_shape


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _x_bits(M, K, seed=0, outlier="entries", frac=0.01, factor=20.0):
    return _bf16_bits(synth.activations_bf16(synth.generator(seed), M, K, outlier=outlier,
                                             frac=frac, factor=factor))


def test_act_quant_max_element_maps_to_448():
    xb = _x_bits(16, 320)
    q, s = Q.act_quant_group(xb)
    x = F.bf16_bits_to_f32(xb)
    lut = F.e4m3_decode_lut()
    for g in range(3):
        cols = slice(128 * g, min(128 * g + 128, 320))
        idx = np.argmax(np.abs(x[:, cols]), axis=1)
        codes = q[:, cols][np.arange(16), idx]
        assert np.all(np.abs(lut[codes]) == 448.0)


def test_act_quant_error_bound():
    """|e4m3(q) * s - x| within half an E4M3 quantum of x / s."""
    xb = _x_bits(32, 640, seed=3)
    q, s = Q.act_quant_group(xb)
    x = F.bf16_bits_to_f32(xb).astype(np.float64)
    deq = F.e4m3_decode_lut()[q] * np.repeat(s.astype(np.float64), 128, axis=1)[:, :640]
    r = np.abs(x / np.repeat(s.astype(np.float64), 128, axis=1)[:, :640])
    quantum = np.where(r < 2 ** -6, 2 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(r, 2 ** -6))) - 3))
    bound = 0.5 * quantum * np.repeat(s.astype(np.float64), 128, axis=1)[:, :640] * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound + 1e-30)


def test_act_quant_scale_is_amax_over_448():
    xb = _x_bits(8, 256, seed=5)
    _, s = Q.act_quant_group(xb)
    x = F.bf16_bits_to_f32(xb).astype(np.float64)
    amax = np.abs(x.reshape(8, 2, 128)).max(axis=2)
    assert np.allclose(s.astype(np.float64) * 448.0, amax, rtol=2 ** -23, atol=0)


def test_act_quant_zero_group_and_tail_isolation():
    x = np.zeros((2, 320), dtype=np.float32)
    x[1, 300] = 100.0                  # inside the 64-wide tail group only
    xb = F.f32_to_bf16_bits(x)
    q, s = Q.act_quant_group(xb)
    assert np.all(q[0] == 0)
    assert np.all(s[0] == np.float32(np.float32(1e-10) / np.float32(448.0)))
    assert s[1, 0] == s[1, 1] == s[0, 0]
    assert s[1, 2] == np.float32(100.0) / np.float32(448.0)
    assert q[1, 300] == 0x7E


def test_act_quant_matches_torch_composition():
    """Same steps with PyTorch's float32 ops and its independent E4M3 cast."""
    xt = synth.activations_bf16(synth.generator(11), 24, 384, outlier="channels", frac=0.005,
                                factor=30.0)
    q, s = Q.act_quant_group(_bf16_bits(xt))
    xf = xt.float().view(24, 3, 128)
    amax = xf.abs().amax(dim=2, keepdim=True)
    st = torch.clamp(amax, min=1e-10) / 448.0
    qt = (xf / st).to(torch.float8_e4m3fn).view(torch.uint8).view(24, 384).numpy()
    assert np.array_equal(q, qt)
    assert np.array_equal(s, st.view(24, 3).numpy())


def test_act_quant_groups_and_tokens_independent():
    xb = _x_bits(4, 384, seed=7)
    q0, s0 = Q.act_quant_group(xb)
    xb2 = xb.copy()
    xb2[2, 128:256] = F.f32_to_bf16_bits(np.full(128, 3.0, np.float32))
    q1, s1 = Q.act_quant_group(xb2)
    changed = np.zeros_like(q0, dtype=bool)
    changed[2, 128:256] = True
    assert np.array_equal(q0[~changed], q1[~changed])
    assert np.array_equal(np.delete(s0.reshape(-1), 2 * 3 + 1), np.delete(s1.reshape(-1), 2 * 3 + 1))


def _grid_rows():
    out = []
    for line in (GOLDEN / "grid_shapes.txt").read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        n, k, mem, gr, gc, src = line.split()
        members = None if mem == "-" else [int(v) for v in mem.split(",")]
        out.append((int(n), int(k), members, (int(gr), int(gc)), src))
    return out


@pytest.mark.parametrize("N,K,members,grid,src", _grid_rows())
def test_grid_shapes(N, K, members, grid, src):
    assert scale_grid_shape(N, K, members) == grid, src


def test_weight_quant_page_grid_example():
    w = synth.weight_f32(synth.generator(0), 128, 256)
    q, s = Q.quantize_weight_blocks(w.numpy())
    assert q.shape == (128, 256) and s.shape == (1, 2)


def test_multiply_versus_divide_separates():
    """Dequant-multiply is within E4M3 error of the pre-quant weights; the
    reciprocal reading is orders of magnitude off [th#1803 decoder PR, "Proof",
    item 2: a divide is ~1e5 out, not 4%]."""
    w = synth.single_tails(0)["w"].numpy()
    q, s = Q.quantize_weight_blocks(w)
    deq = Q.dequantize_block_scaled(q, s).astype(np.float64)
    rel = np.abs(deq - w) / np.maximum(np.abs(w), 1e-30)
    sf = np.repeat(np.repeat(F.bf16_bits_to_f32(s), 128, 0), 128, 1)[:192, :320].astype(np.float64)
    normal = np.abs(w) / sf >= 2 ** -6
    assert np.all(rel[normal] <= 2 ** -4 * (1 + 2 ** -7))       # E4M3 RNE, BF16 scale rounding
    assert np.all(np.abs(deq - w)[~normal] <= sf[~normal] * 2 ** -10 * (1 + 2 ** -7))
    lut = F.e4m3_decode_lut()
    divided = lut[q] / sf
    rel_div = np.linalg.norm(divided - w) / np.linalg.norm(w)
    rel_mul = np.linalg.norm(deq - w) / np.linalg.norm(w)
    assert rel_mul < 0.05
    assert rel_div > 1e3 * rel_mul


def test_dequant_matches_torch_decode():
    w = synth.weight_f32(synth.generator(2), 300, 200).numpy()
    members = [100, 200]
    q = np.zeros((300, 200), np.uint8)
    s_rows = []
    for lo, hi in [(0, 100), (100, 300)]:
        qi, si = Q.quantize_weight_blocks(w[lo:hi])
        q[lo:hi] = qi
        s_rows.append(si)
    s = np.concatenate(s_rows, axis=0)            # member-local grids stacked: [1 + 2, 2]
    assert s.shape == (3, 2)
    got = Q.dequantize_block_scaled(q, s, members)
    qt = torch.from_numpy(q).view(torch.float8_e4m3fn).float()
    sf = torch.from_numpy(F.bf16_bits_to_f32(s))
    rows = torch.tensor([0] * 100 + [1 + i // 128 for i in range(200)])
    cols = torch.arange(200) // 128
    ref = (qt * sf[rows][:, cols]).numpy()
    assert np.array_equal(got, ref)


def test_weight_quant_f32_scales_and_saturation():
    w = synth.weight_f32(synth.generator(4), 130, 260).numpy()
    q32, s32 = Q.quantize_weight_blocks(w, "f32")
    assert s32.dtype == np.float32 and s32.shape == (2, 3)
    lut = F.e4m3_decode_lut()
    assert np.nanmax(np.abs(lut[q32])) == 448.0
    qb, sb = Q.quantize_weight_blocks(w, "bf16")
    assert np.nanmax(np.abs(lut[qb])) <= 448.0


def test_silu_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 2.0], dtype=np.float32)
    u = np.array([5.0, 1.0, 1.0, 1.0, 1.0, -3.0], dtype=np.float32)
    gu = F.f32_to_bf16_bits(np.concatenate([g, u])[None, :])
    h = F.bf16_bits_to_f32(Q.silu_mul_bf16(gu))[0].astype(np.float64)
    expect = [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.exp(1)), 20.0, 0.0,
              -3 * 2 / (1 + math.exp(-2))]
    assert h[0] == 0.0
    for got, want in zip(h[1:], expect[1:]):
        assert abs(got - want) <= 2 ** -8 * abs(want) + 1e-7
    # silu(g) - silu(-g) = g with u = 1
    assert abs((h[1] - h[2]) - 1.0) <= 2 ** -7


def test_silu_mul_quant_is_quant_of_silu():
    gu = _x_bits(6, 512, seed=9, outlier=None)
    q, s = Q.silu_mul_act_quant(gu)
    q2, s2 = Q.act_quant_group(Q.silu_mul_bf16(gu))
    assert q.shape == (6, 256) and np.array_equal(q, q2) and np.array_equal(s, s2)


# ---- per-tensor scaled weights (the degenerate grid) -------------------------

def test_per_tensor_quant_max_element_and_bound():
    rng = np.random.default_rng(21)
    w = (rng.normal(size=(200, 300)) * 0.02).astype(np.float32)
    w[17, 250] = 0.5                                   # the tensor maximum
    for sd in ("f32", "bf16"):
        q, s = Q.quantize_weight_tensor(w, sd)
        s32 = float(F.bf16_bits_to_f32(s)) if sd == "bf16" else float(s)
        lut = F.e4m3_decode_lut().astype(np.float64)
        if sd == "f32":
            assert s32 == float(np.float32(0.5) / np.float32(448.0))
            assert lut[q[17, 250]] == 448.0            # the maximum maps to the top code
        deq = lut[q] * s32
        # every element within half an E4M3 step of w (relative 2^-4 for
        # normals, 2^-10 * s absolute in the subnormal range)
        err = np.abs(deq - w)
        assert np.all(err <= np.maximum(np.abs(w) * 2.0 ** -4, s32 * 2.0 ** -10) * (1 + 2 ** -8))


def test_tensor_scale_grid_is_the_degenerate_block_case():
    rng = np.random.default_rng(22)
    w = (rng.normal(size=(300, 260)) * 0.02).astype(np.float32)
    q, s = Q.quantize_weight_tensor(w, "f32")
    grid = Q.tensor_scale_grid(s, 300, 260)
    assert grid.shape == (3, 3) and grid.dtype == np.float32 and np.all(grid == s)
    # dequantizing through the grid is e4m3(q) * s, element by element
    assert np.array_equal(Q.dequantize_block_scaled(q, grid),
                          (F.e4m3_decode_lut()[q].astype(np.float32) * np.float32(s)))
    # members: one multiplier covers both members' member-local grids
    gm = Q.tensor_scale_grid(F.f32_to_bf16_bits(np.float32(0.125)), 300, 260, [200, 100])
    assert gm.shape == (2 + 1, 3) and gm.dtype == np.uint16
    assert np.all(F.bf16_bits_to_f32(gm) == np.float32(0.125))


def test_per_tensor_projection_is_plain_matmul_of_dequantized_operands():
    rng = np.random.default_rng(23)
    xb = F.f64_to_bf16_bits(rng.normal(size=(5, 200)))
    q, s = Q.quantize_weight_tensor((rng.normal(size=(140, 200)) * 0.05).astype(np.float32), "f32")
    grid = Q.tensor_scale_grid(s, 140, 200)
    x = F.bf16_bits_to_f32(xb).astype(np.float64)
    wdeq = F.e4m3_decode_lut()[q].astype(np.float64) * float(s)
    assert np.allclose(L.linear_w8a16(xb, q, grid), x @ wdeq.T, rtol=1e-12, atol=1e-12)
