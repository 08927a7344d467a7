"""Quantizers and the reference dequantization.

Test infrastructure (CPU oracle); see the package docstring for who may use it.

* Per-token 1x128 dynamic activation quantization, as in the arithmetic
  paragraph of [Module w8a8_prefill] ("the same arithmetic vLLM uses":
  per-token 1x128 FP32 activation scales). For token m and K-group g, which
  covers columns [128g, min(128g+128, K)):
      amax = max |x|           (float32; the tail group covers only real columns)
      s    = max(amax, 1e-10) / 448      (float32, IEEE division)
      q    = E4M3_RNE_sat(x / s)         (float32 IEEE division, then encode)
  The pages leave three points open. Our readings: an all-zero group takes
  the 1e-10 floor, so its codes are zero; the quotient uses a true division,
  not a multiply by a reciprocal; and rounding is to nearest even with
  saturation.
* Ahead-of-time weight quantization, used only to make synthetic checkpoints.
  Quantization happens ahead of time through conversion endpoints, never at
  load [th#1803 decoder PR, "Why the refusals matter more than the load"].
  Per 128x128 block: s32 = max(amax, 1e-10)/448, stored as BF16 (RNE) or
  F32. Then q = E4M3_RNE_sat(w / s) with s the stored scale widened to f32.
* Per-tensor scaled weights [FP8 Native Serving, "The two FP8 checkpoint
  shapes"]: one multiplier for the whole tensor, s = max(amax, 1e-10)/448
  over every element (synthetic checkpoints only), read as a block case whose
  single block covers the tensor: tensor_scale_grid writes that multiplier
  into every 128x128 block of the member-local grid, so the block-scaled
  projections apply it unchanged.
* dequantize_block_scaled: w = e4m3(q) * s in float32, with s a MULTIPLIER
  despite the "_inv" suffix [Qwen checkpoints with block FP8 weights, first
  paragraph; th#1803 decoder PR, "What lands"].
* SiLU(gate) * up between the gate/up and down projections of the dense FFN
  [Module w8a8_prefill, first paragraph: the gate/up/down GEMM arm]. It is
  computed in float64 as g / (1 + exp(-g)) * u, then rounded once to BF16.
"""

from __future__ import annotations

import numpy as np

from .formats import (
    bf16_bits_to_f32,
    e4m3_decode_lut,
    e4m3_encode_rne_sat,
    f32_to_bf16_bits,
    f64_to_bf16_bits,
)
from .linear import scale_rows

BLOCK = 128
SCALE_FLOOR = np.float32(1e-10)
E4M3_MAX_F32 = np.float32(448.0)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def act_quant_group(x_bits: np.ndarray):
    """Per-token 1x128 quantization of BF16 activations.

    x_bits: uint16 [M, K] BF16 bit patterns.
    Returns (q uint8 [M, K] E4M3 codes, s float32 [M, ceil(K/128)]).
    """
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16))
    M, K = x.shape
    Kb = _ceil_div(K, BLOCK)
    q = np.zeros((M, K), dtype=np.uint8)
    s = np.zeros((M, Kb), dtype=np.float32)
    for g in range(Kb):
        c0, c1 = g * BLOCK, min(g * BLOCK + BLOCK, K)
        grp = x[:, c0:c1]
        amax = np.max(np.abs(grp), axis=1) if M else np.zeros(0, np.float32)
        sg = (np.maximum(amax, SCALE_FLOOR) / E4M3_MAX_F32).astype(np.float32)
        q[:, c0:c1] = e4m3_encode_rne_sat((grp / sg[:, None]).astype(np.float32))
        s[:, g] = sg
    return q, s


def quantize_weight_blocks(w: np.ndarray, scale_dtype: str = "bf16"):
    """Ahead-of-time 128x128 block quantization of a float32 weight [N, K].

    Returns (q uint8 [N, K], scale [ceil(N/128), ceil(K/128)]): uint16 BF16
    bits if scale_dtype == "bf16", float32 if "f32".
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    Nb, Kb = _ceil_div(N, BLOCK), _ceil_div(K, BLOCK)
    q = np.zeros((N, K), dtype=np.uint8)
    s_out = np.zeros((Nb, Kb), dtype=np.uint16 if scale_dtype == "bf16" else np.float32)
    if scale_dtype not in ("bf16", "f32"):
        raise ValueError("scale_dtype must be 'bf16' or 'f32'")
    for nb in range(Nb):
        r0, r1 = nb * BLOCK, min(nb * BLOCK + BLOCK, N)
        for kb in range(Kb):
            c0, c1 = kb * BLOCK, min(kb * BLOCK + BLOCK, K)
            blk = w[r0:r1, c0:c1]
            amax = np.float32(np.max(np.abs(blk)))
            s32 = np.float32(np.maximum(amax, SCALE_FLOOR) / E4M3_MAX_F32)
            if scale_dtype == "bf16":
                sb = f32_to_bf16_bits(s32)
                s_out[nb, kb] = sb
                s = bf16_bits_to_f32(sb)
            else:
                s_out[nb, kb] = s32
                s = s32
            q[r0:r1, c0:c1] = e4m3_encode_rne_sat((blk / np.float32(s)).astype(np.float32))
    return q, s_out


def quantize_weight_tensor(w: np.ndarray, scale_dtype: str = "f32"):
    """Per-tensor quantization of a float32 weight [N, K] (one multiplier).

    Returns (q uint8 [N, K], s): s a float32 scalar array (shape ()) if
    scale_dtype == "f32", or uint16 BF16 bits if "bf16"; q = E4M3_RNE_sat(w / s)
    with s the stored multiplier widened to float32."""
    if scale_dtype not in ("bf16", "f32"):
        raise ValueError("scale_dtype must be 'bf16' or 'f32'")
    w = np.asarray(w, dtype=np.float32)
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    s32 = np.float32(np.maximum(amax, SCALE_FLOOR) / E4M3_MAX_F32)
    if scale_dtype == "bf16":
        s_out = f32_to_bf16_bits(s32)
        s = bf16_bits_to_f32(s_out)
    else:
        s_out = np.array(s32, dtype=np.float32)
        s = s32
    return e4m3_encode_rne_sat((w / np.float32(s)).astype(np.float32)), s_out


def tensor_scale_grid(s, N: int, K: int, members=None) -> np.ndarray:
    """The degenerate grid of a per-tensor multiplier s (BF16 bits or float32):
    s in every block of the member-local grid [sum ceil(N_i/128), ceil(K/128)],
    in s's own storage type."""
    s = np.asarray(s)
    rows = members or [N]
    Nb = sum(_ceil_div(int(n), BLOCK) for n in rows)
    return np.full((Nb, _ceil_div(K, BLOCK)), s.reshape(()), dtype=s.dtype)


def scales_to_f32(s: np.ndarray) -> np.ndarray:
    """Widen a stored scale grid to float32: BF16 bits exactly, F32 unchanged."""
    s = np.asarray(s)
    if s.dtype == np.uint16:
        return bf16_bits_to_f32(s)
    return s.astype(np.float32)


def dequantize_block_scaled(q: np.ndarray, s: np.ndarray, members=None) -> np.ndarray:
    """The reference dequantization: float32 e4m3(q) * s[r(n), k // 128].

    q: uint8 [N, K]; s: scale grid (BF16 bits or float32) [rows, Kb];
    members: member row counts for a grouped tensor (None = one member).
    Multiplied, not divided.
    """
    q = np.asarray(q, dtype=np.uint8)
    N, K = q.shape
    sf = scales_to_f32(s)
    r = scale_rows(N, members)
    kb = np.arange(K) // BLOCK
    vals = e4m3_decode_lut()[q].astype(np.float32)
    return (vals * sf[r][:, kb]).astype(np.float32)


def silu_mul_bf16(gu_bits: np.ndarray) -> np.ndarray:
    """h = bf16( silu(g) * u ) with g = gu[:, :I], u = gu[:, I:], in float64.

    gu_bits: uint16 [M, 2I] BF16 bits (the fused gate/up projection output,
    gate rows first). Returns uint16 [M, I] BF16 bits.
    """
    gu = bf16_bits_to_f32(np.asarray(gu_bits, dtype=np.uint16)).astype(np.float64)
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:2 * I]
    with np.errstate(over="ignore"):
        h = g / (1.0 + np.exp(-g)) * u
    return f64_to_bf16_bits(h)


def silu_mul_act_quant(gu_bits: np.ndarray):
    """SiLU(gate)*up rounded to BF16, then the per-token 1x128 quantizer."""
    return act_quant_group(silu_mul_bf16(gu_bits))
