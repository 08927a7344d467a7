"""The dense-FFN glue as one step (gate/up projection, SiLU(gate)*up, 1x128
quantization of h), and the whole dense-FFN decode step, double precision.

Test infrastructure (CPU oracle); see the package docstring for who may use it.

[Module w8a8_prefill, first paragraph: the gate/up/down GEMM arm.] The step
is defined as the composition of the steps it fuses, in this order:
    gu       = bf16_rn( W8A8 projection with members {I, I} )   (linear_w8a8)
    h        = bf16_rn( silu(gu[:, :I]) * gu[:, I:] )           (silu_mul_bf16)
    q_h, s_h = per-token 1x128 quantization of h                (act_quant_group)
so the BF16 rounding of the projection output sits exactly where the unfused
chain stores it. W stacks the gate rows [0, I) over the up rows [I, 2I), and
its scale grid stacks the gate member's grid over the up member's
(member-local origins, ceil(I/128) rows each).
"""

from __future__ import annotations

import numpy as np

from .formats import f64_to_bf16_bits
from .linear import linear_w8a8, linear_w8a16
from .quant import act_quant_group, silu_mul_act_quant, silu_mul_bf16


def gate_up_silu_quant(q_a, s_a, q_w, s_w, rows=None):
    """Dense: q_a [M, K], s_a [M, Kb], q_w [2I, K], s_w [2*ceil(I/128), Kb].
    Returns (q_h uint8 [len(rows), I], s_h float32 [len(rows), ceil(I/128)])."""
    I = q_w.shape[0] // 2
    gu = linear_w8a8(q_a, s_a, q_w, s_w, [I, I], rows=rows)
    return silu_mul_act_quant(f64_to_bf16_bits(gu))


def grouped_gate_up_silu_quant(q_a, s_a, q_w, s_w, offsets, rows=None):
    """Per-expert form over an expert-sorted token table: q_w [G, 2I, K],
    s_w [G, 2*ceil(I/128), Kb]; row t uses the expert e with
    offsets[e] <= t < offsets[e+1]."""
    q_a = np.asarray(q_a, dtype=np.uint8)
    offsets = np.asarray(offsets, dtype=np.int64)
    T = q_a.shape[0]
    G, I = q_w.shape[0], q_w.shape[1] // 2
    ri = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    expert_of_row = np.searchsorted(offsets, ri, side="right") - 1
    gu = np.zeros((len(ri), 2 * I), dtype=np.float64)
    for e in range(G):
        sel = np.nonzero(expert_of_row == e)[0]
        if sel.size:
            gu[sel] = linear_w8a8(q_a, s_a, q_w[e], s_w[e], [I, I], rows=ri[sel])
    return silu_mul_act_quant(f64_to_bf16_bits(gu))


def decode_ffn(x_bits, q_gu, s_gu, q_d, s_d, arith="w8a16"):
    """The dense-FFN decode step [Module w8a8_prefill, "Reachability": one
    GEMV per projection at decode; first paragraph: the gate/up/down arm],
    as the composition of its projections in their order:
      w8a16: gu = bf16(W8A16 gate/up of x); h = bf16(silu(g)*u);
             y  = W8A16 down of h
      w8a8:  x quantized 1x128; gu = bf16(W8A8 gate/up); h = bf16(silu(g)*u)
             quantized 1x128; y = W8A8 down
    x_bits uint16 [M, H]; q_gu [2I, H] (gate rows over up rows) with its
    member-local grid; q_d [H, I]. Returns float64 [M, H], y before its BF16
    rounding."""
    I = q_gu.shape[0] // 2
    if arith == "w8a16":
        gu = linear_w8a16(x_bits, q_gu, s_gu, [I, I])
        return linear_w8a16(silu_mul_bf16(f64_to_bf16_bits(gu)), q_d, s_d)
    if arith != "w8a8":
        raise ValueError(arith)
    q_a, s_a = act_quant_group(x_bits)
    q_h, s_h = gate_up_silu_quant(q_a, s_a, q_gu, s_gu)
    return linear_w8a8(q_h, s_h, q_d, s_d)
