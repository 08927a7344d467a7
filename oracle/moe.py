"""The steps on either side of the grouped MoE projection, and the MoE FFN
layer they close, double precision.

Test infrastructure (CPU oracle); see the package docstring for who may use it.

[Module w8a8_prefill, "WHY": the MoE expert path runs on the block-scaled
W8A8 prefill arm; arithmetic paragraph: per-token 1x128 FP32 activation
scales.] The pages name the expert path but print neither the permutation
nor the combine. The plainest reading, which the rest of the pages support:
  * gather_act_quant: the expert-sorted row r holds token row_token[r]; it is
    quantized exactly as act_quant_group quantizes that token, so permuting
    before or after quantizing gives the same bytes. A row whose token index
    is outside [0, T) is a zero row.
  * combine: out[t] = bf16_rn( sum_j w[t, j] * y[row_of[t, j]] ), the sum
    exact (float64) over the token's top-k slots, with w the renormalized
    router weights (route_topk). A row index outside [0, R) adds nothing.
  * moe_layer: route -> gather + quantize -> per-expert gate/up with
    SiLU(gate)*up and 1x128 quantization of h -> per-expert down, rounded to
    BF16 as the down projection stores it -> combine.
"""

from __future__ import annotations

import numpy as np

from .chain import grouped_gate_up_silu_quant
from .formats import bf16_bits_to_f32, f64_to_bf16_bits
from .linear import grouped_linear_w8a8
from .quant import act_quant_group


def gather_act_quant(x_bits, row_token):
    """x_bits uint16 [T, H] BF16; row_token int [R].
    Returns (q uint8 [R, H], s float32 [R, ceil(H/128)])."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    idx = np.asarray(row_token, dtype=np.int64)
    valid = (idx >= 0) & (idx < T)
    rows = np.zeros((len(idx), H), dtype=np.uint16)
    rows[valid] = x_bits[idx[valid]]
    return act_quant_group(rows)


def combine_f64(y_bits, row_of, weights):
    """The exact weighted sum before rounding: y_bits uint16 [R, H] BF16,
    row_of int [T, k], weights [T, k] (widened to float64). Returns float64 [T, H]."""
    y = bf16_bits_to_f32(np.asarray(y_bits, dtype=np.uint16)).astype(np.float64)
    R, H = y.shape
    rows = np.asarray(row_of, dtype=np.int64)
    w = np.asarray(weights, dtype=np.float64)
    T, k = rows.shape
    out = np.zeros((T, H), dtype=np.float64)
    for j in range(k):
        r = rows[:, j]
        ok = (r >= 0) & (r < R)
        out[ok] += w[ok, j, None] * y[r[ok]]
    return out


def combine(y_bits, row_of, weights):
    """combine_f64 rounded once to BF16 (uint16 bits [T, H])."""
    return f64_to_bf16_bits(combine_f64(y_bits, row_of, weights))


def moe_layer(x_bits, route, q_gu, s_gu, q_d, s_d, tokens=None):
    """The MoE FFN for the tokens listed (all by default).

    x_bits uint16 [T, H]; route from route_topk; q_gu [E, 2I, H] with each
    expert's gate rows over its up rows, s_gu [E, 2*ceil(I/128), ceil(H/128)];
    q_d [E, H, I], s_d [E, ceil(H/128), ceil(I/128)].
    Returns float64 [len(tokens), H]: the combine before its BF16 rounding
    (round with f64_to_bf16_bits to compare bits).
    """
    T = np.asarray(x_bits).shape[0]
    t_idx = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    row_of = np.asarray(route["row_of"], dtype=np.int64)[t_idx]          # [n, k]
    rows = np.unique(row_of.reshape(-1))                                   # sorted routed rows
    offsets = np.asarray(route["offsets"], dtype=np.int64)
    q_a, s_a = gather_act_quant(x_bits, np.asarray(route["row_token"])[rows])
    # each routed row keeps its expert: express the gathered rows as their own
    # offset table (rows are sorted, so experts are contiguous)
    experts = np.searchsorted(offsets, rows, side="right") - 1
    E = q_gu.shape[0]
    sub_off = np.zeros(E + 1, dtype=np.int64)
    sub_off[1:] = np.cumsum(np.bincount(experts, minlength=E))
    q_h, s_h = grouped_gate_up_silu_quant(q_a, s_a, q_gu, s_gu, sub_off)
    y = f64_to_bf16_bits(grouped_linear_w8a8(q_h, s_h, q_d, s_d, sub_off))
    local = np.searchsorted(rows, row_of)                                  # [n, k] into y
    return combine_f64(y, local, route["weights"][t_idx])
