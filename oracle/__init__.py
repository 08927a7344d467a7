"""CPU oracle for the block-scaled FP8 linear projection.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously correct
restatement of what the block-FP8 projection computes, written from the pages'
text and the E4M3 / BF16 format definitions. It is double precision (numpy
float64) wherever the pages leave the precision open.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it. The CUDA library
never links, imports or calls it, and it imports nothing from the CUDA
package: the two share no code.

Modules:
  formats   E4M3 decode table and RNE encoder; BF16 <-> F32 conversions.
  quant     per-token 1x128 activation quantizer, ahead-of-time weight block
            quantizer, reference dequantization, SiLU(gate)*up glue.
  linear    W8A8 and W8A16 block-scaled projections, member-local scale
            origins, grouped (per-expert) projection, MoE top-k routing.
  validate  the weight/scale-grid refusal table.

Parity pins: every function is checked in ``tests/test_oracle_*.py`` against
something other than itself: values the pages print, closed forms, torch's
independent float8/bfloat16 casts, exact rational brute force, and invariants.
The pages print no value for SiLU or for the MoE router. ``quant.silu_mul_bf16``
is therefore pinned by closed forms of SiLU, and ``linear.route_topk`` by a
brute-force sort on a tiny table.
"""

from .formats import (
    E4M3_MAX,
    bf16_bits_to_f32,
    e4m3_decode_lut,
    e4m3_encode_rne_sat,
    e4m3_value,
    f32_to_bf16_bits,
    f64_to_bf16_bits,
)
from .quant import (
    act_quant_group,
    dequantize_block_scaled,
    quantize_weight_blocks,
    silu_mul_bf16,
    silu_mul_act_quant,
)
from .linear import (
    grouped_linear_w8a8,
    linear_w8a16,
    linear_w8a8,
    route_topk,
    scale_grid_shape,
    scale_rows,
)
from .validate import validate_grid

__all__ = [
    "E4M3_MAX", "bf16_bits_to_f32", "e4m3_decode_lut", "e4m3_encode_rne_sat",
    "e4m3_value", "f32_to_bf16_bits", "f64_to_bf16_bits",
    "act_quant_group", "dequantize_block_scaled", "quantize_weight_blocks",
    "silu_mul_bf16", "silu_mul_act_quant",
    "grouped_linear_w8a8", "linear_w8a16", "linear_w8a8", "route_topk",
    "scale_grid_shape", "scale_rows", "validate_grid",
]
