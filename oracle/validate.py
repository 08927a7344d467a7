"""Refusal table for a block-FP8 weight, decided from metadata alone.

Test infrastructure (CPU oracle); see the package docstring for who may use it.

The pages list what must be refused before any weight byte is uploaded:
* E5M2 encodings, ambiguous row/block scales, malformed grids and
  incompatible checkpoint declarations [Qwen checkpoints with block FP8
  weights, third paragraph];
* a row-wise tree (rank-1 per-row ``weight_scale``), a transposed or
  mis-blocked grid, an FP8 weight with no scale, a rank-1 scale, and a config
  that disagrees with the bytes [th#1803 decoder PR, "Why the refusals matter
  more than the load"];
* dense trees [th#1803 decoder PR, "Proof", item 4].
A per-tensor scaled weight (one f32 multiplier in a "weight_scale" leaf) is
the other FP8 checkpoint shape, read as a block case whose single block
covers the tensor [FP8 Native Serving, "The two FP8 checkpoint shapes"].
The checkpoint must declare quant_method fp8 and weight_block_size [128,128],
and the grid is ceil-divided with member-local origins [Qwen checkpoints with
block FP8 weights, first and third paragraphs]. Verification uses headers
only [th#1803 decoder PR, "What lands": inspect from safetensors headers].

The first failing rule below decides the answer, which is a refusal name.
The C library has its own copy of this table; the two share no code, and a
test checks that they agree fixture by fixture.

Readings where the pages are silent:
* "transposed" is only detectable when ceil(N/128) != ceil(K/128). A square
  grid with swapped meaning looks identical in the header and is accepted.
* "ambiguous" covers both leaves present, and also a rank-2 scale whose
  row count equals N (a per-row grid) when N != ceil(N/128).
* a grouped tensor whose grid was built on the stacked rows (ceil(sum N_i /
  128) rows) instead of member-local origins is refused as GROUP.
* per-tensor: its one-element scale next to a block grid or a per-row scale is
  ambiguous; a declared weight_block_size disagrees with it (BLOCK_SIZE); its
  dtype must be BF16 or F32 like a grid's; members must still partition N,
  and the one multiplier covers every member.
"""

from __future__ import annotations

FP8_DTYPES = ("E4M3", "E5M2")
SCALE_DTYPES_OK = ("BF16", "F32")


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def validate_grid(desc: dict) -> str:
    """Return "OK" or the refusal name for a weight descriptor.

    desc keys: weight_dtype ("E4M3", "E5M2", "BF16", "F16", "F32"),
    weight_shape (tuple), scale_dtype (None or a dtype name),
    scale_shape (tuple or None), has_row_scale (bool),
    declared_quant_fp8 (bool), declared_block (pair), member_rows (list or None),
    tensor_scale_dtype (None or a dtype name: a one-element weight_scale).
    """
    shape = tuple(desc.get("weight_shape") or ())
    if len(shape) != 2 or shape[0] <= 0 or shape[1] <= 0:
        return "INVALID_ARG"
    N, K = int(shape[0]), int(shape[1])
    wdt = desc.get("weight_dtype")
    if wdt == "E5M2":
        return "E5M2"
    if wdt != "E4M3":
        return "NOT_FP8"
    if not desc.get("declared_quant_fp8", False):
        return "QUANT_METHOD"
    sdt = desc.get("scale_dtype")
    has_block = sdt is not None
    tdt = desc.get("tensor_scale_dtype")
    if tdt is not None:
        if has_block or desc.get("has_row_scale", False):
            return "AMBIGUOUS_SCALE"
        if tuple(desc.get("declared_block") or (0, 0)) != (0, 0):
            return "BLOCK_SIZE"
        if tdt not in SCALE_DTYPES_OK:
            return "SCALE_DTYPE"
        members = desc.get("member_rows")
        if members is not None:
            members = [int(v) for v in members]
            if len(members) == 0 or any(v <= 0 for v in members) or sum(members) != N:
                return "GROUP"
        return "OK"
    if tuple(desc.get("declared_block") or ()) != (128, 128):
        return "BLOCK_SIZE"
    if desc.get("has_row_scale", False):
        return "AMBIGUOUS_SCALE" if has_block else "ROW_SCALE"
    if not has_block:
        return "NO_SCALE"
    sshape = tuple(desc.get("scale_shape") or ())
    if len(sshape) == 1:
        return "ROW_SCALE"
    if sdt not in SCALE_DTYPES_OK:
        return "SCALE_DTYPE"
    if len(sshape) != 2:
        return "GRID_SHAPE"
    members = desc.get("member_rows")
    if members is not None:
        members = [int(v) for v in members]
        if len(members) == 0 or any(v <= 0 for v in members) or sum(members) != N:
            return "GROUP"
    Kb = _ceil_div(K, 128)
    Nb = sum(_ceil_div(v, 128) for v in members) if members else _ceil_div(N, 128)
    if sshape == (Nb, Kb):
        return "OK"
    if sshape == (Kb, Nb) and Nb != Kb:
        return "GRID_TRANSPOSED"
    if sshape[0] == N and N != Nb:
        return "AMBIGUOUS_SCALE"
    if members and sshape == (_ceil_div(N, 128), Kb):
        return "GROUP"
    return "GRID_SHAPE"
