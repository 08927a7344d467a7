"""The C ABI: libbfp8.so loads on a CPU-only machine, exports every function
include/bfp8.h declares, names every status code the header enumerates, and
rejects bad arguments before touching the GPU."""

import ctypes
import re
from pathlib import Path

import pytest

HEADER = Path(__file__).resolve().parent.parent / "include" / "bfp8.h"


def _declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(bfp8_[a-z0-9_]+)\s*\(", text)))


def _status_enum():
    text = HEADER.read_text()
    body = re.search(r"enum bfp8_status \{(.*?)\};", text, re.S).group(1)
    out = {}
    for name, val in re.findall(r"BFP8_(?:ERR_)?([A-Z0-9_]+)\s*=\s*(\d+)", body):
        out[int(val)] = name
    return out


def test_header_declares_the_entry_points():
    fns = _declared_functions()
    for want in ["bfp8_validate_grid", "bfp8_act_quant_group", "bfp8_linear_w8a8",
                 "bfp8_linear_w8a16", "bfp8_gemv_decode", "bfp8_grouped_linear"]:
        assert want in fns


def test_library_exports_every_declared_symbol(bfp8):
    lib = ctypes.CDLL(str(bfp8.library_path()))
    missing = [f for f in _declared_functions() if not hasattr(lib, f)]
    assert not missing, missing


def test_status_strings_match_header(bfp8):
    enum = _status_enum()
    assert len(enum) == 16
    for val, name in enum.items():
        assert bfp8.bfp8_status_string(val) == name
        assert bfp8.STATUS_NAMES[val] == name
    assert bfp8.bfp8_status_string(999) == "UNKNOWN"


def test_argument_errors_without_gpu(bfp8):
    lib = bfp8._lib
    inval = 1
    # negative sizes / null pointers are refused before any CUDA call
    assert lib.bfp8_act_quant_group(None, -1, 4, 4, None, 4, None, 1, 1, None) == inval
    assert lib.bfp8_act_quant_group(None, 0, 4, 4, None, 4, None, 1, 1, None) == 0   # empty: no-op
    assert lib.bfp8_linear_w8a8(None, None, 1, 1, None, None, 3, 4, 8, 16, None, 8, None, None, 0, None) == inval
    assert lib.bfp8_linear_w8a8(None, None, 1, 1, None, None, 3, 0, 8, 16, None, 8, None, None, 0, None) == 0
    assert lib.bfp8_gemv_decode(None, 16, None, None, 3, 17, 8, 16, None, 8, None, None, 0, None) == inval
    assert lib.bfp8_grouped_linear(None, None, 1, 1, None, None, 3, None, 0, 8, 8, 16, None, 8, None, 0, None) == inval
    # a weight-scale dtype other than BF16/F32 is refused by name
    p = ctypes.c_void_p(16)
    assert lib.bfp8_linear_w8a8(p, p, 1, 1, p, p, 4, 4, 8, 16, p, 8, None, None, 0, None) == 8
    # members that do not partition N
    rows = (ctypes.c_int64 * 2)(3, 3)
    mem = bfp8.bfp8_members(2, rows)
    assert lib.bfp8_linear_w8a8(p, p, 1, 1, p, p, 3, 4, 8, 16, p, 8, ctypes.byref(mem), None, 0, None) == 11


def test_binding_refuses_host_tensors(bfp8):
    """A host tensor never reaches the library: the kernels would read its
    address as device memory."""
    import torch

    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    q = torch.empty(4, 128, dtype=torch.uint8)
    s = torch.empty(4, 1, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bfp8.bfp8_act_quant_group(x, q, s)
    w = torch.zeros(128, 128, dtype=torch.uint8)
    sw = torch.ones(1, 1, dtype=torch.bfloat16)
    y = torch.empty(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bfp8.bfp8_linear_w8a8(q, s, w, sw, y)


def test_every_entry_point_refuses_bad_arguments_without_gpu(bfp8):
    """Each refusal below is decided from the arguments alone, before any CUDA
    call (placeholder pointers are never dereferenced)."""
    lib, p = bfp8._lib, ctypes.c_void_p(256)
    INVAL, SCALE_DTYPE, UNSUPPORTED = 1, 8, 13
    cases = [
        # act quant: negative size, row pitch below K, zero scale stride over several rows
        (lib.bfp8_act_quant_group(p, 4, -1, 4, p, 4, p, 1, 1, None), INVAL),
        (lib.bfp8_act_quant_group(p, 4, 256, 255, p, 256, p, 2, 1, None), INVAL),
        (lib.bfp8_act_quant_group(p, 4, 256, 256, p, 255, p, 2, 1, None), INVAL),
        (lib.bfp8_act_quant_group(p, 4, 256, 256, p, 256, p, 0, 1, None), INVAL),
        # SiLU*up quant: the gate/up pitch must hold 2I values
        (lib.bfp8_silu_mul_act_quant(p, 4, 128, 255, p, 128, p, 1, 4, None), INVAL),
        # weight quantization
        (lib.bfp8_quantize_weight_block(p, -1, 128, 128, p, 128, p, 3, None), INVAL),
        (lib.bfp8_quantize_weight_block(p, 128, 128, 127, p, 128, p, 3, None), INVAL),
        (lib.bfp8_quantize_weight_block(p, 128, 128, 128, p, 128, p, 4, None), SCALE_DTYPE),
        # W8A16: activation pitch below K
        (lib.bfp8_linear_w8a16(p, 127, p, p, 3, 4, 128, 128, p, 128, None, None), INVAL),
        # decode GEMV, W8A8 arm: more than 16 tokens
        (lib.bfp8_gemv_decode_w8a8(p, p, 1, 1, p, p, 3, 17, 128, 128, p, 128, None, p, 1 << 20,
                                   None), INVAL),
        # grouped: more experts than the schedule holds; fused: h pitch below I
        (lib.bfp8_grouped_linear(p, p, 1, 1, p, p, 3, p, 1025, 8, 128, 128, p, 128, None, 0, None),
         INVAL),
        (lib.bfp8_linear_w8a8_silu_quant(p, p, 1, 1, p, p, 3, 4, 128, 128, p, 127, p, 1, 1, None,
                                         0, None), INVAL),
        (lib.bfp8_grouped_linear_silu_quant(p, p, 1, 1, p, p, 3, p, 0, 8, 128, 128, p, 128, p, 1,
                                            1, None, 0, None), INVAL),
        # decode step: unknown arithmetic, 17 tokens, sizes not multiples of 16
        (lib.bfp8_decode_ffn(7, p, 256, p, p, p, p, 3, 4, 256, 256, p, 256, p, 1 << 24, None),
         INVAL),
        (lib.bfp8_decode_ffn(0, p, 256, p, p, p, p, 3, 17, 256, 256, p, 256, p, 1 << 24, None),
         INVAL),
        (lib.bfp8_decode_ffn(0, p, 264, p, p, p, p, 3, 4, 264, 256, p, 264, p, 1 << 24, None),
         UNSUPPORTED),
        # MoE glue: a negative routed-row count; top-k of zero; output pitch below H
        (lib.bfp8_moe_gather_act_quant(p, 8, 256, 256, p, -1, p, 256, p, 2, 1, None), INVAL),
        (lib.bfp8_moe_combine(p, 16, 256, 256, p, p, 8, 0, p, 256, None), INVAL),
        (lib.bfp8_moe_combine(p, 16, 256, 256, p, p, 8, 2, p, 255, None), INVAL),
        # wait self-test: the limit must lie in (0, 2 s]
        (lib.bfp8_selftest_wait_timeout(0, None), INVAL),
        (lib.bfp8_selftest_wait_timeout(2_000_000_001, None), INVAL),
    ]
    for i, (got, want) in enumerate(cases):
        assert got == want, (i, got, want)
