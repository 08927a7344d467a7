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
