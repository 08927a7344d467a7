"""Grid validation: the oracle's refusal table and the C library's
bfp8_validate_grid, checked fixture by fixture against the refusal each
passage calls for (tests/golden/refusals.json). Host only; no GPU."""

import json

import pytest

from conftest import GOLDEN
from oracle.validate import validate_grid

CASES = json.loads((GOLDEN / "refusals.json").read_text())["cases"]
DT = {"E4M3": 1, "E5M2": 2, "BF16": 3, "F16": 4, "F32": 5}


def _oracle_desc(d):
    return {
        "weight_dtype": d["weight_dtype"],
        "weight_shape": tuple(d["weight_shape"]),
        "scale_dtype": d.get("scale_dtype"),
        "scale_shape": tuple(d["scale_shape"]) if "scale_shape" in d else None,
        "has_row_scale": d.get("has_row_scale", False),
        "declared_quant_fp8": d.get("declared_quant_fp8", True),
        "declared_block": tuple(d.get("declared_block", (128, 128))),
        "member_rows": d.get("member_rows"),
        "tensor_scale_dtype": d.get("tensor_scale_dtype"),
    }


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_refusals(case):
    assert validate_grid(_oracle_desc(case["desc"])) == case["expect"]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_library_refusals(case, bfp8):
    d = case["desc"]
    desc, _keep = bfp8.make_weight_desc(
        DT[d["weight_dtype"]], d["weight_shape"],
        scale_dtype=DT.get(d.get("scale_dtype"), 0) if d.get("scale_dtype") else 0,
        scale_shape=d.get("scale_shape"), has_row_scale=d.get("has_row_scale", False),
        declared_quant_fp8=d.get("declared_quant_fp8", True),
        declared_block=d.get("declared_block", (128, 128)), member_rows=d.get("member_rows"),
        tensor_scale_dtype=DT.get(d.get("tensor_scale_dtype"), 0))
    rc, msg = bfp8.bfp8_validate_grid(desc)
    assert bfp8.bfp8_status_string(rc) == case["expect"], msg
    assert msg


def test_library_null_descriptor(bfp8):
    import ctypes
    rc = bfp8._lib.bfp8_validate_grid(None, None, 0)
    assert bfp8.bfp8_status_string(rc) == "INVALID_ARG"
