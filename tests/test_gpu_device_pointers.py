"""Every entry point refuses memory that is not on the current GPU.

Kernels and TMA descriptors read their pointers as device memory of the
current device, so the C ABI checks each pointer (cudaPointerGetAttributes)
before it encodes a descriptor or launches anything: pinned host memory,
pageable host memory and stray addresses return INVALID_ARG, whoever the
caller is (the Python binding refuses host tensors earlier, so these calls
go through ctypes directly). A refused call leaves no error behind: a valid
call right after it succeeds.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

INVALID = 1


def _calls(lib, d, h):
    """(name, status) for each entry point with `h` in one pointer slot and
    device memory (offsets into d, 256-byte aligned) everywhere else."""
    a = lambda i: ctypes.c_void_p(d + i * (1 << 20))   # noqa: E731
    H = ctypes.c_void_p(h)
    bf16, f32 = 3, 5
    two = (ctypes.c_int64 * 2)(128, 128)
    return [
        ("act_quant", lib.bfp8_act_quant_group(H, 4, 256, 256, a(1), 256, a(2), 2, 1, None)),
        ("act_quant out", lib.bfp8_act_quant_group(a(0), 4, 256, 256, a(1), 256, H, 2, 1, None)),
        ("silu_mul_act_quant", lib.bfp8_silu_mul_act_quant(a(0), 4, 128, 256, H, 128, a(2), 1, 1,
                                                          None)),
        ("silu_mul", lib.bfp8_silu_mul(a(0), 4, 128, 256, H, 128, None)),
        ("weight quant", lib.bfp8_quantize_weight_block(H, 128, 128, 128, a(1), 128, a(2), bf16,
                                                        None)),
        ("w8a8 weight", lib.bfp8_linear_w8a8(a(0), a(1), 2, 1, H, a(3), bf16, 4, 256, 256, a(4),
                                             256, None, None, 0, None)),
        ("w8a8 workspace", lib.bfp8_linear_w8a8(a(0), a(1), 2, 1, a(2), a(3), bf16, 4, 256, 256,
                                                a(4), 256, None, H, 1 << 20, None)),
        ("w8a16", lib.bfp8_linear_w8a16(H, 256, a(2), a(3), bf16, 4, 256, 256, a(4), 256, None,
                                        None)),
        ("gemv workspace", lib.bfp8_gemv_decode(a(0), 256, a(2), a(3), bf16, 4, 256, 256, a(4), 256,
                                                None, H, 1 << 20, None)),
        ("gemv w8a8 scales", lib.bfp8_gemv_decode_w8a8(a(0), H, 2, 1, a(2), a(3), bf16, 4, 256,
                                                       256, a(4), 256, None, a(5), 4 << 20, None)),
        ("gemv noalloc", lib.bfp8_gemv_decode_noalloc(H, 256, a(2), a(3), bf16, 4, 256, 256, a(4),
                                                      256, None, None)),
        ("grouped offsets", lib.bfp8_grouped_linear(a(0), a(1), 2, 1, a(2), a(3), bf16, H, 2, 8,
                                                    256, 256, a(4), 256, None, 0, None)),
        ("fused gate/up", lib.bfp8_linear_w8a8_silu_quant(a(0), a(1), 2, 1, a(2), a(3), bf16, 4, 128,
                                                          256, H, 128, a(5), 1, 1, None, 0, None)),
        ("grouped fused", lib.bfp8_grouped_linear_silu_quant(a(0), a(1), 2, 1, a(2), a(3), bf16,
                                                             a(6), 2, 8, 128, 256, a(4), 128, H,
                                                             1, 1, None, 0, None)),
        ("decode step", lib.bfp8_decode_ffn(0, a(0), 256, a(1), a(2), a(3), a(4), bf16, 2, 256, 128,
                                            H, 256, a(8), 8 << 20, None)),
        ("moe gather", lib.bfp8_moe_gather_act_quant(a(0), 8, 256, 256, H, 4, a(2), 256, a(3), 2,
                                                     1, None)),
        ("moe combine", lib.bfp8_moe_combine(a(0), 16, 256, 256, a(1), a(2), 4, 2, H, 256, None)),
        ("members", lib.bfp8_linear_w8a8(H, a(1), 2, 1, a(2), a(3), f32, 4, 256, 256, a(4), 256,
                                         ctypes.byref(lib_members(two)), None, 0, None)),
    ]


def lib_members(rows):
    from block_scaled_fp8_token_gb300 import bfp8
    return bfp8.bfp8_members(2, rows)


def test_entry_points_refuse_memory_not_on_the_gpu(bfp8, cuda_device):
    lib = bfp8._lib
    d = torch.zeros(16 << 20, dtype=torch.uint8, device=cuda_device)
    pinned = torch.zeros(1 << 20, dtype=torch.uint8, pin_memory=True)
    pageable = torch.zeros(1 << 20, dtype=torch.uint8)
    arr = np.zeros(1 << 16, np.uint8)
    for what, h in [("pinned host", pinned.data_ptr()), ("pageable host", pageable.data_ptr()),
                    ("numpy host", arr.ctypes.data), ("stray address", 1 << 20)]:
        for name, rc in _calls(lib, d.data_ptr(), h):
            assert rc == INVALID, (what, name, bfp8.bfp8_status_string(rc))
    # nothing was launched and no error is left behind
    x = torch.randn(4, 256, device=cuda_device).to(torch.bfloat16)
    q = torch.empty(4, 256, dtype=torch.uint8, device=cuda_device)
    s = torch.empty(4, 2, dtype=torch.float32, device=cuda_device)
    bfp8.bfp8_act_quant_group(x, q, s)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    assert bool((s > 0).all())
