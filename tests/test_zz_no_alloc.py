"""bfp8_gemv_decode_noalloc: the decode GEMV for callers that cannot allocate
device memory (code running under someone else's allocator, or code that must
keep device memory fixed while serving). Its scratch is a fixed array inside
the library instead of a caller-provided workspace.

Checked through the C ABI against bfp8_gemv_decode on the same inputs, within
the GEMM tolerance used everywhere in these tests, on two calls in a row. The
second call reuses the shared array, which still holds what the first call
left there. The file name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import assert_close, bits16, gpu_bf16_to_f64, quantize_members, scale_to_dev, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,members", [(16, 5120, 4096, None), (3, 1000, 2048, [500, 500])])
def test_noalloc_matches_gemv_two_calls(bfp8, cuda_device, M, N, K, members):
    dev = cuda_device
    g = synth.generator(M * 100 + N)
    q, s = quantize_members(synth.weight_f32(g, N, K).numpy(), members)
    x = to_dev_bf16(bits16(synth.activations_bf16(g, M, K)), dev)
    w = to_dev_u8(q, dev)
    sw = scale_to_dev(s, dev)

    y_ref = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(bfp8.bfp8_gemv_decode_workspace(M, N, K), dtype=torch.uint8, device=dev)
    bfp8.bfp8_gemv_decode(x, w, sw, y_ref, ws, member_rows=members)
    torch.cuda.synchronize()
    ref = gpu_bf16_to_f64(y_ref)

    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        bfp8.bfp8_gemv_decode_noalloc(x, w, sw, y, member_rows=members)
        torch.cuda.synchronize()
        assert bfp8.bfp8_device_status() == 0
        assert_close(gpu_bf16_to_f64(y), ref, f"no-alloc call {call + 1}")


def test_noalloc_rejects_problems_beyond_its_scratch(bfp8, cuda_device):
    # 2^31 - 1 weight rows need far more than the fixed scratch: refused before any
    # GPU work, so the placeholder pointers are never dereferenced.
    N = 2 ** 31 - 1
    p = ctypes.c_void_p(256)
    rc = bfp8._lib.bfp8_gemv_decode_noalloc(p, 4096, p, p, bfp8.BFP8_DT_BF16, 16, N, 4096, p, N,
                                            None, None)
    assert bfp8.bfp8_status_string(rc) == "UNSUPPORTED"
    assert bfp8.bfp8_gemv_decode_workspace(16, N, 4096) > 4 * 1024 * 1024
