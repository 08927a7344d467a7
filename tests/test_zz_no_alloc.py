"""bfp8_gemv_decode_noalloc: the decode GEMV for callers that cannot allocate
device memory (code running under someone else's allocator, or code that must
keep device memory fixed while serving). Its scratch is a fixed array inside
the library instead of a caller-provided workspace.

Checked through the C ABI against bfp8_gemv_decode on the same inputs, on two
calls in a row: both run the same kernels on the same scratch layout, so the
outputs must be identical bytes. The second call reuses the shared array,
which still holds what the first call left there. A problem at the largest K
the array holds runs; one block of K more is refused. The file name makes
pytest collect it last.
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
        assert np.array_equal(bits16(y), bits16(y_ref)), f"no-alloc call {call + 1}"
        assert_close(gpu_bf16_to_f64(y), ref, f"no-alloc call {call + 1}")


def test_noalloc_at_the_largest_k_its_scratch_holds(bfp8, cuda_device):
    """K = the largest multiple of 128 whose scratch fits the fixed array
    (token tiles and factors grow with K): it runs and matches
    bfp8_gemv_decode byte for byte; K + 128 is refused before any GPU work."""
    dev = cuda_device
    M, N = 2, 256
    cap = 4 * 1024 * 1024
    K = 128
    while bfp8.bfp8_gemv_decode_workspace(M, N, K + 128) <= cap:
        K += 128
    assert K > 40000, K
    g = synth.generator(K)
    q, s = quantize_members(synth.weight_f32(g, N, K).numpy())
    x = to_dev_bf16(bits16(synth.activations_bf16(g, M, K)), dev)
    w, sw = to_dev_u8(q, dev), scale_to_dev(s, dev)
    y_ref = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(bfp8.bfp8_gemv_decode_workspace(M, N, K), dtype=torch.uint8, device=dev)
    bfp8.bfp8_gemv_decode(x, w, sw, y_ref, ws)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    bfp8.bfp8_gemv_decode_noalloc(x, w, sw, y)
    torch.cuda.synchronize()
    assert bfp8.bfp8_device_status() == 0
    assert np.array_equal(bits16(y), bits16(y_ref))
    K2 = K + 128
    p = ctypes.c_void_p(256)
    rc = bfp8._lib.bfp8_gemv_decode_noalloc(p, K2, p, p, bfp8.BFP8_DT_BF16, M, N, K2, p, N, None,
                                            None)
    assert bfp8.bfp8_status_string(rc) == "UNSUPPORTED"


def test_noalloc_rejects_problems_beyond_its_scratch(bfp8, cuda_device):
    # 2^31 - 1 weight rows need far more than the fixed scratch: refused before any
    # GPU work, so the placeholder pointers are never dereferenced.
    N = 2 ** 31 - 1
    p = ctypes.c_void_p(256)
    rc = bfp8._lib.bfp8_gemv_decode_noalloc(p, 4096, p, p, bfp8.BFP8_DT_BF16, 16, N, 4096, p, N,
                                            None, None)
    assert bfp8.bfp8_status_string(rc) == "UNSUPPORTED"
    assert bfp8.bfp8_gemv_decode_workspace(16, N, 4096) > 4 * 1024 * 1024
