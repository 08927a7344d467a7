"""GPU: a bounded device wait that runs out.

Every barrier wait in the library's kernels gives up after a time limit, sets
the CTA's abort flag and records BFP8_ERR_TIMEOUT in the device error word
instead of hanging the GPU. bfp8_selftest_wait_timeout launches one CTA whose
barrier never gets its second arrival, waited on in both forms the kernels
use (spinning and suspending) with a short limit. The timeout must come back
through bfp8_device_status(), once, and the context must stay usable: a
quantization launched afterwards is still bit-exact against the oracle.
"""

import time

import numpy as np
import pytest
import torch

from block_scaled_fp8_token_gb300 import synth
from gpu_util import bits16, to_dev_bf16
from oracle import quant as Q

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, 15


def test_bounded_wait_runs_out_and_the_gpu_still_answers(bfp8, cuda_device):
    assert bfp8.bfp8_device_status() == OK
    limit_ns = 5_000_000   # 5 ms
    t0 = time.perf_counter()
    bfp8.bfp8_selftest_wait_timeout(limit_ns)
    status = bfp8.bfp8_device_status()
    elapsed = time.perf_counter() - t0
    assert status == TIMEOUT
    # the short limit applied, not the kernels' 2 s one
    assert elapsed < 1.0
    # read and cleared
    assert bfp8.bfp8_device_status() == OK

    xb = bits16(synth.activations_bf16(synth.generator(11), 33, 640, outlier="entries"))
    x = to_dev_bf16(xb, cuda_device)
    q = torch.zeros(33, 640, dtype=torch.uint8, device=cuda_device)
    s = torch.zeros(33, 5, dtype=torch.float32, device=cuda_device)
    bfp8.bfp8_act_quant_group(x, q, s)
    assert bfp8.bfp8_device_status() == OK
    qr, sr = Q.act_quant_group(xb)
    assert np.array_equal(q.cpu().numpy(), qr)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))
