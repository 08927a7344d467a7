"""Helpers shared by the GPU parity tests: input construction through the
oracle's own quantizers, device transfer, and the acceptance checks.

Acceptance for GEMM outputs (floating point):
    |gpu - oracle| <= 4e-3 * |oracle| + 1e-3 * rms(oracle)   elementwise.
BF16 output rounding alone is <= 2^-8 ~ 3.9e-3 relative (an 8-bit
significand), and FP32 accumulation over K <= 17408 adds < 1e-5 relative;
the rms term covers outputs that cancel to near zero.
Quantized bytes and scales must be bit-exact.
"""

from __future__ import annotations

import functools

import numpy as np
import torch

from block_scaled_fp8_token_gb300 import synth
from oracle import formats as F
from oracle import quant as Q

REL_TOL = 4e-3
RMS_TOL = 1e-3


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_dev_bf16(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def to_dev_u8(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def scale_to_dev(s: np.ndarray, dev) -> torch.Tensor:
    """BF16 scale bits (uint16) -> bfloat16 tensor; float32 stays float32."""
    if s.dtype == np.uint16:
        return to_dev_bf16(s, dev)
    return torch.from_numpy(np.ascontiguousarray(s)).to(dev)


def gpu_bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(gpu - ref)
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; rms={rms:.4g}; first "
            + ", ".join(f"{tuple(i)} gpu={gpu[tuple(i)]:.6g} ref={ref[tuple(i)]:.6g}" for i in idx))


def cos_rrms(a: np.ndarray, b: np.ndarray) -> tuple[float, float]:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    cos = float(a @ b / np.sqrt((a @ a) * (b @ b)))
    rrms = float(np.sqrt(np.mean((a - b) ** 2) / np.mean(b ** 2)))
    return cos, rrms


def quantize_members(w: np.ndarray, members=None, scale_dtype="bf16"):
    """Oracle AOT quantization with member-local grids stacked in order."""
    rows = members or [w.shape[0]]
    qs, ss, r0 = [], [], 0
    for n in rows:
        q, s = Q.quantize_weight_blocks(w[r0:r0 + n], scale_dtype)
        qs.append(q)
        ss.append(s)
        r0 += n
    return np.concatenate(qs), np.concatenate(ss)


@functools.lru_cache(maxsize=None)
def dense_ffn_weights(seed: int = 0):
    """Oracle-quantized dense-FFN weights [34816, 5120] and [5120, 17408] plus
    the 949-token activations (cached for the session)."""
    d = synth.dense_ffn(seed)
    qgu, sgu = Q.quantize_weight_blocks(d["w_gate_up"].numpy())
    qd, sd = Q.quantize_weight_blocks(d["w_down"].numpy())
    return qgu, sgu, qd, sd, bits16(d["x"])


def sample_indices(n: int, k: int, seed: int) -> np.ndarray:
    """k sorted indices in [0, n) that always include both ends and both
    sides of every 128 boundary near the ends."""
    rng = np.random.default_rng(seed)
    must = {0, n - 1, min(n - 1, 127), min(n - 1, 128), max(0, n - 128), max(0, n - 129)}
    rest = rng.choice(n, size=min(n, k), replace=False)
    return np.array(sorted(must | set(rest.tolist())), dtype=np.int64)


def dec_e4m3(q: np.ndarray) -> np.ndarray:
    return F.e4m3_decode_lut()[q]
