"""Seeded synthetic inputs for the block-FP8 projection workloads.

This module only draws random numbers. It holds none of the projection's
arithmetic: no quantization, scaling, rounding to FP8 or matrix products.
Tests feed its draws to the CPU oracle, and ``bench.py`` feeds them to the CUDA
library's own conversion entry point. Everything is drawn on the CPU from
``torch.Generator().manual_seed(seed)``, so the same seed gives the same bytes
on any machine.

The pages measure on real checkpoints and prompts (Qwen3.6-27B-FP8 with a
949-token prompt, Qwen3.6-35B-A3B). Those are not available, so these draws
stand in for them with the same shapes:
  * weights: float32 N(0, 0.02^2) before ahead-of-time block quantization;
  * activations: BF16 N(0, 1) with outliers. The outliers are either scattered
    entries (Bernoulli(p) mask, times a factor) or whole channels (a seeded
    random choice of round(frac * K) columns, times a factor, on every token);
  * MoE router logits: float32 N(0, 1) [tokens, experts].
Draw order within one workload: weights, activations, outlier mask or
channels, router logits.
"""

from __future__ import annotations

import torch


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def weight_f32(g: torch.Generator, N: int, K: int, std: float = 0.02) -> torch.Tensor:
    """float32 [N, K] drawn from N(0, std^2)."""
    return torch.randn(N, K, generator=g, dtype=torch.float32) * std


def weight_stack_f32(g: torch.Generator, G: int, N: int, K: int, std: float = 0.02) -> torch.Tensor:
    """float32 [G, N, K] drawn from N(0, std^2) (one matrix per expert)."""
    return torch.randn(G, N, K, generator=g, dtype=torch.float32) * std


def activations_bf16(g: torch.Generator, M: int, K: int, *, outlier: str | None = None,
                     frac: float = 0.0, factor: float = 1.0) -> torch.Tensor:
    """BF16 [M, K] from N(0, 1) with optional outliers.

    outlier == "entries": each entry independently with probability ``frac``
    is multiplied by ``factor``. outlier == "channels": round(frac * K)
    columns, picked by a seeded permutation, are multiplied by ``factor``
    on every token.
    """
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    if outlier == "entries":
        mask = torch.rand(M, K, generator=g) < frac
        x = torch.where(mask, x * factor, x)
    elif outlier == "channels":
        n_ch = int(round(frac * K))
        ch = torch.randperm(K, generator=g)[:n_ch]
        x[:, ch] *= factor
    elif outlier is not None:
        raise ValueError(f"unknown outlier mode {outlier!r}")
    return x.to(torch.bfloat16)


def router_logits(g: torch.Generator, T: int, E: int) -> torch.Tensor:
    """float32 [T, E] drawn from N(0, 1)."""
    return torch.randn(T, E, generator=g, dtype=torch.float32)


# The five workloads, by their shapes. Sizes only; no arithmetic.
SINGLE_TAILS = dict(M=8, N=192, K=320, outlier="entries", frac=0.01, factor=20.0)
DECODE = dict(M=(1, 4, 16), gate_up=(34816, 5120), down=(5120, 17408))
DENSE_FFN_PREFILL = dict(M=949, hidden=5120, inter=17408, outlier="channels", frac=0.005, factor=30.0)
ATTENTION_PROJ = dict(M=4096, hidden=5120, q=8192, k=1024, v=1024, o_in=8192)
MOE_PREFILL = dict(tokens=8192, hidden=2048, experts=128, top_k=8, inter=768)


def single_tails(seed: int = 0) -> dict:
    """Weight [192, 320] and BF16 activations [8, 320] with 1% x20 entry outliers."""
    c = SINGLE_TAILS
    g = generator(seed)
    w = weight_f32(g, c["N"], c["K"])
    x = activations_bf16(g, c["M"], c["K"], outlier=c["outlier"], frac=c["frac"], factor=c["factor"])
    return {"w": w, "x": x}


def dense_ffn(seed: int = 0, M: int | None = None) -> dict:
    """Gate/up [2*inter, hidden], down [hidden, inter], activations [M, hidden]."""
    c = DENSE_FFN_PREFILL
    g = generator(seed)
    H, I = c["hidden"], c["inter"]
    w_gu = weight_f32(g, 2 * I, H)
    w_d = weight_f32(g, H, I)
    M = c["M"] if M is None else M
    x = activations_bf16(g, M, H, outlier=c["outlier"], frac=c["frac"], factor=c["factor"])
    return {"w_gate_up": w_gu, "w_down": w_d, "x": x}


# outlier recipes of the activation workloads: 1% of entries x20 (the single
# linear) and 0.5% of channels x30 (the dense-FFN prefill)
OUTLIERS = {"entries": dict(frac=0.01, factor=20.0), "channels": dict(frac=0.005, factor=30.0)}


def decode_tokens(seed: int, M: int, K: int, outlier: str | None = None) -> torch.Tensor:
    """BF16 [M, K] N(0, 1) decode tokens, optionally with one of the
    activation workloads' outlier patterns (OUTLIERS)."""
    if outlier is None:
        return activations_bf16(generator(seed), M, K)
    return activations_bf16(generator(seed), M, K, outlier=outlier, **OUTLIERS[outlier])


def attention(seed: int = 0, M: int | None = None) -> dict:
    """Q/K/V member weights, O weight and activations [M, hidden]."""
    c = ATTENTION_PROJ
    g = generator(seed)
    H = c["hidden"]
    w_q = weight_f32(g, c["q"], H)
    w_k = weight_f32(g, c["k"], H)
    w_v = weight_f32(g, c["v"], H)
    w_o = weight_f32(g, H, c["o_in"])
    M = c["M"] if M is None else M
    x = activations_bf16(g, M, H)
    return {"w_q": w_q, "w_k": w_k, "w_v": w_v, "w_o": w_o, "x": x}


def moe(seed: int = 0, tokens: int | None = None, experts: int | None = None) -> dict:
    """Per-expert gate/up [E, 2*inter, hidden], down [E, hidden, inter],
    tokens [T, hidden] and router logits [T, E]."""
    c = MOE_PREFILL
    g = generator(seed)
    E = c["experts"] if experts is None else experts
    H, I = c["hidden"], c["inter"]
    w_gu = weight_stack_f32(g, E, 2 * I, H)
    w_d = weight_stack_f32(g, E, H, I)
    T = c["tokens"] if tokens is None else tokens
    x = activations_bf16(g, T, H)
    logits = router_logits(g, T, E)
    return {"w_gate_up": w_gu, "w_down": w_d, "x": x, "logits": logits}
