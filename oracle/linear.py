"""Block-scaled FP8 projections, double precision.

Test infrastructure (CPU oracle); see the package docstring for who may use it.

All projections compute y[M, N] = x[M, K] . W^T with W [N, K] row-major
([out, in], [th#1803 decoder PR, "What lands"]) and one scale per 128x128
block of W.

* Scale grids are ceil-divided, so a partial tail block row or column still
  has its own scale. A grouped (fused) tensor keeps a block-row origin per
  member [Qwen checkpoints with block FP8 weights, third paragraph]. For
  output row n inside member i, which starts at row0_i:
      r(n) = base_i + (n - row0_i) // 128,   base_i = sum_{j<i} ceil(N_j / 128).
* W8A8 (per-token 1x128 activation scales times 128x128 weight scales, an
  FP32 epilogue per K-block [Module w8a8_prefill, arithmetic paragraph]):
      y[m,n] = sum_kb s_a[m,kb] * s_w[r(n),kb] * sum_{k in kb} e4m3(qa[m,k]) * e4m3(qw[n,k])
* W8A16 (BF16 activations, weights decoded exactly and block multipliers
  applied inside the reduction [Qwen checkpoints with block FP8 weights,
  second paragraph; FP8 Native Serving, "Native FP8 vs dequant-to-BF16"]):
      y[m,n] = sum_kb s_w[r(n),kb] * sum_{k in kb} bf16(x[m,k]) * e4m3(qw[n,k])
  Every product and sum is in float64. The per-K-block partial is a float64
  matrix product (a library primitive) over that block's columns, which is
  exactly the definition's inner sum.
* Grouped (MoE expert) projection: rows offsets[e] .. offsets[e+1]-1 of the
  expert-sorted activations use expert e's weight and scale grid.
* MoE routing for the synthetic expert workload: softmax over the router
  logits, top-k by probability (ties go to the lower expert id), top-k weights
  renormalised to sum to 1, then rows sorted by expert (token-major inside an
  expert) with an offsets table. The pages do not describe the router. This
  is the plainest reading of "top-8 routing from softmax", and it only feeds
  the expert-sorted layout the grouped projection consumes.
"""

from __future__ import annotations

import numpy as np

from .formats import bf16_bits_to_f32, e4m3_decode_lut

BLOCK = 128


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _members(N: int, members) -> list[int]:
    if members is None:
        return [int(N)]
    members = [int(v) for v in members]
    if sum(members) != N or any(v <= 0 for v in members):
        raise ValueError(f"member rows {members} do not partition N={N}")
    return members


def scale_grid_shape(N: int, K: int, members=None) -> tuple[int, int]:
    """[sum_i ceil(N_i/128), ceil(K/128)]: the stacked member-local scale grid."""
    return (sum(_ceil_div(v, BLOCK) for v in _members(N, members)), _ceil_div(K, BLOCK))


def scale_rows(N: int, members=None) -> np.ndarray:
    """r(n) for every output row n: the scale-grid row that multiplies it."""
    r = np.empty(int(N), dtype=np.int64)
    row0 = 0
    base = 0
    for n_i in _members(N, members):
        r[row0:row0 + n_i] = base + np.arange(n_i) // BLOCK
        row0 += n_i
        base += _ceil_div(n_i, BLOCK)
    return r


def _scales_f64(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s)
    if s.dtype == np.uint16:          # BF16 bit patterns: widen exactly
        return bf16_bits_to_f32(s).astype(np.float64)
    return s.astype(np.float32).astype(np.float64)


def _sel(n: int, idx):
    return np.arange(n) if idx is None else np.asarray(idx, dtype=np.int64)


def linear_w8a8(q_a, s_a, q_w, s_w, members=None, rows=None, cols=None) -> np.ndarray:
    """W8A8 block-scaled projection in float64.

    q_a: uint8 [M, K] E4M3; s_a: float32 [M, ceil(K/128)];
    q_w: uint8 [N, K] E4M3; s_w: scale grid (BF16 bits or float32);
    rows / cols: optional output row / column subsets (default all).
    Returns float64 [len(rows), len(cols)].
    """
    q_a = np.asarray(q_a, dtype=np.uint8)
    q_w = np.asarray(q_w, dtype=np.uint8)
    M, K = q_a.shape
    N = q_w.shape[0]
    lut = e4m3_decode_lut()
    ri, ci = _sel(M, rows), _sel(N, cols)
    A = lut[q_a[ri]]
    W = lut[q_w[ci]]
    sa = np.asarray(s_a, dtype=np.float32).astype(np.float64)[ri]
    sw = _scales_f64(s_w)[scale_rows(N, members)[ci]]
    y = np.zeros((len(ri), len(ci)), dtype=np.float64)
    for kb in range(_ceil_div(K, BLOCK)):
        c0, c1 = kb * BLOCK, min(kb * BLOCK + BLOCK, K)
        partial = A[:, c0:c1] @ W[:, c0:c1].T
        y += partial * (sa[:, kb][:, None] * sw[:, kb][None, :])
    return y


def linear_w8a16(x_bits, q_w, s_w, members=None, rows=None, cols=None) -> np.ndarray:
    """W8A16 block-scaled projection in float64 (BF16 activations).

    x_bits: uint16 [M, K] BF16 bits; the other arguments as in linear_w8a8.
    """
    q_w = np.asarray(q_w, dtype=np.uint8)
    x = bf16_bits_to_f32(np.asarray(x_bits, dtype=np.uint16)).astype(np.float64)
    M, K = x.shape
    N = q_w.shape[0]
    ri, ci = _sel(M, rows), _sel(N, cols)
    X = x[ri]
    W = e4m3_decode_lut()[q_w[ci]]
    sw = _scales_f64(s_w)[scale_rows(N, members)[ci]]
    y = np.zeros((len(ri), len(ci)), dtype=np.float64)
    for kb in range(_ceil_div(K, BLOCK)):
        c0, c1 = kb * BLOCK, min(kb * BLOCK + BLOCK, K)
        y += (X[:, c0:c1] @ W[:, c0:c1].T) * sw[:, kb][None, :]
    return y


def grouped_linear_w8a8(q_a, s_a, q_w, s_w, offsets, rows=None, cols=None) -> np.ndarray:
    """Per-expert W8A8 projection over an expert-sorted token table.

    q_a: uint8 [T, K] rows sorted by expert; s_a: float32 [T, Kb];
    q_w: uint8 [G, N, K]; s_w: [G, ceil(N/128), Kb]; offsets: int [G+1].
    Row t belongs to the expert e with offsets[e] <= t < offsets[e+1].
    """
    q_a = np.asarray(q_a, dtype=np.uint8)
    offsets = np.asarray(offsets, dtype=np.int64)
    T = q_a.shape[0]
    G, N = q_w.shape[0], q_w.shape[1]
    ri, ci = _sel(T, rows), _sel(N, cols)
    expert_of_row = np.searchsorted(offsets, ri, side="right") - 1
    y = np.zeros((len(ri), len(ci)), dtype=np.float64)
    for e in range(G):
        sel = np.nonzero(expert_of_row == e)[0]
        if sel.size == 0:
            continue
        y[sel] = linear_w8a8(q_a, s_a, q_w[e], s_w[e], rows=ri[sel], cols=ci)
    return y


def route_topk(logits, k: int):
    """Softmax top-k routing and the expert-sorted row table.

    logits: float32 [T, E]. Returns a dict:
      experts [T, k] (chosen experts, by decreasing probability),
      weights [T, k] float64 (renormalised to sum to 1 per token),
      row_token [T*k], row_expert [T*k], row_slot [T*k] (rows sorted by
      expert, token-major within an expert), offsets int64 [E+1],
      row_of [T, k] (the sorted row holding token t's j-th choice).
    """
    z = np.asarray(logits, dtype=np.float64)
    T, E = z.shape
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")      # ties -> lower expert id
    experts = order[:, :k]
    top_p = np.take_along_axis(p, experts, axis=1)
    weights = top_p / top_p.sum(axis=1, keepdims=True)
    flat_expert = experts.reshape(-1)
    flat_token = np.repeat(np.arange(T), k)
    flat_slot = np.tile(np.arange(k), T)
    perm = np.argsort(flat_expert, kind="stable")
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(np.bincount(flat_expert, minlength=E))
    row_of = np.empty((T, k), dtype=np.int64)
    row_of[flat_token[perm], flat_slot[perm]] = np.arange(T * k)
    return {
        "experts": experts,
        "weights": weights,
        "row_token": flat_token[perm],
        "row_expert": flat_expert[perm],
        "row_slot": flat_slot[perm],
        "offsets": offsets,
        "row_of": row_of,
    }
