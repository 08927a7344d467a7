"""The Python binding's argument checks, on the CPU.

Every pointer the library takes must be device memory of the current GPU,
and every tensor must hold all the elements the call will address (rows x
columns at the strides passed, in the library's element size). Both are
refused in the binding, before the library sees the call: a kernel reading
a host address, or past a too-small tensor, would fault the GPU.

A valid call made with host tensors must fail on the device check alone,
which shows that the extent checks accept every argument layout the library
supports (strided outputs, token-contiguous scales, member grids, expert
stacks, per-tensor multipliers)."""

import pytest
import torch

M, K, N = 20, 320, 384
Kb, Nb = 3, 3
bf16, u8, f32, i32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32


def _device_error(fn, *args, **kw):
    with pytest.raises(ValueError, match="CUDA tensor"):
        fn(*args, **kw)


def _too_small(fn, *args, **kw):
    with pytest.raises(ValueError, match="too small"):
        fn(*args, **kw)


def _bad_layout(fn, *args, **kw):
    with pytest.raises(ValueError, match="has shape|strides|per-tensor scale needs"):
        fn(*args, **kw)


def test_valid_dense_calls_pass_the_extent_checks(bfp8):
    x = torch.zeros(M, K, dtype=bf16)
    q = torch.zeros(M, K, dtype=u8)
    s = torch.zeros(M, Kb, dtype=f32)
    _device_error(bfp8.bfp8_act_quant_group, x, q, s)
    st = torch.zeros(Kb, M, dtype=f32)          # token-contiguous scales
    _device_error(bfp8.bfp8_act_quant_group, x, q, st, s_stride_m=1, s_stride_kb=M)
    gu = torch.zeros(M, 2 * K, dtype=bf16)
    _device_error(bfp8.bfp8_silu_mul_act_quant, gu, q, s)
    _device_error(bfp8.bfp8_quantize_weight_block, torch.zeros(N, K, dtype=f32),
                  torch.zeros(N, K, dtype=u8), torch.zeros(Nb, Kb, dtype=bf16))
    w = torch.zeros(N, K, dtype=u8)
    yb = torch.zeros(M, N + 8, dtype=bf16)
    y = yb[:, :N]                                # strided output
    for sw in (torch.zeros(Nb, Kb, dtype=bf16), torch.zeros(Nb, Kb, dtype=f32),
               torch.ones((), dtype=f32)):
        _device_error(bfp8.bfp8_linear_w8a8, q, s, w, sw, y)
        _device_error(bfp8.bfp8_linear_w8a16, x, w, sw, y)
        _device_error(bfp8.bfp8_gemv_decode_noalloc, x[:4], w, sw, y[:4])
    members = [200, 184]                         # grid rows 2 + 2
    swm = torch.zeros(4, Kb, dtype=bf16)
    _device_error(bfp8.bfp8_linear_w8a8, q, s, w, swm, y, member_rows=members)
    ws = torch.zeros(1 << 16, dtype=u8)
    _device_error(bfp8.bfp8_gemv_decode, x[:4], w, swm, y[:4], ws, member_rows=members)
    _device_error(bfp8.bfp8_gemv_decode_w8a8, q[:4], s[:4], w, swm, y[:4], ws,
                  member_rows=members)
    I = N // 2                                   # fused gate/up: grid rows 2 * ceil(I / 128)
    _device_error(bfp8.bfp8_linear_w8a8_silu_quant, q, s, w, torch.zeros(4, Kb, dtype=bf16),
                  torch.zeros(M, I, dtype=u8), torch.zeros(M, 2, dtype=f32))


def test_valid_grouped_moe_and_decode_calls_pass_the_extent_checks(bfp8):
    G, T = 4, 50
    q = torch.zeros(T, K, dtype=u8)
    s = torch.zeros(T, Kb, dtype=f32)
    off = torch.tensor([0, 10, 10, 30, 50], dtype=i32)
    w = torch.zeros(G, N, K, dtype=u8)
    y = torch.zeros(T, N, dtype=bf16)
    for sw in (torch.zeros(G, Nb, Kb, dtype=bf16), torch.ones(G, dtype=f32)):
        _device_error(bfp8.bfp8_grouped_linear, q, s, w, sw, off, y)
    I = N // 2
    _device_error(bfp8.bfp8_grouped_linear_silu_quant, q, s, w, torch.zeros(G, 4, Kb, dtype=bf16),
                  off, torch.zeros(T, I, dtype=u8), torch.zeros(T, 2, dtype=f32))
    H, R, k = 256, 12, 3
    x = torch.zeros(6, H, dtype=bf16)
    _device_error(bfp8.bfp8_moe_gather_act_quant, x, torch.zeros(R, dtype=i32),
                  torch.zeros(R, H, dtype=u8), torch.zeros(R, 2, dtype=f32))
    _device_error(bfp8.bfp8_moe_combine, torch.zeros(R, H, dtype=bf16),
                  torch.zeros(4, k, dtype=i32), torch.zeros(4, k, dtype=f32),
                  torch.zeros(4, H, dtype=bf16))
    Hh, Ii = 256, 384
    _device_error(bfp8.bfp8_decode_ffn, torch.zeros(2, Hh, dtype=bf16),
                  torch.zeros(2 * Ii, Hh, dtype=u8), torch.zeros(6, 2, dtype=bf16),
                  torch.zeros(Hh, Ii, dtype=u8), torch.zeros(2, 3, dtype=bf16),
                  torch.zeros(2, Hh, dtype=bf16), torch.zeros(1 << 16, dtype=u8))


def test_tensors_too_small_for_the_call_are_refused(bfp8):
    x = torch.zeros(M, K, dtype=bf16)
    q = torch.zeros(M, K, dtype=u8)
    s = torch.zeros(M, Kb, dtype=f32)
    _too_small(bfp8.bfp8_act_quant_group, x, q[: M - 1], s)           # shape [M-1, K]
    _too_small(bfp8.bfp8_act_quant_group, x, q, s[:, :2])             # strides reach past
    _too_small(bfp8.bfp8_act_quant_group, x, q, torch.zeros(Kb, M - 1, dtype=f32),
               s_stride_m=1, s_stride_kb=M)
    w = torch.zeros(N, K, dtype=u8)
    y = torch.zeros(M, N, dtype=bf16)
    _bad_layout(bfp8.bfp8_linear_w8a8, q, s, w, torch.zeros(Nb - 1, Kb, dtype=bf16), y)
    _too_small(bfp8.bfp8_linear_w8a8, q, s, w, torch.zeros(Nb, Kb, dtype=bf16), y[: M - 1])
    _bad_layout(bfp8.bfp8_linear_w8a8, q, s, w, torch.zeros(3, Kb, dtype=bf16), y,
                member_rows=[200, 184])                               # needs 4 grid rows
    G, T = 4, 50
    off = torch.tensor([0, 10, 10, 30], dtype=i32)                     # needs G + 1 entries
    _bad_layout(bfp8.bfp8_grouped_linear, torch.zeros(T, K, dtype=u8), torch.zeros(T, Kb, dtype=f32),
               torch.zeros(G, N, K, dtype=u8), torch.zeros(G, Nb, Kb, dtype=bf16), off,
               torch.zeros(T, N, dtype=bf16))
    _bad_layout(bfp8.bfp8_moe_combine, torch.zeros(12, 256, dtype=bf16),
                torch.zeros(4, 3, dtype=i32), torch.zeros(4, 2, dtype=f32),
                torch.zeros(4, 256, dtype=bf16))


def test_layouts_the_library_would_misread_are_refused(bfp8):
    """The kernels read weights, quantized activations and scale grids as dense
    row-major data with the pitch implied by K. A transposed grid, a column
    slice of a wider weight, or a transposed activation would be misread
    silently, so the binding refuses them by shape and stride."""
    q = torch.zeros(M, K, dtype=u8)
    s = torch.zeros(M, Kb, dtype=f32)
    w = torch.zeros(N, K, dtype=u8)
    y = torch.zeros(M, N, dtype=bf16)
    K2 = 256                                             # Kb = 2, Nb = 3: the transpose has another shape
    q2, s2, w2 = torch.zeros(M, K2, dtype=u8), torch.zeros(M, 2, dtype=f32), torch.zeros(N, K2, dtype=u8)
    _bad_layout(bfp8.bfp8_linear_w8a8, q2, s2, w2, torch.zeros(2, Nb, dtype=bf16), y)   # [Kb, Nb]
    _bad_layout(bfp8.bfp8_linear_w8a8, q, s, w, torch.zeros(Kb, Nb, dtype=bf16).t(), y)  # .t() view
    wide = torch.zeros(N, K + 64, dtype=u8)
    _bad_layout(bfp8.bfp8_linear_w8a8, q, s, wide[:, :K], torch.zeros(Nb, Kb, dtype=bf16), y)
    _bad_layout(bfp8.bfp8_linear_w8a16, torch.zeros(M, K, dtype=bf16), wide[:, :K],
                torch.zeros(Nb, Kb, dtype=bf16), y)
    _bad_layout(bfp8.bfp8_gemv_decode, torch.zeros(4, K, dtype=bf16), w.t().contiguous().t(),
                torch.zeros(Nb, Kb, dtype=bf16), y[:4], torch.zeros(1 << 16, dtype=u8))
    _bad_layout(bfp8.bfp8_linear_w8a8, torch.zeros(K, M, dtype=u8).t(), s, w,
                torch.zeros(Nb, Kb, dtype=bf16), y)               # transposed activations
    with pytest.raises(ValueError, match="contiguous columns"):
        bfp8.bfp8_linear_w8a16(torch.zeros(K, M, dtype=bf16).t(), w,
                               torch.zeros(Nb, Kb, dtype=bf16), y)
    with pytest.raises(ValueError, match="contiguous columns"):
        bfp8.bfp8_linear_w8a8(q, s, w, torch.zeros(Nb, Kb, dtype=bf16),
                              torch.zeros(N, M, dtype=bf16).t())  # transposed output
    G, T = 4, 50
    off = torch.tensor([0, 10, 10, 30, 50], dtype=i32)
    _bad_layout(bfp8.bfp8_grouped_linear, torch.zeros(T, K2, dtype=u8), torch.zeros(T, 2, dtype=f32),
                torch.zeros(G, N, K2, dtype=u8), torch.zeros(G, 2, Nb, dtype=bf16), off,
                torch.zeros(T, N, dtype=bf16))                   # per-expert grids transposed
    _bad_layout(bfp8.bfp8_grouped_linear, torch.zeros(T, K, dtype=u8), torch.zeros(T, Kb, dtype=f32),
                torch.zeros(G, N, K, dtype=u8), torch.ones(G - 1, dtype=f32), off,
                torch.zeros(T, N, dtype=bf16))                   # one multiplier per expert


def test_decode_step_scales_must_share_one_dtype_and_kind(bfp8):
    """bfp8_decode_ffn takes one scale dtype code for its two grids, so a
    BF16 grid beside an F32 one, or a block grid beside one multiplier, would
    be misread (a one-element tensor read as a grid, past its end)."""
    Hh, Ii = 256, 384
    x = torch.zeros(2, Hh, dtype=bf16)
    wgu, wd = torch.zeros(2 * Ii, Hh, dtype=u8), torch.zeros(Hh, Ii, dtype=u8)
    y, ws = torch.zeros(2, Hh, dtype=bf16), torch.zeros(1 << 16, dtype=u8)
    for sgu, sd in ((torch.zeros(6, 2, dtype=bf16), torch.zeros(2, 3, dtype=f32)),
                    (torch.zeros(6, 2, dtype=bf16), torch.ones((), dtype=bf16)),
                    (torch.ones((), dtype=f32), torch.zeros(2, 3, dtype=f32))):
        with pytest.raises(ValueError, match="same dtype and kind"):
            bfp8.bfp8_decode_ffn(x, wgu, sgu, wd, sd, y, ws)
    for sgu, sd in ((torch.ones((), dtype=f32), torch.ones((), dtype=f32)),
                    (torch.zeros(6, 2, dtype=f32), torch.zeros(2, 3, dtype=f32))):
        _device_error(bfp8.bfp8_decode_ffn, x, wgu, sgu, wd, sd, y, ws)


def test_tensors_of_another_element_type_are_refused(bfp8):
    """The library reads each argument as one element type; a tensor of another
    type (a float32 activation, int64 offsets, a BF16 weight to quantize) would
    be reinterpreted byte for byte, so the binding refuses it by dtype. E4M3
    data is accepted as uint8 or float8_e4m3fn."""
    x = torch.zeros(M, K, dtype=bf16)
    q = torch.zeros(M, K, dtype=u8)
    s = torch.zeros(M, Kb, dtype=f32)
    w = torch.zeros(N, K, dtype=u8)
    sw = torch.zeros(Nb, Kb, dtype=bf16)
    y = torch.zeros(M, N, dtype=bf16)

    def refused(fn, *args, **kw):
        with pytest.raises(ValueError, match="must be torch"):
            fn(*args, **kw)

    refused(bfp8.bfp8_act_quant_group, x.float(), q, s)
    refused(bfp8.bfp8_act_quant_group, x, q, s.double())
    refused(bfp8.bfp8_linear_w8a8, q, s, w, sw, y.float())
    refused(bfp8.bfp8_linear_w8a8, q.to(torch.int8), s, w, sw, y)
    refused(bfp8.bfp8_linear_w8a16, x.half(), w, sw, y)
    refused(bfp8.bfp8_quantize_weight_block, torch.zeros(N, K, dtype=bf16), w, sw)
    G, T = 4, 50
    refused(bfp8.bfp8_grouped_linear, torch.zeros(T, K, dtype=u8), torch.zeros(T, Kb, dtype=f32),
            torch.zeros(G, N, K, dtype=u8), torch.zeros(G, Nb, Kb, dtype=bf16),
            torch.tensor([0, 10, 10, 30, 50]), torch.zeros(T, N, dtype=bf16))   # int64 offsets
    refused(bfp8.bfp8_moe_combine, torch.zeros(12, 256, dtype=bf16),
            torch.zeros(4, 3, dtype=i32), torch.zeros(4, 3, dtype=bf16),
            torch.zeros(4, 256, dtype=bf16))
    # float8_e4m3fn views of the same bytes pass the dtype check (and stop at the device check)
    _device_error(bfp8.bfp8_linear_w8a8, q.view(torch.float8_e4m3fn), s,
                  w.view(torch.float8_e4m3fn), sw, y)
