"""Python binding of libbfp8: the C ABI of include/bfp8.h, name for name.

Argument marshalling only. Every function takes torch tensors (device memory
and shapes come from them), passes raw pointers, sizes and the current CUDA
stream to the library, and raises Bfp8Error on a non-zero status. Nothing
here computes. If libbfp8.so is missing, importing this module raises.
Nothing falls back to another implementation.
"""

from __future__ import annotations

import ctypes
import os
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libbfp8.so"

if not _LIB_PATH.exists():
    raise ImportError(
        f"{_LIB_PATH} is missing: build it with "
        "`python -m block_scaled_fp8_token_gb300.build` (needs nvcc). "
        "There is no fallback implementation.")

_lib = ctypes.CDLL(os.fspath(_LIB_PATH))

# ---- enums (include/bfp8.h) ------------------------------------------------
BFP8_OK = 0
STATUS_NAMES = {
    0: "OK", 1: "INVALID_ARG", 2: "E5M2", 3: "NO_SCALE", 4: "ROW_SCALE",
    5: "AMBIGUOUS_SCALE", 6: "GRID_TRANSPOSED", 7: "GRID_SHAPE", 8: "SCALE_DTYPE",
    9: "BLOCK_SIZE", 10: "QUANT_METHOD", 11: "GROUP", 12: "NOT_FP8",
    13: "UNSUPPORTED", 14: "CUDA", 15: "TIMEOUT",
}
BFP8_DT_NONE, BFP8_DT_E4M3, BFP8_DT_E5M2, BFP8_DT_BF16, BFP8_DT_F16, BFP8_DT_F32 = range(6)
BFP8_MAX_MEMBERS = 8


class Bfp8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bfp8_status_string(status)} ({status})")


class bfp8_weight_desc(ctypes.Structure):
    _fields_ = [
        ("weight_dtype", ctypes.c_int32),
        ("weight_rank", ctypes.c_int32),
        ("weight_shape", ctypes.c_int64 * 2),
        ("scale_dtype", ctypes.c_int32),
        ("scale_rank", ctypes.c_int32),
        ("scale_shape", ctypes.c_int64 * 2),
        ("has_row_scale", ctypes.c_int32),
        ("declared_quant_fp8", ctypes.c_int32),
        ("declared_block", ctypes.c_int32 * 2),
        ("n_members", ctypes.c_int32),
        ("member_rows", ctypes.POINTER(ctypes.c_int64)),
        ("tensor_scale_dtype", ctypes.c_int32),
    ]


class bfp8_members(ctypes.Structure):
    _fields_ = [("n_members", ctypes.c_int32), ("member_rows", ctypes.POINTER(ctypes.c_int64))]


_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
_SIGS = {
    "bfp8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bfp8_validate_grid": (ctypes.c_int, [ctypes.POINTER(bfp8_weight_desc), ctypes.c_char_p, _sz]),
    "bfp8_act_quant_group": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp]),
    "bfp8_silu_mul_act_quant": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp]),
    "bfp8_silu_mul": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp]),
    "bfp8_quantize_weight_block": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i32, _vp]),
    "bfp8_linear_w8a8": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i32, _i64, _i64, _i64,
                                        _vp, _i64, ctypes.POINTER(bfp8_members), _vp, _sz, _vp]),
    "bfp8_linear_w8a8_workspace": (_sz, [_i64, _i64, _i64, ctypes.POINTER(bfp8_members)]),
    "bfp8_linear_w8a16": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _i64,
                                         ctypes.POINTER(bfp8_members), _vp]),
    "bfp8_gemv_decode": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _i64, _i64, _i64, _vp, _i64,
                                        ctypes.POINTER(bfp8_members), _vp, _sz, _vp]),
    "bfp8_gemv_decode_workspace": (_sz, [_i64, _i64, _i64]),
    "bfp8_gemv_decode_w8a8": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i32, _i64, _i64,
                                             _i64, _vp, _i64, ctypes.POINTER(bfp8_members), _vp,
                                             _sz, _vp]),
    "bfp8_gemv_decode_noalloc": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _i64, _i64, _i64, _vp,
                                                _i64, ctypes.POINTER(bfp8_members), _vp]),
    "bfp8_grouped_linear": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i32, _vp, _i32, _i64,
                                           _i64, _i64, _vp, _i64, _vp, _sz, _vp]),
    "bfp8_grouped_linear_workspace": (_sz, [_i64, _i32, _i64, _i64]),
    "bfp8_linear_w8a8_silu_quant": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i32, _i64,
                                                   _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp,
                                                   _sz, _vp]),
    "bfp8_linear_w8a8_silu_quant_workspace": (_sz, [_i64, _i64, _i64]),
    "bfp8_grouped_linear_silu_quant": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i32, _vp,
                                                      _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                                      _i64, _vp, _sz, _vp]),
    "bfp8_grouped_linear_silu_quant_workspace": (_sz, [_i64, _i32, _i64, _i64]),
    "bfp8_decode_ffn": (ctypes.c_int, [_i32, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64,
                                       _vp, _i64, _vp, _sz, _vp]),
    "bfp8_decode_ffn_workspace": (_sz, [_i64, _i64, _i64, _i32]),
    "bfp8_moe_gather_act_quant": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp,
                                                 _i64, _i64, _vp]),
    "bfp8_moe_combine": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _i32, _vp, _i64,
                                        _vp]),
    "bfp8_device_status": (ctypes.c_int, [_vp]),
    "bfp8_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def library_path() -> Path:
    return _LIB_PATH


def bfp8_status_string(status: int) -> str:
    return _lib.bfp8_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != BFP8_OK:
        raise Bfp8Error(status, where)


def _ptr(t) -> int | None:
    """A tensor's device address. Every pointer the library takes is memory of
    the current device; a host tensor, or one on another GPU, is refused here,
    before any kernel could read it."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"bfp8: expected a CUDA tensor, got one on {t.device}")
    if t.get_device() != torch.cuda.current_device():
        raise ValueError(f"bfp8: tensor on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


BFP8_SCALE_PER_TENSOR = 0x100


def _scale_dtype(t: torch.Tensor) -> int:
    """The dtype code of a scale tensor. A block grid has rank 2 (rank 3 for
    experts); a scale of rank 0 or 1 (one multiplier, or one per expert) is a
    per-tensor scale and carries BFP8_SCALE_PER_TENSOR."""
    code = {torch.bfloat16: BFP8_DT_BF16, torch.float32: BFP8_DT_F32,
            torch.float16: BFP8_DT_F16}.get(t.dtype, BFP8_DT_NONE)
    return code | BFP8_SCALE_PER_TENSOR if code and t.dim() <= 1 else code


def _members(member_rows):
    if member_rows is None:
        return None, None
    arr = (ctypes.c_int64 * len(member_rows))(*[int(v) for v in member_rows])
    m = bfp8_members(len(member_rows), arr)
    return ctypes.byref(m), (m, arr)


def bfp8_validate_grid(desc: bfp8_weight_desc, msg_len: int = 256) -> tuple[int, str]:
    """Returns (status, message). Host only: needs no GPU."""
    buf = ctypes.create_string_buffer(msg_len)
    rc = _lib.bfp8_validate_grid(ctypes.byref(desc), buf, msg_len)
    return rc, buf.value.decode()


def make_weight_desc(weight_dtype: int, weight_shape, scale_dtype: int = BFP8_DT_NONE,
                     scale_shape=None, has_row_scale: bool = False,
                     declared_quant_fp8: bool = True, declared_block=(128, 128),
                     member_rows=None, tensor_scale_dtype: int = BFP8_DT_NONE):
    """Builds a bfp8_weight_desc; returns (desc, keepalive)."""
    d = bfp8_weight_desc()
    d.weight_dtype = weight_dtype
    d.weight_rank = len(weight_shape)
    for i, v in enumerate(list(weight_shape)[:2]):
        d.weight_shape[i] = int(v)
    d.scale_dtype = scale_dtype
    sshape = list(scale_shape) if scale_shape is not None else []
    d.scale_rank = len(sshape)
    for i, v in enumerate(sshape[:2]):
        d.scale_shape[i] = int(v)
    d.has_row_scale = int(bool(has_row_scale))
    d.declared_quant_fp8 = int(bool(declared_quant_fp8))
    d.declared_block[0], d.declared_block[1] = int(declared_block[0]), int(declared_block[1])
    d.tensor_scale_dtype = tensor_scale_dtype
    keep = None
    if member_rows is not None:
        keep = (ctypes.c_int64 * len(member_rows))(*[int(v) for v in member_rows])
        d.n_members = len(member_rows)
        d.member_rows = keep
    return d, keep


def bfp8_act_quant_group(x, q, scales, s_stride_m=None, s_stride_kb=None, stream=None) -> None:
    M, K = x.shape
    ssm = scales.stride(0) if s_stride_m is None else s_stride_m
    sskb = scales.stride(1) if s_stride_kb is None else s_stride_kb
    _dtypes(x=(x, "bf16"), q=(q, "e4m3"), scales=(scales, "f32"))
    _rows(x, "x")
    _span(x, "x", M, K, x.stride(0), 1, 2)
    _out(q, "q", M, K, 1)
    _scales_out(scales, "scales", M, -(-K // 128), ssm, sskb,
                s_stride_m is not None or s_stride_kb is not None)
    _check(_lib.bfp8_act_quant_group(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0),
                                     _ptr(scales), ssm, sskb, _stream(stream)),
           "bfp8_act_quant_group")


def bfp8_silu_mul_act_quant(gu, q, scales, s_stride_m=None, s_stride_kb=None, stream=None) -> None:
    M, two_i = gu.shape
    ssm = scales.stride(0) if s_stride_m is None else s_stride_m
    sskb = scales.stride(1) if s_stride_kb is None else s_stride_kb
    _dtypes(gu=(gu, "bf16"), q=(q, "e4m3"), scales=(scales, "f32"))
    _rows(gu, "gu")
    _span(gu, "gu", M, two_i, gu.stride(0), 1, 2)
    _out(q, "q", M, two_i // 2, 1)
    _scales_out(scales, "scales", M, -(-(two_i // 2) // 128), ssm, sskb,
                s_stride_m is not None or s_stride_kb is not None)
    _check(_lib.bfp8_silu_mul_act_quant(_ptr(gu), M, two_i // 2, gu.stride(0), _ptr(q),
                                        q.stride(0), _ptr(scales), ssm, sskb, _stream(stream)),
           "bfp8_silu_mul_act_quant")


def bfp8_silu_mul(gu, h, stream=None) -> None:
    """h = bf16(silu(gate) * up) for gu = [gate | up] ([M, 2I] BF16); h [M, I] BF16."""
    M, two_i = gu.shape
    _dtypes(gu=(gu, "bf16"), h=(h, "bf16"))
    _rows(gu, "gu")
    _span(gu, "gu", M, two_i, gu.stride(0), 1, 2)
    _out(h, "h", M, two_i // 2, 2)
    _check(_lib.bfp8_silu_mul(_ptr(gu), M, two_i // 2, gu.stride(0), _ptr(h), h.stride(0),
                              _stream(stream)),
           "bfp8_silu_mul")


def bfp8_quantize_weight_block(w, q, scale, stream=None) -> None:
    N, K = w.shape
    _dtypes(w=(w, "f32"), q=(q, "e4m3"))
    _rows(w, "w")
    _span(w, "w", N, K, w.stride(0), 1, 4)  # float32, as the library reads it
    _out(q, "q", N, K, 1)
    _grid_span(scale, "scale", -(-N // 128), -(-K // 128))
    _check(_lib.bfp8_quantize_weight_block(_ptr(w), N, K, w.stride(0), _ptr(q), q.stride(0),
                                           _ptr(scale), _scale_dtype(scale), _stream(stream)),
           "bfp8_quantize_weight_block")


def _span(t, name: str, rows: int, cols: int, rs: int, cs: int, elem_bytes: int) -> None:
    """Refuse a call that would make the library touch memory past the end of
    t's storage: rows x cols elements of elem_bytes bytes at element strides
    (rs, cs) from t's first element, as the library addresses them."""
    if t is None or isinstance(t, int) or rows <= 0 or cols <= 0:
        return
    if rs < 0 or cs < 0:
        raise ValueError(f"bfp8: {name}: negative stride ({rs}, {cs})")
    need = ((rows - 1) * rs + (cols - 1) * cs + 1) * elem_bytes
    if need <= t.numel() * t.element_size() and t.is_contiguous():
        return  # within the tensor's own elements
    st = t.untyped_storage()
    if t.data_ptr() + need > st.data_ptr() + st.nbytes():
        raise ValueError(f"bfp8: {name} is too small for the call: {rows} x {cols} elements "
                         f"at strides ({rs}, {cs}) reach past its storage")


def _layout(t, name: str, shape, pitch: int | None = None) -> None:
    """t must have exactly `shape` and unit stride along its last dimension
    (row pitch `pitch` when given, dense strides for higher ranks): the
    library reads it as dense row-major data, so a transposed view, a column
    slice or a permuted grid would be misread silently. Strides of size-1
    dimensions do not matter and are not checked."""
    if t is None or isinstance(t, int):
        return
    shape = tuple(int(v) for v in shape)
    if tuple(t.shape) != shape:
        raise ValueError(f"bfp8: {name} has shape {list(t.shape)}, expected {list(shape)}")
    want = [1] * len(shape)
    for d in range(len(shape) - 2, -1, -1):
        want[d] = want[d + 1] * shape[d + 1]
    if pitch is not None and len(shape) >= 2:
        want[-2] = int(pitch)
    for d, (st, w) in enumerate(zip(t.stride(), want)):
        if shape[d] > 1 and st != w:
            raise ValueError(f"bfp8: {name} has strides {list(t.stride())}; the library reads it "
                             f"as row-major with strides {want}")


_KINDS = {"bf16": (torch.bfloat16,), "e4m3": (torch.uint8, torch.float8_e4m3fn),
          "f32": (torch.float32,), "i32": (torch.int32,)}


def _dtypes(**args) -> None:
    """Each tensor must hold the element type the library reads or writes at
    that argument (name=(tensor, kind)): a tensor of another type would be
    reinterpreted byte for byte. E4M3 data may be uint8 or float8_e4m3fn."""
    for name, (t, kind) in args.items():
        if t is None or isinstance(t, int):
            continue
        if t.dtype not in _KINDS[kind]:
            allowed = " or ".join(str(d) for d in _KINDS[kind])
            raise ValueError(f"bfp8: {name} must be {allowed}, got {t.dtype}")


def _rows(t, name: str) -> None:
    """An activation or output matrix passed with its own row pitch: the
    columns must be contiguous (unit stride along the last dimension)."""
    if t is None or isinstance(t, int) or t.dim() != 2:
        return
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"bfp8: {name} must have contiguous columns, got strides "
                         f"{list(t.stride())}")


def _out(t, name: str, rows: int, cols: int, elem_bytes: int) -> None:
    """An output the library writes as rows x cols row-major elements at
    t.stride(0): the view must cover them, not only its storage."""
    if rows <= 0 or cols <= 0:
        return
    if t.dim() != 2 or t.shape[0] < rows or t.shape[1] < cols:
        raise ValueError(f"bfp8: {name} is too small for the call: needs [{rows}, {cols}], "
                         f"got {list(t.shape)}")
    _rows(t, name)
    _span(t, name, rows, cols, t.stride(0), 1, elem_bytes)


def _scales_out(t, name: str, rows: int, cols: int, s_m: int, s_kb: int, explicit: bool) -> None:
    """A float32 scale output [rows, cols]: with the view's own strides the
    view must cover it; with caller strides (for example token-contiguous
    scales) only the storage can be checked."""
    if not explicit and rows > 0 and cols > 0 and (
            t.dim() != 2 or t.shape[0] < rows or t.shape[1] < cols):
        raise ValueError(f"bfp8: {name} is too small for the call: needs [{rows}, {cols}], "
                         f"got {list(t.shape)}")
    _span(t, name, rows, cols, s_m, s_kb, 4)


_SCALE_BYTES = {BFP8_DT_BF16: 2, BFP8_DT_F16: 2, BFP8_DT_F32: 4}


def _grid_span(t, name: str, rows: int, kb: int, experts: int | None = None) -> None:
    """A weight-scale argument: the block grid [rows, kb] (rows = the sum of
    ceil(N_i / 128) over members, kb = ceil(K / 128)), or [experts, rows, kb]
    for expert stacks, dense row-major; or one multiplier (one per expert) as
    a tensor of rank 0 or 1. A transposed or mis-shaped grid is refused here
    (the library would read it as this layout)."""
    eb = _SCALE_BYTES.get(_scale_dtype(t) & 0xFF)
    if eb is None:
        return  # refused by the library (SCALE_DTYPE) before anything is read
    n = 1 if experts is None else experts
    if t.dim() <= 1:
        if t.numel() != n:
            raise ValueError(f"bfp8: {name}: a per-tensor scale needs {n} element(s), "
                             f"got {t.numel()}")
        _span(t, name, n, 1, 1, 1, eb)
        return
    _layout(t, name, (rows, kb) if experts is None else (experts, rows, kb))
    _span(t, name, n * rows, kb, kb, 1, eb)


def _scale_rows(N: int, member_rows) -> int:
    return sum(-(-int(m) // 128) for m in member_rows) if member_rows else -(-N // 128)


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def bfp8_linear_w8a8_workspace(M: int, N: int, K: int, member_rows=None) -> int:
    mref, _keep = _members(member_rows)
    return int(_lib.bfp8_linear_w8a8_workspace(M, N, K, mref))


def bfp8_linear_w8a8(q_a, s_a, w, w_scale, y, member_rows=None, s_stride_m=None,
                     s_stride_kb=None, workspace=None, stream=None) -> None:
    M, K = q_a.shape
    N = w.shape[0]
    ssm = s_a.stride(0) if s_stride_m is None else s_stride_m
    sskb = s_a.stride(1) if s_stride_kb is None else s_stride_kb
    Kb = -(-K // 128)
    _dtypes(q_a=(q_a, "e4m3"), s_a=(s_a, "f32"), w=(w, "e4m3"), y=(y, "bf16"))
    _layout(q_a, "q_a", (M, K))
    _span(s_a, "s_a", M, Kb, ssm, sskb, 4)
    _layout(w, "w", (N, K))
    _grid_span(w_scale, "w_scale", _scale_rows(N, member_rows), Kb)
    _out(y, "y", M, N, 2)
    mref, _keep = _members(member_rows)
    wsp, wsb = _ws(workspace)
    _check(_lib.bfp8_linear_w8a8(_ptr(q_a), _ptr(s_a), ssm, sskb, _ptr(w), _ptr(w_scale),
                                 _scale_dtype(w_scale), M, N, K, _ptr(y), y.stride(0), mref,
                                 wsp, wsb, _stream(stream)),
           "bfp8_linear_w8a8")


def bfp8_linear_w8a16(x, w, w_scale, y, member_rows=None, stream=None) -> None:
    M, K = x.shape
    N = w.shape[0]
    _dtypes(x=(x, "bf16"), w=(w, "e4m3"), y=(y, "bf16"))
    _rows(x, "x")
    _span(x, "x", M, K, x.stride(0), 1, 2)
    _layout(w, "w", (N, K))
    _grid_span(w_scale, "w_scale", _scale_rows(N, member_rows), -(-K // 128))
    _out(y, "y", M, N, 2)
    mref, _keep = _members(member_rows)
    _check(_lib.bfp8_linear_w8a16(_ptr(x), x.stride(0), _ptr(w), _ptr(w_scale),
                                  _scale_dtype(w_scale), M, N, K, _ptr(y), y.stride(0), mref,
                                  _stream(stream)),
           "bfp8_linear_w8a16")


def bfp8_gemv_decode_workspace(M: int, N: int, K: int) -> int:
    return int(_lib.bfp8_gemv_decode_workspace(M, N, K))


def bfp8_gemv_decode(x, w, w_scale, y, workspace, member_rows=None, stream=None) -> None:
    M, K = x.shape
    N = w.shape[0]
    _dtypes(x=(x, "bf16"), w=(w, "e4m3"), y=(y, "bf16"))
    _rows(x, "x")
    _span(x, "x", M, K, x.stride(0), 1, 2)
    _layout(w, "w", (N, K))
    _grid_span(w_scale, "w_scale", _scale_rows(N, member_rows), -(-K // 128))
    _out(y, "y", M, N, 2)
    mref, _keep = _members(member_rows)
    _check(_lib.bfp8_gemv_decode(_ptr(x), x.stride(0), _ptr(w), _ptr(w_scale),
                                 _scale_dtype(w_scale), M, N, K, _ptr(y), y.stride(0), mref,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)),
           "bfp8_gemv_decode")


def bfp8_gemv_decode_w8a8(q_a, s_a, w, w_scale, y, workspace, member_rows=None, s_stride_m=None,
                          s_stride_kb=None, stream=None) -> None:
    """Decode GEMV (M <= 16) on E4M3 tokens with 1x128 scales (W8A8 arithmetic)."""
    M, K = q_a.shape
    N = w.shape[0]
    ssm = s_a.stride(0) if s_stride_m is None else s_stride_m
    sskb = s_a.stride(1) if s_stride_kb is None else s_stride_kb
    Kb = -(-K // 128)
    _dtypes(q_a=(q_a, "e4m3"), s_a=(s_a, "f32"), w=(w, "e4m3"), y=(y, "bf16"))
    _layout(q_a, "q_a", (M, K))
    _span(s_a, "s_a", M, Kb, ssm, sskb, 4)
    _layout(w, "w", (N, K))
    _grid_span(w_scale, "w_scale", _scale_rows(N, member_rows), Kb)
    _out(y, "y", M, N, 2)
    mref, _keep = _members(member_rows)
    _check(_lib.bfp8_gemv_decode_w8a8(_ptr(q_a), _ptr(s_a), ssm, sskb, _ptr(w), _ptr(w_scale),
                                      _scale_dtype(w_scale), M, N, K, _ptr(y), y.stride(0), mref,
                                      _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(stream)),
           "bfp8_gemv_decode_w8a8")


def bfp8_gemv_decode_noalloc(x, w, w_scale, y, member_rows=None, stream=None) -> None:
    """bfp8_gemv_decode without a workspace argument, for callers that cannot
    allocate device memory; its scratch is a fixed array inside the library."""
    M, K = x.shape
    N = w.shape[0]
    _dtypes(x=(x, "bf16"), w=(w, "e4m3"), y=(y, "bf16"))
    _rows(x, "x")
    _span(x, "x", M, K, x.stride(0), 1, 2)
    _layout(w, "w", (N, K))
    _grid_span(w_scale, "w_scale", _scale_rows(N, member_rows), -(-K // 128))
    _out(y, "y", M, N, 2)
    mref, _keep = _members(member_rows)
    _check(_lib.bfp8_gemv_decode_noalloc(_ptr(x), x.stride(0), _ptr(w), _ptr(w_scale),
                                         _scale_dtype(w_scale), M, N, K, _ptr(y), y.stride(0),
                                         mref, _stream(stream)),
           "bfp8_gemv_decode_noalloc")


def bfp8_grouped_linear_workspace(total_M: int, G: int, N: int, K: int) -> int:
    return int(_lib.bfp8_grouped_linear_workspace(total_M, G, N, K))


def bfp8_grouped_linear(q_a, s_a, w, w_scale, offsets, y, s_stride_m=None, s_stride_kb=None,
                        workspace=None, stream=None) -> None:
    T, K = q_a.shape
    G, N = w.shape[0], w.shape[1]
    ssm = s_a.stride(0) if s_stride_m is None else s_stride_m
    sskb = s_a.stride(1) if s_stride_kb is None else s_stride_kb
    Kb = -(-K // 128)
    _dtypes(q_a=(q_a, "e4m3"), s_a=(s_a, "f32"), w=(w, "e4m3"), offsets=(offsets, "i32"),
            y=(y, "bf16"))
    _layout(q_a, "q_a", (T, K))
    _span(s_a, "s_a", T, Kb, ssm, sskb, 4)
    _layout(w, "w", (G, N, K))
    _grid_span(w_scale, "w_scale", -(-N // 128), Kb, G)
    _layout(offsets, "offsets", (G + 1,))
    _out(y, "y", T, N, 2)
    wsp, wsb = _ws(workspace)
    _check(_lib.bfp8_grouped_linear(_ptr(q_a), _ptr(s_a), ssm, sskb, _ptr(w), _ptr(w_scale),
                                    _scale_dtype(w_scale), _ptr(offsets), G, T, N, K, _ptr(y),
                                    y.stride(0), wsp, wsb, _stream(stream)),
           "bfp8_grouped_linear")


def bfp8_linear_w8a8_silu_quant_workspace(M: int, I: int, K: int) -> int:
    return int(_lib.bfp8_linear_w8a8_silu_quant_workspace(M, I, K))


def bfp8_linear_w8a8_silu_quant(q_a, s_a, w, w_scale, q_h, s_h, s_stride_m=None,
                                s_stride_kb=None, sh_stride_m=None, sh_stride_kb=None,
                                workspace=None, stream=None) -> None:
    """Gate/up projection (w = gate rows over up rows, [2I, K]) with SiLU(gate)*up
    and the 1x128 quantization of h fused into its epilogue: q_h [M, I], s_h."""
    M, K = q_a.shape
    I = w.shape[0] // 2
    ssm = s_a.stride(0) if s_stride_m is None else s_stride_m
    sskb = s_a.stride(1) if s_stride_kb is None else s_stride_kb
    hsm = s_h.stride(0) if sh_stride_m is None else sh_stride_m
    hskb = s_h.stride(1) if sh_stride_kb is None else sh_stride_kb
    Kb = -(-K // 128)
    _dtypes(q_a=(q_a, "e4m3"), s_a=(s_a, "f32"), w=(w, "e4m3"), q_h=(q_h, "e4m3"),
            s_h=(s_h, "f32"))
    _layout(q_a, "q_a", (M, K))
    _span(s_a, "s_a", M, Kb, ssm, sskb, 4)
    _layout(w, "w", (2 * I, K))
    _grid_span(w_scale, "w_scale", _scale_rows(2 * I, [I, I]), Kb)
    _out(q_h, "q_h", M, I, 1)
    _scales_out(s_h, "s_h", M, -(-I // 128), hsm, hskb,
                sh_stride_m is not None or sh_stride_kb is not None)
    wsp, wsb = _ws(workspace)
    _check(_lib.bfp8_linear_w8a8_silu_quant(_ptr(q_a), _ptr(s_a), ssm, sskb, _ptr(w),
                                            _ptr(w_scale), _scale_dtype(w_scale), M, I, K,
                                            _ptr(q_h), q_h.stride(0), _ptr(s_h), hsm, hskb, wsp,
                                            wsb, _stream(stream)),
           "bfp8_linear_w8a8_silu_quant")


def bfp8_grouped_linear_silu_quant_workspace(total_M: int, G: int, I: int, K: int) -> int:
    return int(_lib.bfp8_grouped_linear_silu_quant_workspace(total_M, G, I, K))


def bfp8_grouped_linear_silu_quant(q_a, s_a, w, w_scale, offsets, q_h, s_h, s_stride_m=None,
                                   s_stride_kb=None, sh_stride_m=None, sh_stride_kb=None,
                                   workspace=None, stream=None) -> None:
    """Per-expert gate/up projection (w [G, 2I, K]) with the fused SiLU*up +
    1x128 quant epilogue over the token-offset table."""
    T, K = q_a.shape
    G, I = w.shape[0], w.shape[1] // 2
    ssm = s_a.stride(0) if s_stride_m is None else s_stride_m
    sskb = s_a.stride(1) if s_stride_kb is None else s_stride_kb
    hsm = s_h.stride(0) if sh_stride_m is None else sh_stride_m
    hskb = s_h.stride(1) if sh_stride_kb is None else sh_stride_kb
    Kb = -(-K // 128)
    _dtypes(q_a=(q_a, "e4m3"), s_a=(s_a, "f32"), w=(w, "e4m3"), offsets=(offsets, "i32"),
            q_h=(q_h, "e4m3"), s_h=(s_h, "f32"))
    _layout(q_a, "q_a", (T, K))
    _span(s_a, "s_a", T, Kb, ssm, sskb, 4)
    _layout(w, "w", (G, 2 * I, K))
    _grid_span(w_scale, "w_scale", _scale_rows(2 * I, [I, I]), Kb, G)
    _layout(offsets, "offsets", (G + 1,))
    _out(q_h, "q_h", T, I, 1)
    _scales_out(s_h, "s_h", T, -(-I // 128), hsm, hskb,
                sh_stride_m is not None or sh_stride_kb is not None)
    wsp, wsb = _ws(workspace)
    _check(_lib.bfp8_grouped_linear_silu_quant(_ptr(q_a), _ptr(s_a), ssm, sskb, _ptr(w),
                                               _ptr(w_scale), _scale_dtype(w_scale),
                                               _ptr(offsets), G, T, I, K, _ptr(q_h),
                                               q_h.stride(0), _ptr(s_h), hsm, hskb, wsp, wsb,
                                               _stream(stream)),
           "bfp8_grouped_linear_silu_quant")


BFP8_DECODE_W8A16, BFP8_DECODE_W8A8 = 0, 1


def bfp8_decode_ffn_workspace(M: int, H: int, I: int, arith: int = BFP8_DECODE_W8A16) -> int:
    return int(_lib.bfp8_decode_ffn_workspace(M, H, I, arith))


def bfp8_decode_ffn(x, w_gate_up, s_gate_up, w_down, s_down, y, workspace,
                    arith: int = BFP8_DECODE_W8A16, stream=None) -> None:
    """One dense-FFN decode step: gate/up GEMV -> SiLU*up -> down GEMV."""
    M, H = x.shape
    I = w_down.shape[1]
    Hb, Ib = -(-H // 128), -(-I // 128)
    _dtypes(x=(x, "bf16"), w_gate_up=(w_gate_up, "e4m3"), w_down=(w_down, "e4m3"),
            y=(y, "bf16"))
    _rows(x, "x")
    _span(x, "x", M, H, x.stride(0), 1, 2)
    _layout(w_gate_up, "w_gate_up", (2 * I, H))
    _grid_span(s_gate_up, "s_gate_up", 2 * Ib, Hb)
    _layout(w_down, "w_down", (H, I))
    _grid_span(s_down, "s_down", Hb, Ib)
    _out(y, "y", M, H, 2)
    # the library takes one scale dtype code for both grids
    sdt = _scale_dtype(s_gate_up)
    if _scale_dtype(s_down) != sdt:
        raise ValueError("bfp8: s_gate_up and s_down must have the same dtype and kind (both "
                         "block grids or both one multiplier): the call reads both with one "
                         f"scale dtype, got {s_gate_up.dtype} rank {s_gate_up.dim()} and "
                         f"{s_down.dtype} rank {s_down.dim()}")
    _check(_lib.bfp8_decode_ffn(arith, _ptr(x), x.stride(0), _ptr(w_gate_up), _ptr(s_gate_up),
                                _ptr(w_down), _ptr(s_down), sdt, M, H, I,
                                _ptr(y), y.stride(0), *_ws(workspace),
                                _stream(stream)),
           "bfp8_decode_ffn")


def bfp8_moe_gather_act_quant(x, row_token, q, scales, s_stride_m=None, s_stride_kb=None,
                              stream=None) -> None:
    """q[r], scales[r] = 1x128 quantization of x[row_token[r]] (int32 on the device)."""
    T, H = x.shape
    R = row_token.shape[0]
    ssm = scales.stride(0) if s_stride_m is None else s_stride_m
    sskb = scales.stride(1) if s_stride_kb is None else s_stride_kb
    _dtypes(x=(x, "bf16"), row_token=(row_token, "i32"), q=(q, "e4m3"), scales=(scales, "f32"))
    _rows(x, "x")
    _span(x, "x", T, H, x.stride(0), 1, 2)
    _layout(row_token, "row_token", (R,))
    _out(q, "q", R, H, 1)
    _scales_out(scales, "scales", R, -(-H // 128), ssm, sskb,
                s_stride_m is not None or s_stride_kb is not None)
    _check(_lib.bfp8_moe_gather_act_quant(_ptr(x), T, H, x.stride(0), _ptr(row_token), R, _ptr(q),
                                          q.stride(0), _ptr(scales), ssm, sskb, _stream(stream)),
           "bfp8_moe_gather_act_quant")


def bfp8_moe_combine(y, token_rows, token_weights, out, stream=None) -> None:
    """out[t] = bf16(sum_j token_weights[t, j] * y[token_rows[t, j]]), slot order j."""
    R, H = y.shape
    T, topk = token_rows.shape
    _dtypes(y=(y, "bf16"), token_rows=(token_rows, "i32"), token_weights=(token_weights, "f32"),
            out=(out, "bf16"))
    _rows(y, "y")
    _span(y, "y", R, H, y.stride(0), 1, 2)
    _layout(token_rows, "token_rows", (T, topk))
    _layout(token_weights, "token_weights", (T, topk))
    _out(out, "out", T, H, 2)
    _check(_lib.bfp8_moe_combine(_ptr(y), R, H, y.stride(0), _ptr(token_rows),
                                 _ptr(token_weights), T, topk, _ptr(out), out.stride(0),
                                 _stream(stream)),
           "bfp8_moe_combine")


def bfp8_device_status(stream=None) -> int:
    return int(_lib.bfp8_device_status(_stream(stream)))


def bfp8_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch the bounded-wait self-test (a barrier whose second arrival never
    comes); the next bfp8_device_status() reports the timeout."""
    _check(_lib.bfp8_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "bfp8_selftest_wait_timeout")
