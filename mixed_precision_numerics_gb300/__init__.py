"""GB300 mixed-precision hot path: Python binding of libmpnum.so.

The functions below carry the C entry points' names and only marshal
arguments (tensor data pointers, the current CUDA stream, host structs); every
step of the computation runs in the library's CUDA kernels.  Importing this
package fails loudly when ``libmpnum.so`` has not been built: there is no
other implementation to fall back to.

PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmpnum.so")

MP_OK, MP_EINVAL, MP_EALIGN, MP_ESHAPE, MP_EWORKSPACE, MP_ECUDA = 0, -1, -2, -3, -4, -5
MP_F32, MP_F16, MP_BF16, MP_E4M3, MP_E5M2, MP_E2M1, MP_E2M3, MP_E3M2 = 0, 1, 2, 3, 4, 5, 6, 7


class MpParam(ctypes.Structure):
    _fields_ = [
        ("master", ctypes.c_void_p),
        ("exp_avg", ctypes.c_void_p),
        ("exp_avg_sq", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("working", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
    ]


class AdamwHparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")]


class ScalerState(ctypes.Structure):
    _fields_ = [
        ("scale", ctypes.c_float),
        ("growth_tracker", ctypes.c_int32),
        ("found_inf", ctypes.c_int32),
        ("error_flags", ctypes.c_int32),
        ("step", ctypes.c_int64),
        ("beta1_pow", ctypes.c_double),
        ("beta2_pow", ctypes.c_double),
        ("skipped", ctypes.c_int64),
        ("grad_norm", ctypes.c_float),
        ("clip_coef", ctypes.c_float),
        ("internal_found", ctypes.c_uint32),
        ("internal_ticket", ctypes.c_uint32),
        ("internal_scalars", ctypes.c_float * 6),
    ]


class ScalerCfg(ctypes.Structure):
    _fields_ = [
        ("growth_factor", ctypes.c_float),
        ("backoff_factor", ctypes.c_float),
        ("growth_interval", ctypes.c_int32),
        ("enabled", ctypes.c_int32),
    ]


class Fp8Meta(ctypes.Structure):
    _fields_ = [
        ("scale", ctypes.c_float),
        ("scale_inv", ctypes.c_float),
        ("amax", ctypes.c_float),
        ("pos", ctypes.c_int32),
        ("internal_amax", ctypes.c_uint32),
        ("internal_ticket", ctypes.c_uint32),
        ("internal_hrest", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
    ]


assert ctypes.sizeof(ScalerState) == 88 and ctypes.sizeof(Fp8Meta) == 32 and ctypes.sizeof(MpParam) == 48


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc, sm_103a). There is no fallback implementation."
        )
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, U16, U64, F, S = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint16,
                                   ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t)
    sig = {
        "mp_status_str": (ctypes.c_char_p, [I32]),
        "mp_version": (I32, []),
        "mp_launch_count": (U64, []),
        "mp_wait_failures": (I32, [P]),
        "mp_scaler_state_init": (None, [P, F]),
        "mp_fp8_meta_init": (None, [P]),
        "mp_adamw_workspace_size": (S, [P, I32]),
        "mp_adamw_step": (I32, [P, I32, I32, I32, P, P, P, S, P]),
        "mp_adamw_check": (I32, [P, I32, I32, P, P, P, S, P]),
        "mp_adamw_apply": (I32, [P, I32, I32, I32, P, P, P]),
        "loss_scale_update": (I32, [P, P, P]),
        "fp8_cast_delayed": (I32, [P, I32, I64, P, I32, P, P, I32, F, I32, P]),
        "fp8_cast_transpose_delayed": (I32, [P, I32, I64, I64, P, P, I32, P, P, I32, F, I32, P]),
        "fp8_cast_delayed_count": (I32, [P, I32, I64, P, I32, P, P, I32, F, I32, P, P]),
        "fp8_quantize_blockwise": (I32, [P, I32, I64, I64, I32, I32, P, I32, P, P]),
        "nvfp4_workspace_size": (S, []),
        "nvfp4_quantize": (I32, [P, I64, I64, I32, I32, U64, I32, U16, P, P, P, P, P, P, S, P]),
        "rht16": (I32, [P, I64, I64, U16, P, I32, P]),
        "e2m1_stochastic_round": (I32, [P, P, I64, P, P]),
        "nvfp4_noalloc_scratch_bytes": (S, []),
        "nvfp4_quantize_noalloc": (I32, [P, I64, I64, I32, I32, U64, I32, U16, P, P, P, P, P, P]),
        "mx_quantize": (I32, [P, I32, I64, I64, I32, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


lib = _load()


class MpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {lib.mp_status_str(status).decode()} (status {status})")
        self.status = status


def _check(fn: str, status: int) -> None:
    if status != MP_OK:
        raise MpError(fn, status)


def _dev(t, name: str, nbytes: int = 0, like=None, align: int = 16) -> None:
    """Checks a tensor before its pointer crosses the C ABI, which cannot tell
    host from device memory: it must live on the CUDA device the call runs on
    (the current device, or that of `like`), be contiguous, and hold at least
    `nbytes`.  The size is not checked when the pointer breaks the argument's
    alignment rule (`align` bytes): the library reports that itself, before
    any launch.  Raw integer pointers and None pass unchecked."""
    if t is None or isinstance(t, int):
        return
    import torch

    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name}: a CUDA tensor is required (the kernels read and write device memory)")
    want = like.device if like is not None and not isinstance(like, int) else torch.device(
        "cuda", torch.cuda.current_device())
    if t.device != want:
        raise ValueError(f"{name}: on {t.device}, the call runs on {want}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: a contiguous tensor is required")
    have = t.numel() * t.element_size()
    if t.data_ptr() % align == 0 and have < nbytes:
        raise ValueError(f"{name}: {have} bytes, the call needs {nbytes}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch

    return {torch.float32: MP_F32, torch.float16: MP_F16, torch.bfloat16: MP_BF16}[t.dtype]


def mp_status_str(status: int) -> str:
    return lib.mp_status_str(status).decode()


def mp_launch_count() -> int:
    return int(lib.mp_launch_count())


def mp_wait_failures() -> int:
    """Bounded tile-copy waits that gave up in the library's FP8 kernels (0 normally)."""
    out = ctypes.c_uint32(0)
    _check("mp_wait_failures", lib.mp_wait_failures(ctypes.byref(out)))
    return int(out.value)


def nvfp4_workspace_size() -> int:
    return int(lib.nvfp4_workspace_size())


# ---- state helpers ------------------------------------------------------------------


def scaler_state_bytes(init_scale: float = 65536.0) -> bytes:
    st = ScalerState()
    lib.mp_scaler_state_init(ctypes.byref(st), float(init_scale))
    return bytes(st)


def fp8_meta_bytes() -> bytes:
    m = Fp8Meta()
    lib.mp_fp8_meta_init(ctypes.byref(m))
    return bytes(m)


def new_scaler_state(init_scale: float = 65536.0, device="cuda"):
    """Device buffer (uint8[88]) holding an initialised mp_scaler_state."""
    import torch

    return torch.frombuffer(bytearray(scaler_state_bytes(init_scale)), dtype=torch.uint8).to(device)


def new_fp8_meta(device="cuda"):
    import torch

    return torch.frombuffer(bytearray(fp8_meta_bytes()), dtype=torch.uint8).to(device)


def new_nvfp4_workspace(device="cuda"):
    import torch

    return torch.zeros(nvfp4_workspace_size(), dtype=torch.uint8, device=device)


def read_scaler_state(t) -> ScalerState:
    return ScalerState.from_buffer_copy(t.cpu().numpy().tobytes())


def read_fp8_meta(t) -> Fp8Meta:
    return Fp8Meta.from_buffer_copy(t.cpu().numpy().tobytes())


# ---- entry points ---------------------------------------------------------------------


@dataclass
class Param:
    """One parameter tensor of the step (torch CUDA tensors, contiguous)."""

    master: object
    exp_avg: object
    exp_avg_sq: object
    grad: object
    working: object


def make_param_array(params: Sequence[Param]):
    for i, p in enumerate(params):
        n = p.master.numel() if not isinstance(p.master, int) else 0
        ref = params[0].master
        for name, t, es in (("master", p.master, 4), ("exp_avg", p.exp_avg, 4), ("exp_avg_sq", p.exp_avg_sq, 4),
                            ("grad", p.grad, 2), ("working", p.working, 2)):
            _dev(t, f"params[{i}].{name}", n * es, like=ref)
    arr = (MpParam * max(1, len(params)))()
    for i, p in enumerate(params):
        arr[i] = MpParam(_ptr(p.master), _ptr(p.exp_avg), _ptr(p.exp_avg_sq), _ptr(p.grad), _ptr(p.working),
                         p.master.numel())
    return arr


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def mp_adamw_workspace_size(params) -> int:
    arr = params if isinstance(params, ctypes.Array) else make_param_array(params)
    return int(lib.mp_adamw_workspace_size(arr, len(params)))


def mp_adamw_step(params, hp: AdamwHparams, state, grad_dtype: int | None = None,
                  working_dtype: int | None = None, workspace=None, stream=None) -> None:
    """params: a sequence of Param, or a prebuilt ctypes MpParam array (then give
    dtypes).  workspace: device buffer of mp_adamw_workspace_size bytes, needed
    only when hp.max_grad_norm > 0."""
    arr, n, g, w = _marshal(params, grad_dtype, working_dtype)
    _dev(state, "state", ctypes.sizeof(ScalerState), align=8)
    _dev(workspace, "workspace", align=8)
    wp, wb = _ws(workspace)
    _check("mp_adamw_step", lib.mp_adamw_step(arr, n, g, w, ctypes.byref(hp), _ptr(state), wp, wb, _stream(stream)))


def _marshal(params, grad_dtype, working_dtype):
    if isinstance(params, ctypes.Array):
        if grad_dtype is None or working_dtype is None:
            raise ValueError("a prebuilt parameter array needs grad_dtype and working_dtype")
        return params, len(params), grad_dtype, working_dtype
    n = len(params)
    arr = make_param_array(params)
    if grad_dtype is None:
        grad_dtype = _dtype_code(params[0].grad) if n else MP_F16
    if working_dtype is None:
        working_dtype = _dtype_code(params[0].working) if n else MP_F16
    return arr, n, grad_dtype, working_dtype


def mp_adamw_check(params, hp: AdamwHparams, state, grad_dtype: int | None = None, workspace=None,
                   stream=None) -> None:
    arr, n, g, _ = _marshal(params, grad_dtype, MP_F16 if grad_dtype is not None else None)
    _dev(state, "state", ctypes.sizeof(ScalerState), align=8)
    _dev(workspace, "workspace", align=8)
    wp, wb = _ws(workspace)
    _check("mp_adamw_check", lib.mp_adamw_check(arr, n, g, ctypes.byref(hp), _ptr(state), wp, wb, _stream(stream)))


def mp_adamw_apply(params, hp: AdamwHparams, state, grad_dtype: int | None = None,
                   working_dtype: int | None = None, stream=None) -> None:
    arr, n, g, w = _marshal(params, grad_dtype, working_dtype)
    _dev(state, "state", ctypes.sizeof(ScalerState), align=8)
    _check("mp_adamw_apply", lib.mp_adamw_apply(arr, n, g, w, ctypes.byref(hp), _ptr(state), _stream(stream)))


def loss_scale_update(state, cfg: ScalerCfg, stream=None) -> None:
    _dev(state, "state", ctypes.sizeof(ScalerState), align=8)
    _check("loss_scale_update", lib.loss_scale_update(_ptr(state), ctypes.byref(cfg), _stream(stream)))


MP_AMAX_HISTORY_MAX, MP_AMAX_MOST_RECENT = 0, 1


def fp8_cast_delayed(x, y, fp8_dtype: int, meta, history, margin: float = 1.0, stream=None,
                     n: int | None = None, amax_algo: int = MP_AMAX_HISTORY_MAX) -> None:
    """y: uint8 (or float8) tensor with x.numel() elements; history: float32 device tensor."""
    ne = x.numel() if n is None else n
    _fp8_args(x, y, ne, meta, history)
    _check("fp8_cast_delayed",
           lib.fp8_cast_delayed(_ptr(x), _dtype_code(x), x.numel() if n is None else n, _ptr(y), fp8_dtype,
                                _ptr(meta), _ptr(history), history.numel(), float(margin), amax_algo,
                                _stream(stream)))


def _fp8_args(x, y, n, meta, history, y_t=None):
    if isinstance(x, int):
        return
    _dev(x, "x", n * x.element_size())
    _dev(y, "y", n, like=x)
    _dev(y_t, "y_t", n, like=x)
    _dev(meta, "meta", ctypes.sizeof(Fp8Meta), like=x)
    _dev(history, "history", 4, like=x, align=4)


def fp8_cast_delayed_count(x, y, fp8_dtype: int, meta, history, saturated, margin: float = 1.0,
                           amax_algo: int = MP_AMAX_HISTORY_MAX, stream=None) -> None:
    """fp8_cast_delayed that also adds the number of saturated elements to
    `saturated` (an int64 device tensor of one element)."""
    _fp8_args(x, y, x.numel(), meta, history)
    _dev(saturated, "saturated", 8, like=x, align=8)
    _check("fp8_cast_delayed_count",
           lib.fp8_cast_delayed_count(_ptr(x), _dtype_code(x), x.numel(), _ptr(y), fp8_dtype, _ptr(meta),
                                      _ptr(history), history.numel(), float(margin), amax_algo, _ptr(saturated),
                                      _stream(stream)))


def fp8_cast_transpose_delayed(x, y, y_t, fp8_dtype: int, meta, history, margin: float = 1.0,
                               amax_algo: int = MP_AMAX_HISTORY_MAX, stream=None) -> None:
    """x: [rows, cols]; y: rows*cols bytes; y_t: cols*rows bytes (the transpose)."""
    rows, cols = x.shape
    _fp8_args(x, y, rows * cols, meta, history, y_t)
    _check("fp8_cast_transpose_delayed",
           lib.fp8_cast_transpose_delayed(_ptr(x), _dtype_code(x), rows, cols, _ptr(y), _ptr(y_t), fp8_dtype,
                                          _ptr(meta), _ptr(history), history.numel(), float(margin), amax_algo,
                                          _stream(stream)))


def fp8_quantize_blockwise(x, y, scales, block_rows: int = 1, block_cols: int = 128, fp8_dtype: int = MP_E4M3,
                           stream=None) -> None:
    """x: [rows, cols]; y: rows*cols bytes; scales: float32 [ceil(rows/br), ceil(cols/bc)]."""
    rows, cols = x.shape
    _dev(x, "x", rows * cols * x.element_size())
    _dev(y, "y", rows * cols, like=x)
    if (block_rows, block_cols) in ((1, 128), (128, 128)):
        _dev(scales, "scales", 4 * (-(-rows // block_rows)) * (-(-cols // block_cols)), like=x, align=4)
    else:
        _dev(scales, "scales", like=x, align=4)
    _check("fp8_quantize_blockwise",
           lib.fp8_quantize_blockwise(_ptr(x), _dtype_code(x), rows, cols, block_rows, block_cols, _ptr(y), fp8_dtype,
                                      _ptr(scales), _stream(stream)))


def _nvfp4_args(x, codes, block_scales, tensor_scale, nonfinite, dequant, rows, cols, block_2d):
    n = rows * cols
    _dev(x, "x", 2 * n)
    _dev(codes, "codes", n // 2, like=x)
    shape_ok = cols % 16 == 0 and (not block_2d or rows % 16 == 0)
    _dev(block_scales, "block_scales", ((rows // 16 if block_2d else rows) * (cols // 16)) if shape_ok else 0,
         like=x, align=1)
    _dev(tensor_scale, "tensor_scale", 4, like=x, align=4)
    _dev(nonfinite, "nonfinite", 4, like=x, align=4)
    _dev(dequant, "dequant", 2 * n, like=x)


def nvfp4_quantize(x, codes, block_scales, tensor_scale, nonfinite, workspace, *, block_2d: bool = False,
                   stochastic: bool = False, seed: int = 0, apply_rht: bool = False, sign_mask: int = 0,
                   dequant=None, rows: int | None = None, cols: int | None = None, stream=None) -> None:
    if rows is None:
        rows, cols = x.shape
    _nvfp4_args(x, codes, block_scales, tensor_scale, nonfinite, dequant, rows, cols, block_2d)
    _dev(workspace, "workspace", like=x, align=8)
    _check("nvfp4_quantize",
           lib.nvfp4_quantize(_ptr(x), rows, cols, int(block_2d), int(stochastic), seed & (2**64 - 1),
                              int(apply_rht), sign_mask & 0xFFFF, _ptr(codes), _ptr(block_scales),
                              _ptr(tensor_scale), _ptr(nonfinite), _ptr(dequant), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)))


def nvfp4_quantize_noalloc(x, codes, block_scales, tensor_scale, nonfinite, *, block_2d: bool = False,
                           stochastic: bool = False, seed: int = 0, apply_rht: bool = False, sign_mask: int = 0,
                           dequant=None, rows: int | None = None, cols: int | None = None, stream=None) -> None:
    """nvfp4_quantize for callers that cannot allocate a workspace: the
    library's own fixed device scratch is used instead (calls that overlap
    on the GPU race on it; see the C header)."""
    if rows is None:
        rows, cols = x.shape
    _nvfp4_args(x, codes, block_scales, tensor_scale, nonfinite, dequant, rows, cols, block_2d)
    _check("nvfp4_quantize_noalloc",
           lib.nvfp4_quantize_noalloc(_ptr(x), rows, cols, int(block_2d), int(stochastic), seed & (2**64 - 1),
                                      int(apply_rht), sign_mask & 0xFFFF, _ptr(codes), _ptr(block_scales),
                                      _ptr(tensor_scale), _ptr(nonfinite), _ptr(dequant), _stream(stream)))


def rht16(x, y, sign_mask: int, stream=None) -> None:
    rows, cols = x.shape
    _dev(x, "x", 2 * rows * cols)
    if not isinstance(y, int):
        _dev(y, "y", rows * cols * y.element_size(), like=x)
    _check("rht16", lib.rht16(_ptr(x), rows, cols, sign_mask & 0xFFFF, _ptr(y), _dtype_code(y), _stream(stream)))


def e2m1_stochastic_round(y, r16, codes, stream=None) -> None:
    """y: FP32 [n]; r16: 16-bit [n] random values (int16 or uint16 storage);
    codes: uint8 [(n + 1) // 2], element 2j in the low nibble of byte j."""
    n = y.numel()
    _dev(y, "y", 4 * n)
    _dev(r16, "r16", 2 * n, like=y)
    _dev(codes, "codes", (n + 1) // 2, like=y)
    _check("e2m1_stochastic_round", lib.e2m1_stochastic_round(_ptr(y), _ptr(r16), n, _ptr(codes), _stream(stream)))


def mx_quantize(x, codes, scales, elem_dtype: int = MP_E2M1, dequant=None, stream=None) -> None:
    """x: [rows, cols], cols % 32 == 0; codes: rows*cols bytes (FP8, FP6) or
    rows*cols/2 (E2M1); scales: uint8 [rows, cols/32] (UE8M0)."""
    rows, cols = x.shape
    n = rows * cols
    ok = cols % 32 == 0 and elem_dtype in (MP_E4M3, MP_E5M2, MP_E2M1, MP_E2M3, MP_E3M2)  # else the library says why
    _dev(x, "x", n * x.element_size())
    _dev(codes, "codes", (n // 2 if elem_dtype == MP_E2M1 else n) if ok else 0, like=x)
    _dev(scales, "scales", n // 32 if ok else 0, like=x, align=1)
    _dev(dequant, "dequant", 2 * n if ok else 0, like=x)
    _check("mx_quantize", lib.mx_quantize(_ptr(x), _dtype_code(x), rows, cols, elem_dtype, _ptr(codes),
                                          _ptr(scales), _ptr(dequant), _stream(stream)))


__all__ = [
    "AdamwHparams", "Fp8Meta", "MpError", "MpParam", "Param", "ScalerCfg", "ScalerState",
    "MP_F32", "MP_F16", "MP_BF16", "MP_E4M3", "MP_E5M2", "MP_E2M1", "MP_E2M3", "MP_E3M2", "mx_quantize",
    "mp_adamw_step", "mp_adamw_check", "mp_adamw_apply", "mp_adamw_workspace_size", "loss_scale_update",
    "fp8_cast_transpose_delayed", "fp8_cast_delayed_count", "fp8_quantize_blockwise", "MP_AMAX_HISTORY_MAX", "MP_AMAX_MOST_RECENT",
    "nvfp4_quantize_noalloc", "fp8_cast_delayed", "nvfp4_quantize", "rht16", "e2m1_stochastic_round",
    "nvfp4_workspace_size", "mp_status_str", "mp_launch_count", "mp_wait_failures",
    "new_scaler_state", "new_fp8_meta", "new_nvfp4_workspace", "read_scaler_state", "read_fp8_meta",
    "make_param_array",
]
