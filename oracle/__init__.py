"""CPU oracle for the mixed-precision hot path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg import this package.  It loads ``liboracle.so``, a plain scalar C
build of ``oracle.c``; nothing here is shared with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16, E4M3, E5M2, E2M1, E2M3, E3M2 = 0, 1, 2, 3, 4, 5, 6, 7

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class AdamwHp(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")]


class ScalerState(ctypes.Structure):
    _fields_ = [
        ("scale", ctypes.c_float),
        ("growth_tracker", ctypes.c_int32),
        ("found_inf", ctypes.c_int32),
        ("pad0", ctypes.c_int32),
        ("step", ctypes.c_int64),
        ("beta1_pow", ctypes.c_double),
        ("beta2_pow", ctypes.c_double),
        ("skipped", ctypes.c_int64),
    ]


class ScalerCfg(ctypes.Structure):
    _fields_ = [
        ("growth_factor", ctypes.c_float),
        ("backoff_factor", ctypes.c_float),
        ("growth_interval", ctypes.c_int32),
        ("enabled", ctypes.c_int32),
    ]


class StepScalars(ctypes.Structure):
    _fields_ = [
        (n, ctypes.c_float)
        for n in ("inv_scale", "step_size", "bc2_sqrt", "decay", "omb1", "omb2", "beta1", "beta2", "eps", "clip")
    ]


class Fp8Meta(ctypes.Structure):
    _fields_ = [
        ("scale", ctypes.c_float),
        ("scale_inv", ctypes.c_float),
        ("amax", ctypes.c_float),
        ("pos", ctypes.c_int32),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I64, I32, U8, U16, U32, U64, F = (
            ctypes.c_void_p,
            ctypes.c_int64,
            ctypes.c_int32,
            ctypes.c_uint8,
            ctypes.c_uint16,
            ctypes.c_uint32,
            ctypes.c_uint64,
            ctypes.c_float,
        )
        sig = {
            "orc_f32_to_f16": (U16, [F]),
            "orc_f16_to_f32": (F, [U16]),
            "orc_f32_to_bf16": (U16, [F]),
            "orc_bf16_to_f32": (F, [U16]),
            "orc_f32_to_fp8_sat": (U8, [F, ctypes.c_int]),
            "orc_fp8_to_f32": (F, [U8, ctypes.c_int]),
            "orc_f32_to_e2m1": (U8, [F]),
            "orc_f32_to_e2m1_sr": (U8, [F, U32]),
            "orc_e2m1_to_f32": (F, [U8]),
            "orc_convert": (None, [P, ctypes.c_int, I64, P, ctypes.c_int]),
            "orc_amax": (F, [P, ctypes.c_int, I64]),
            "orc_philox4x32_10": (None, [P, P, P]),
            "orc_sr_bits": (U32, [U64, U64]),
            "orc_e2m1_sr_array": (None, [P, I64, U64, U64, P]),
            "orc_e2m1_sr_bits_array": (None, [P, P, I64, P]),
            "orc_rht16_tile": (None, [P, U16, P]),
            "orc_rht16": (ctypes.c_int, [P, I64, I64, U16, P, ctypes.c_int]),
            "orc_nonfinite_any": (ctypes.c_int, [P, ctypes.c_int, I64]),
            "orc_adamw_begin": (None, [P, P, ctypes.c_int, P]),
            "orc_adamw_apply": (None, [P, P, P, P, P, ctypes.c_int, P, ctypes.c_int, I64]),
            "orc_loss_scale_update": (None, [P, P]),
            "orc_grad_sumsq": (ctypes.c_double, [P, ctypes.c_int, I64, F]),
            "orc_clip_coef": (F, [ctypes.c_double, F]),
            "orc_fp8_cast_one": (U8, [F, F, ctypes.c_int]),
            "orc_fp8_cast_array": (None, [P, ctypes.c_int, I64, P, ctypes.c_int, F]),
            "orc_fp8_history_update": (None, [P, P, I32, F, F, ctypes.c_int, ctypes.c_int]),
            "orc_fp8_cast_delayed": (None, [P, ctypes.c_int, I64, P, ctypes.c_int, P, P, I32, F, ctypes.c_int]),
            "orc_transpose_u8": (None, [P, I64, I64, P]),
            "orc_fp8_quantize_blockwise": (None, [P, ctypes.c_int, I64, I64, I32, I32, ctypes.c_int, P, P]),
            "orc_mx_quantize": (None, [P, ctypes.c_int, I64, I64, ctypes.c_int, P, P, P]),
            "orc_fp8_saturation_count": (I64, [P, ctypes.c_int, I64, ctypes.c_int, ctypes.c_float]),
            "orc_nvfp4_prepare": (ctypes.c_int, [P, I64, I64, ctypes.c_int, U16, P]),
            "orc_nvfp4_tensor_scale": (F, [F, P]),
            "orc_nvfp4_encode_rows": (
                None,
                [P, I64, I64, I64, ctypes.c_int, ctypes.c_int, U64, F, I32, P, P, P],
            ),
            "orc_nvfp4_quantize": (
                ctypes.c_int,
                [P, I64, I64, ctypes.c_int, ctypes.c_int, U64, ctypes.c_int, U16, P, P, P, P, P],
            ),
            "orc_nvfp4_block_scale": (None, [F, F, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


_NP = {F32: np.float32, F16: np.uint16, BF16: np.uint16, E4M3: np.uint8, E5M2: np.uint8, E2M1: np.uint8,
       E2M3: np.uint8, E3M2: np.uint8}


def convert(x: np.ndarray, in_fmt: int, out_fmt: int) -> np.ndarray:
    """Element-wise format conversion (bit patterns for the narrow formats)."""
    x = np.ascontiguousarray(x, dtype=_NP[in_fmt])
    out = np.empty(x.shape, dtype=_NP[out_fmt])
    lib().orc_convert(_p(x), in_fmt, x.size, _p(out), out_fmt)
    return out


def amax(x: np.ndarray, fmt: int) -> float:
    x = np.ascontiguousarray(x, dtype=_NP[fmt])
    return float(np.float32(lib().orc_amax(_p(x), fmt, x.size)))


def amax_f32_bits(x: np.ndarray, fmt: int) -> int:
    return int(np.array([amax(x, fmt)], dtype=np.float32).view(np.uint32)[0])


def philox(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.empty(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_bits(seed: int, idx) -> np.ndarray:
    L = lib()
    return np.array([L.orc_sr_bits(seed, int(i)) for i in np.asarray(idx).ravel()], dtype=np.uint32)


def e2m1_sr_array(y: np.ndarray, seed: int, i0: int = 0) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.size, dtype=np.uint8)
    lib().orc_e2m1_sr_array(_p(y), y.size, seed, i0, _p(out))
    return out


def e2m1_sr_with_bits(y: np.ndarray, r16: np.ndarray) -> np.ndarray:
    """Stochastic E2M1 code of each y[k] with the 16 random bits r16[k] (one code per byte)."""
    y = np.ascontiguousarray(y, dtype=np.float32).reshape(-1)
    r16 = np.ascontiguousarray(r16, dtype=np.uint16).reshape(-1)
    assert y.size == r16.size
    out = np.empty(y.size, dtype=np.uint8)
    lib().orc_e2m1_sr_bits_array(_p(y), _p(r16), y.size, _p(out))
    return out


def rht16(x_bf16: np.ndarray, sign_mask: int, out_fmt: int = F32) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    y = np.empty((rows, cols), dtype=_NP[out_fmt])
    rc = lib().orc_rht16(_p(x), rows, cols, sign_mask, _p(y), out_fmt)
    if rc:
        raise ValueError("cols must be a multiple of 16")
    return y


def rht16_tile(v: np.ndarray, sign_mask: int) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(16, dtype=np.float32)
    lib().orc_rht16_tile(_p(a), sign_mask, _p(out))
    return out


# --- optimizer ----------------------------------------------------------------


def new_scaler_state(scale: float = 65536.0) -> ScalerState:
    return ScalerState(scale, 0, 0, 0, 0, 1.0, 1.0, 0)


def nonfinite_any(g: np.ndarray, fmt: int) -> int:
    g = np.ascontiguousarray(g, dtype=np.uint16)
    return int(lib().orc_nonfinite_any(_p(g), fmt, g.size))


def adamw_begin(hp: AdamwHp, st: ScalerState, found_inf: int) -> StepScalars:
    s = StepScalars()
    lib().orc_adamw_begin(ctypes.byref(hp), ctypes.byref(st), int(found_inf), ctypes.byref(s))
    return s


def adamw_apply(s: StepScalars, w, m, v, g, g_fmt: int, w16, w16_fmt: int) -> None:
    """In place on numpy arrays w, m, v (float32) and w16 (uint16)."""
    for a, dt in ((w, np.float32), (m, np.float32), (v, np.float32), (g, np.uint16), (w16, np.uint16)):
        assert a.dtype == dt and a.flags["C_CONTIGUOUS"]
    lib().orc_adamw_apply(ctypes.byref(s), _p(w), _p(m), _p(v), _p(g), g_fmt, _p(w16), w16_fmt, w.size)


def loss_scale_update(st: ScalerState, cfg: ScalerCfg) -> None:
    lib().orc_loss_scale_update(ctypes.byref(st), ctypes.byref(cfg))


# --- FP8 delayed scaling -------------------------------------------------------


def new_fp8_meta() -> Fp8Meta:
    return Fp8Meta(1.0, 1.0, 0.0, 0)


def fp8_cast_array(x: np.ndarray, x_fmt: int, fmt: int, scale: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=_NP[x_fmt])
    y = np.empty(x.shape, dtype=np.uint8)
    lib().orc_fp8_cast_array(_p(x), x_fmt, x.size, _p(y), fmt, np.float32(scale))
    return y


def fp8_saturation_count(x: np.ndarray, x_fmt: int, fmt: int, scale: float) -> int:
    x = np.ascontiguousarray(x, dtype=_NP[x_fmt])
    return int(lib().orc_fp8_saturation_count(_p(x), x_fmt, x.size, fmt, np.float32(scale)))


AMAX_HISTORY_MAX, AMAX_MOST_RECENT = 0, 1


def fp8_history_update(meta: Fp8Meta, history: np.ndarray, margin: float, amax_v: float, fmt: int,
                       amax_algo: int = AMAX_HISTORY_MAX) -> None:
    assert history.dtype == np.float32
    lib().orc_fp8_history_update(
        ctypes.byref(meta), _p(history), history.size, np.float32(margin), np.float32(amax_v), fmt, amax_algo
    )


def fp8_cast_delayed(x: np.ndarray, x_fmt: int, fmt: int, meta: Fp8Meta, history: np.ndarray, margin: float,
                     amax_algo: int = AMAX_HISTORY_MAX):
    x = np.ascontiguousarray(x, dtype=_NP[x_fmt])
    y = np.empty(x.shape, dtype=np.uint8)
    lib().orc_fp8_cast_delayed(
        _p(x), x_fmt, x.size, _p(y), fmt, ctypes.byref(meta), _p(history), history.size, np.float32(margin),
        amax_algo
    )
    return y


def fp8_quantize_blockwise(x: np.ndarray, x_fmt: int, block_rows: int, block_cols: int, fmt: int = E4M3):
    """Returns (y [rows, cols] u8, scales [ceil(rows/br), ceil(cols/bc)] f32)."""
    x = np.ascontiguousarray(x, dtype=_NP[x_fmt])
    rows, cols = x.shape
    y = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty((-(-rows // block_rows), -(-cols // block_cols)), dtype=np.float32)
    lib().orc_fp8_quantize_blockwise(_p(x), x_fmt, rows, cols, block_rows, block_cols, fmt, _p(y), _p(sc))
    return y, sc


def mx_quantize(x: np.ndarray, x_fmt: int, elem_fmt: int, want_dequant: bool = True):
    """Returns (codes, scales [rows, cols/32] u8 UE8M0, dequant u16 | None)."""
    x = np.ascontiguousarray(x, dtype=_NP[x_fmt])
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2 if elem_fmt == E2M1 else cols), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    dq = np.zeros((rows, cols), dtype=np.uint16) if want_dequant else None
    lib().orc_mx_quantize(_p(x), x_fmt, rows, cols, elem_fmt, _p(codes), _p(scales), _p(dq))
    return codes, scales, dq


def transpose_u8(y: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.uint8)
    rows, cols = y.shape
    out = np.empty((cols, rows), dtype=np.uint8)
    lib().orc_transpose_u8(_p(y), rows, cols, _p(out))
    return out


# --- NVFP4 -----------------------------------------------------------------------


def nvfp4_quantize(
    x_bf16: np.ndarray,
    block_2d: bool,
    stochastic: bool,
    seed: int = 0,
    apply_rht: bool = False,
    sign_mask: int = 0,
    want_dequant: bool = True,
):
    """Returns (codes [rows, cols/2] u8, scales u8, tensor_scale f32, nonfinite, dequant u16|None)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    if block_2d:
        scales = np.zeros((rows // 16, cols // 16), dtype=np.uint8)
    else:
        scales = np.zeros((rows, cols // 16), dtype=np.uint8)
    ts = np.zeros(1, dtype=np.float32)
    nf = np.zeros(1, dtype=np.int32)
    dq = np.zeros((rows, cols), dtype=np.uint16) if want_dequant else None
    rc = lib().orc_nvfp4_quantize(
        _p(x), rows, cols, int(block_2d), int(stochastic), seed, int(apply_rht), sign_mask,
        _p(codes), _p(scales), _p(ts), _p(nf), _p(dq),
    )
    if rc:
        raise ValueError(f"nvfp4 shape error ({rows}x{cols}, block_2d={block_2d})")
    return codes, scales, float(ts[0]), int(nf[0]), dq


def nvfp4_prepare(x_bf16: np.ndarray, apply_rht: bool, sign_mask: int) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    xp = np.empty((rows, cols), dtype=np.float32)
    if lib().orc_nvfp4_prepare(_p(x), rows, cols, int(apply_rht), sign_mask, _p(xp)):
        raise ValueError("shape")
    return xp


def nvfp4_tensor_scale(amax_v: float):
    nf = np.zeros(1, dtype=np.int32)
    s = lib().orc_nvfp4_tensor_scale(np.float32(amax_v), _p(nf))
    return float(np.float32(s)), int(nf[0])


def nvfp4_encode_rows(xprime_rows: np.ndarray, row0: int, cols: int, block_2d: bool, stochastic: bool,
                      seed: int, s_t: float, nonfinite: int, want_dequant: bool = True):
    """Encode rows [row0, row0+nrows) given x' for exactly those rows.

    Returns codes, scales and dequant for those rows only."""
    xp = np.ascontiguousarray(xprime_rows, dtype=np.float32)
    nrows = xp.shape[0]
    # The C routine indexes outputs by absolute row; give it views offset back.
    codes = np.zeros((nrows, cols // 2), dtype=np.uint8)
    if block_2d:
        scales = np.zeros((nrows // 16, cols // 16), dtype=np.uint8)
    else:
        scales = np.zeros((nrows, cols // 16), dtype=np.uint8)
    dq = np.zeros((nrows, cols), dtype=np.uint16) if want_dequant else None
    base_codes = codes.ctypes.data - row0 * cols // 2
    base_scales = scales.ctypes.data - ((row0 // 16) if block_2d else row0) * (cols // 16)
    base_dq = (dq.ctypes.data - row0 * cols * 2) if want_dequant else None
    lib().orc_nvfp4_encode_rows(
        _p(xp), row0, nrows, cols, int(block_2d), int(stochastic), seed, np.float32(s_t), nonfinite,
        ctypes.c_void_p(base_codes), ctypes.c_void_p(base_scales),
        ctypes.c_void_p(base_dq) if want_dequant else None,
    )
    return codes, scales, dq


def nvfp4_block_scale(bamax: float, s_t: float):
    c = np.zeros(1, dtype=np.uint8)
    d = np.zeros(1, dtype=np.float32)
    r = np.zeros(1, dtype=np.float32)
    lib().orc_nvfp4_block_scale(np.float32(bamax), np.float32(s_t), _p(c), _p(d), _p(r))
    return int(c[0]), float(d[0]), float(r[0])


def grad_sumsq(g: np.ndarray, g_fmt: int, inv_scale: float) -> float:
    """Sum of squares of one tensor's unscaled grads, binary64, element order."""
    g = np.ascontiguousarray(g, dtype=np.uint16)
    return float(lib().orc_grad_sumsq(_p(g), g_fmt, g.size, np.float32(inv_scale)))


def clip_coef(norm: float, max_norm: float) -> float:
    return float(np.float32(lib().orc_clip_coef(float(norm), np.float32(max_norm))))


def grad_norm(grads, g_fmt: int, inv_scale: float) -> float:
    """Global L2 norm of the unscaled grads: the tensors' binary64 sums of
    squares added in list order, then the square root."""
    return norm_of_sumsqs([grad_sumsq(g, g_fmt, inv_scale) for g in grads])


def norm_of_sumsqs(sums) -> float:
    total = 0.0
    for x in sums:
        total = total + x
    return float(np.sqrt(total))


def adamw_step(hp: AdamwHp, st: ScalerState, tensors, g_fmt: int, w16_fmt: int, clip=None):
    """One optimizer step over a list of (w, m, v, g, w16) numpy tensors.

    found_inf is the OR over every grad of the step; when set the step is
    skipped and nothing is written.  With hp.max_grad_norm > 0 the unscaled
    grads are clipped to that global norm.  ``clip``, when given, is the
    binary32 clip coefficient to multiply by in place of the one formed from
    this norm (a test applies a coefficient it has checked separately).
    Returns (found_inf, grad norm or None, clip coefficient of the norm)."""
    found = 0
    for (_, _, _, g, _) in tensors:
        if nonfinite_any(g, g_fmt):
            found = 1
            break
    s = adamw_begin(hp, st, found)
    norm = None
    if hp.max_grad_norm > 0:
        norm = grad_norm([g for (_, _, _, g, _) in tensors], g_fmt, s.inv_scale)
        s.clip = clip_coef(norm, hp.max_grad_norm)
    coef = s.clip
    if clip is not None:
        s.clip = float(np.float32(clip))
    if not found:
        for (w, m, v, g, w16) in tensors:
            adamw_apply(s, w, m, v, g, g_fmt, w16, w16_fmt)
    return found, norm, coef
