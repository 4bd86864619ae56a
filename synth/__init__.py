"""Seeded, counter-based synthetic inputs shared by the tests and the benchmark.

Values are pure functions of (seed, stream, index) (see ``synth.h``), so the
host build (``libsynth_host.so``) and the device build (``libsynth_dev.so``)
produce the same bits, and any element of a full-size tensor can be
regenerated on its own.  This module generates inputs only; it holds none of
the arithmetic of the method under test.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")

F32, F16, BF16 = 0, 1, 2
OUT_NONE, OUT_SCALE, OUT_T3 = 0, 1, 2
_NP = {F32: np.float32, F16: np.uint16, BF16: np.uint16}


class Recipe(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("stream", ctypes.c_uint64),
        ("outlier_stream", ctypes.c_uint64),
        ("sigma", ctypes.c_float),
        ("outlier_mult", ctypes.c_float),
        ("outlier_thr", ctypes.c_uint32),
        ("outlier_kind", ctypes.c_int32),
    ]


def recipe(seed: int, stream: int, sigma: float, outlier_p: float = 0.0, outlier_mult: float = 1.0,
           outlier_kind: int = OUT_NONE, outlier_stream: int | None = None) -> Recipe:
    thr = int(np.floor(outlier_p * 2.0**32)) if outlier_kind != OUT_NONE else 0
    return Recipe(seed, stream, stream if outlier_stream is None else outlier_stream,
                  float(np.float32(sigma)), float(np.float32(outlier_mult)), min(thr, 2**32 - 1),
                  outlier_kind)


def _sources():
    return [os.path.join(_HERE, f) for f in ("synth.h", "synth_host.c", "synth_dev.cu")]


def _stale(target: str) -> bool:
    return not os.path.exists(target) or os.path.getmtime(target) < max(os.path.getmtime(s) for s in _sources())


def build_host(force: bool = False) -> str:
    if force or _stale(HOST_LIB):
        tmp = HOST_LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
                        "-o", tmp, os.path.join(_HERE, "synth_host.c"), "-lpthread", "-lm"], check=True)
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_dev_cmd(out: str = DEV_LIB) -> list[str]:
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-shared",
            "-Xcompiler", "-fPIC", "-o", out, os.path.join(_HERE, "synth_dev.cu")]


def build_dev(force: bool = False) -> str:
    if force or _stale(DEV_LIB):
        tmp = DEV_LIB + f".tmp{os.getpid()}"
        subprocess.run(build_dev_cmd(tmp), check=True)
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


_host = None
_dev = None


def host():
    global _host
    if _host is None:
        L = ctypes.CDLL(build_host())
        L.synth_fill.argtypes = [ctypes.POINTER(Recipe), ctypes.c_int, ctypes.c_uint64, ctypes.c_int64,
                                 ctypes.c_void_p, ctypes.c_int]
        L.synth_fill_at.argtypes = [ctypes.POINTER(Recipe), ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_int]
        L.synth_normal_at.restype = ctypes.c_float
        L.synth_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        L.synth_logf_host.restype = ctypes.c_float
        L.synth_logf_host.argtypes = [ctypes.c_float]
        L.synth_cos2pi_host.restype = ctypes.c_float
        L.synth_cos2pi_host.argtypes = [ctypes.c_float]
        L.synth_hash_host.restype = ctypes.c_uint64
        L.synth_hash_host.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        _host = L
    return _host


def dev():
    global _dev
    if _dev is None:
        L = ctypes.CDLL(build_dev())
        L.synth_fill_dev.restype = ctypes.c_int
        L.synth_fill_dev.argtypes = [ctypes.POINTER(Recipe), ctypes.c_int, ctypes.c_uint64, ctypes.c_int64,
                                     ctypes.c_void_p, ctypes.c_void_p]
        L.synth_fill_at_dev.restype = ctypes.c_int
        L.synth_fill_at_dev.argtypes = [ctypes.POINTER(Recipe), ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p]
        _dev = L
    return _dev


def hash64(seed: int, stream: int, index: int) -> int:
    return int(host().synth_hash_host(seed, stream, index))


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fill(r: Recipe, dtype: int, n: int, start: int = 0, shape=None) -> np.ndarray:
    """Host array of value(start .. start+n) in dtype (bit patterns for 16-bit types)."""
    out = np.empty(n, dtype=_NP[dtype])
    host().synth_fill(ctypes.byref(r), dtype, start, n, out.ctypes.data_as(ctypes.c_void_p), _threads())
    return out.reshape(shape) if shape is not None else out


def fill_at(r: Recipe, dtype: int, idx: np.ndarray) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.size, dtype=_NP[dtype])
    host().synth_fill_at(ctypes.byref(r), dtype, idx.ctypes.data_as(ctypes.c_void_p), idx.size,
                         out.ctypes.data_as(ctypes.c_void_p), _threads())
    return out


def fill_device(r: Recipe, dtype: int, out_tensor, start: int = 0) -> None:
    """Fill a contiguous CUDA tensor (any element type of the right width) on the current stream."""
    import torch

    assert out_tensor.is_cuda and out_tensor.is_contiguous()
    n = out_tensor.numel() * out_tensor.element_size() // np.dtype(_NP[dtype]).itemsize
    rc = dev().synth_fill_dev(ctypes.byref(r), dtype, start, n, ctypes.c_void_p(out_tensor.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc:
        raise RuntimeError(f"synth_fill_dev failed: cuda error {rc}")


def fill_device_at(r: Recipe, dtype: int, idx_tensor, out_tensor) -> None:
    import torch

    rc = dev().synth_fill_at_dev(ctypes.byref(r), dtype, ctypes.c_void_p(idx_tensor.data_ptr()),
                                 idx_tensor.numel(), ctypes.c_void_p(out_tensor.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc:
        raise RuntimeError(f"synth_fill_at_dev failed: cuda error {rc}")
