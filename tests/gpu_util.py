"""Helpers shared by the GPU parity tests: host<->device byte moves, ulp
distances, and a multi-threaded driver that runs the oracle's own functions
on row chunks (the C oracle releases the GIL inside each call)."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle as O


def to_dev(a: np.ndarray, dtype=None):
    """numpy -> CUDA tensor with the same bytes; dtype reinterprets 16-bit data
    as torch.float16 / torch.bfloat16."""
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
        t = t.view(dtype) if dtype is not None else t
    elif a.dtype == np.uint32:
        t = torch.from_numpy(a.view(np.int32))
    else:
        t = torch.from_numpy(a)
    return t.cuda()


def to_host(t, np_dtype) -> np.ndarray:
    import torch

    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.float16, torch.bfloat16, torch.int16):
        return t.view(torch.int16).numpy().view(np.uint16).astype(np_dtype, copy=False)
    if t.dtype == torch.int32 and np_dtype == np.uint32:
        return t.numpy().view(np.uint32)
    return t.numpy().view(np_dtype) if t.numpy().dtype.itemsize == np.dtype(np_dtype).itemsize else t.numpy()


def ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|ulp distance| between float32 arrays (NaN pairs count as 0 if both NaN)."""
    def ordered(x):
        i = x.view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)

    d = np.abs(ordered(np.ascontiguousarray(a, np.float32)) - ordered(np.ascontiguousarray(b, np.float32)))
    both_nan = np.isnan(a) & np.isnan(b)
    return np.where(both_nan, 0, d)


def threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def nvfp4_oracle(x_u16: np.ndarray, block_2d: bool, stochastic: bool, seed: int, rht: bool, mask: int,
                 want_dequant: bool = True):
    """The oracle's NVFP4 quantiser, evaluated on row chunks in parallel:
    x' per chunk, amax = max over chunk amaxes, then encode per chunk."""
    rows, cols = x_u16.shape
    step = max(16, ((rows // (4 * threads())) // 16) * 16) if rows >= 64 else rows
    chunks = [(r, min(rows, r + step)) for r in range(0, rows, step)] or [(0, 0)]
    xp = np.empty((rows, cols), np.float32)

    def prep(c):
        r0, r1 = c
        if r1 > r0:
            xp[r0:r1] = O.nvfp4_prepare(x_u16[r0:r1], rht, mask)
        return O.amax(xp[r0:r1], O.F32) if r1 > r0 else 0.0

    with cf.ThreadPoolExecutor(threads()) as ex:
        amaxes = list(ex.map(prep, chunks))
    nan = any(np.isnan(a) for a in amaxes)
    amax = float("nan") if nan else max(amaxes)
    s_t, nf = O.nvfp4_tensor_scale(amax)
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros(((rows // 16) if block_2d else rows, cols // 16), np.uint8)
    dq = np.zeros((rows, cols), np.uint16) if want_dequant else None

    def enc(c):
        r0, r1 = c
        if r1 <= r0:
            return
        cd, sc, d = O.nvfp4_encode_rows(xp[r0:r1], r0, cols, block_2d, stochastic, seed, s_t, nf, want_dequant)
        codes[r0:r1] = cd
        if block_2d:
            scales[r0 // 16:r1 // 16] = sc
        else:
            scales[r0:r1] = sc
        if want_dequant:
            dq[r0:r1] = d

    with cf.ThreadPoolExecutor(threads()) as ex:
        list(ex.map(enc, chunks))
    return codes, scales, s_t, nf, dq
