"""Every binary32 and every binary16 bit pattern through the FP8 cast (E4M3 and
E5M2, scale 1) on the GPU, against the oracle's cast of the same values."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle as O
from tests.gpu_util import threads

import mixed_precision_numerics_gb300 as M  # noqa: E402

pytestmark = pytest.mark.gpu
CHUNK = 1 << 27


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def oracle_cast(x: np.ndarray, x_fmt: int, fmt: int) -> np.ndarray:
    parts = np.array_split(x, threads())
    with cf.ThreadPoolExecutor(len(parts)) as ex:
        outs = list(ex.map(lambda p: O.fp8_cast_array(p, x_fmt, fmt, 1.0), parts))
    return np.concatenate(outs)


@pytest.mark.parametrize("fmt", [M.MP_E4M3, M.MP_E5M2])
def test_every_fp32_pattern(fmt):
    ofmt = {M.MP_E4M3: O.E4M3, M.MP_E5M2: O.E5M2}[fmt]
    meta, hist = M.new_fp8_meta(), torch.zeros(4, device="cuda")
    xd = torch.empty(CHUNK, dtype=torch.float32, device="cuda")
    yd = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    for start in range(0, 1 << 32, CHUNK):
        bits = np.arange(start, start + CHUNK, dtype=np.uint32)
        x = bits.view(np.float32)
        meta.copy_(M.new_fp8_meta())  # scale 1 for every chunk (a cast sets the next call's scale)
        xd.copy_(torch.from_numpy(x))
        M.fp8_cast_delayed(xd, yd, fmt, meta, hist, 1.0)
        got = yd.cpu().numpy()
        want = oracle_cast(x, O.F32, ofmt)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"{bad.size} mismatches from 0x{start:08x}, first 0x{int(bits[bad[0]]):08x}"


@pytest.mark.parametrize("fmt", [M.MP_E4M3, M.MP_E5M2])
def test_every_fp16_pattern(fmt):
    ofmt = {M.MP_E4M3: O.E4M3, M.MP_E5M2: O.E5M2}[fmt]
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xd = torch.from_numpy(bits.view(np.int16)).view(torch.float16).cuda()
    y = torch.empty(65536, dtype=torch.uint8, device="cuda")
    M.fp8_cast_delayed(xd, y, fmt, M.new_fp8_meta(), torch.zeros(4, device="cuda"), 1.0)
    np.testing.assert_array_equal(y.cpu().numpy(), O.fp8_cast_array(bits, O.F16, ofmt, 1.0))
