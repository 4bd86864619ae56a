"""The device build of the input generator produces the host build's bits."""
import numpy as np
import pytest
import torch

import synth
import synth.workloads as W
from tests.gpu_util import to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


RECIPES = [
    (synth.recipe(0, 5, 1.0), synth.F32),
    (W.TINY.grad_recipe(3, 65536.0), synth.F16),
    (W.FP8.act_recipe(17), synth.BF16),
    (W.NVFP4_GRAD.recipe(), synth.BF16),
    (W.FULL.master_recipe(11), synth.F32),
]


@pytest.mark.parametrize("k", range(len(RECIPES)))
def test_device_fill_matches_host(k):
    r, dt = RECIPES[k]
    n = 1_000_003
    tdt = {synth.F32: torch.float32, synth.F16: torch.float16, synth.BF16: torch.bfloat16}[dt]
    t = torch.empty(n, dtype=tdt, device="cuda")
    synth.fill_device(r, dt, t, start=12345)
    torch.cuda.synchronize()
    host = synth.fill(r, dt, n, start=12345)
    got = to_host(t, np.float32 if dt == synth.F32 else np.uint16)
    np.testing.assert_array_equal(got.view(np.uint32) if dt == synth.F32 else got,
                                  host.view(np.uint32) if dt == synth.F32 else host)
    idx = np.array([0, 7, 999_999, 123_456_789_012], np.int64)
    out = torch.empty(idx.size, dtype=tdt, device="cuda")
    synth.fill_device_at(r, dt, torch.from_numpy(idx).cuda(), out)
    got = to_host(out, np.float32 if dt == synth.F32 else np.uint16)
    ref = synth.fill_at(r, dt, idx)
    np.testing.assert_array_equal(got.view(np.uint8), ref.view(np.uint8))
