"""GPU: the 16-bit NaN (reading R-NaN16) against a library, and where the
library's kernels write one.

torch's CUDA casts (a library, not this repository's kernels) write every
binary32 NaN, of either sign and any payload, as 0x7FFF in FP16 and BF16:
the oracle's encoding.  The kernels' own 16-bit NaN outputs are then checked
against the oracle: the BF16 output of rht16 for tiles holding a NaN or
infinities of both signs, and the optimizer's working copy of a NaN master.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

import mixed_precision_numerics_gb300 as M  # noqa: E402


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def all_f32_nans():
    m = np.arange(1, 1 << 23, dtype=np.uint32)
    return np.concatenate([0x7F800000 | m, 0xFF800000 | m]).view(np.float32)


@pytest.mark.parametrize("fmt,dt", [(O.F16, torch.float16), (O.BF16, torch.bfloat16)])
def test_torch_cuda_casts_of_every_nan_match_the_oracle(fmt, dt):
    nans = all_f32_nans()
    got = to_host(torch.from_numpy(nans).cuda().to(dt), np.uint16)
    np.testing.assert_array_equal(got, O.convert(nans, O.F32, fmt))


def test_rht16_bf16_output_of_non_finite_tiles():
    rows, cols = 8, 64
    x = synth.fill(synth.recipe(90, 0, 1.0), synth.BF16, rows * cols, shape=(rows, cols))
    x[0, 3] = 0x7FC0   # NaN
    x[1, 20] = 0xFFC1  # negative NaN with a payload
    x[2, 5] = 0x7F80   # +inf alone in its tile: +-inf outputs
    # +inf and -inf side by side: the first butterfly stage makes inf - inf
    # at one position, whose NaN then reaches every even position of the tile
    x[3, 40], x[3, 41] = 0x7F80, 0xFF80
    mask = 0x9C31
    for out, fmt in ((torch.bfloat16, O.BF16), (torch.float32, O.F32)):
        y = torch.empty((rows, cols), dtype=out, device="cuda")
        M.rht16(to_dev(x, torch.bfloat16), y, mask)
        torch.cuda.synchronize()
        ref = O.rht16(x, mask, fmt)
        if fmt == O.BF16:
            got = to_host(y, np.uint16)
            assert (got == 0x7FFF).sum() == 16 + 16 + 8
            np.testing.assert_array_equal(got, ref.view(np.uint16))
        else:
            # a binary32 NaN's bits are not part of the method's result: the
            # NaN positions and every other value bit for bit
            got = y.cpu().numpy()
            nan = np.isnan(ref)
            assert nan.sum() == 16 + 16 + 8
            np.testing.assert_array_equal(np.isnan(got), nan)
            np.testing.assert_array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


@pytest.mark.parametrize("w_fmt,dt,mpd", [(O.F16, torch.float16, M.MP_F16), (O.BF16, torch.bfloat16, M.MP_BF16)])
def test_working_copy_of_a_nan_master(w_fmt, dt, mpd):
    n = 1000
    w0 = synth.fill(synth.recipe(91, 0, 0.02), synth.F32, n)
    w0[[3, 500]] = np.array([0x7FC00000, 0xFFC00001], np.uint32).view(np.float32)
    g = synth.fill(synth.recipe(92, 0, 1e-3), synth.F16, n)
    w, m, v = to_dev(w0), torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    w16 = torch.empty(n, dtype=dt, device="cuda")
    st = M.new_scaler_state(1.0)
    M.mp_adamw_step([M.Param(w, m, v, to_dev(g, torch.float16), w16)], M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01),
                    st, grad_dtype=M.MP_F16, working_dtype=mpd)
    torch.cuda.synchronize()
    ow, om, ov, ow16 = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    O.adamw_step(O.AdamwHp(1e-3, 0.9, 0.999, 1e-8, 0.01), O.new_scaler_state(1.0), [(ow, om, ov, g, ow16)],
                 O.F16, w_fmt)
    got = to_host(w16, np.uint16)
    assert got[3] == got[500] == 0x7FFF
    np.testing.assert_array_equal(got, ow16)
