"""Pins for the oracle's fine-grained FP8 (online 1x128 / 128x128 block scales)."""
import numpy as np
import pytest
import torch

import oracle as O


def bf16(x):
    return O.convert(np.asarray(x, np.float32), O.F32, O.BF16)


@pytest.mark.parametrize("br,bc", [(1, 128), (128, 128)])
def test_block_scales_are_block_amax_over_448(br, bc):
    rng = np.random.default_rng(br)
    rows, cols = 300, 400  # partial blocks at both edges
    x = bf16(rng.standard_normal((rows, cols)) * rng.choice([1e-3, 1.0, 50.0], size=(rows, 1)))
    y, sc = O.fp8_quantize_blockwise(x, O.BF16, br, bc)
    xf = O.convert(x, O.BF16, O.F32)
    for i in range(sc.shape[0]):
        for j in range(sc.shape[1]):
            blk = xf[i * br:(i + 1) * br, j * bc:(j + 1) * bc]
            amax = np.float32(np.abs(blk).max())
            assert sc[i, j] == amax / np.float32(448.0)
            r = np.float32(448.0) / amax
            ref = torch.from_numpy(blk * r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(y[i * br:(i + 1) * br, j * bc:(j + 1) * bc], ref)


def test_block_maximum_maps_to_448_and_nothing_saturates():
    x = np.zeros((2, 256), np.float32)
    x[0, :128] = np.linspace(-3, 3, 128)
    x[0, 7] = 4.0  # amax a power of two: 448 / 4 is exact
    x[1, 128:] = np.linspace(-1e-3, 2e-3, 128)
    y, sc = O.fp8_quantize_blockwise(bf16(x), O.BF16, 1, 128)
    assert y[0, 7] == 0x7E and sc[0, 0] == np.float32(4.0) / np.float32(448.0)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert np.abs(table[y]).max() <= 448.0
    assert sc[0, 1] == 0.0 and not y[0, 128:].any()  # an all-zero block
    assert sc[1, 0] == 0.0


def test_dequantised_error_is_within_half_an_e4m3_step():
    rng = np.random.default_rng(2)
    x = bf16(rng.standard_normal((128, 512)))
    y, sc = O.fp8_quantize_blockwise(x, O.BF16, 128, 128)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    xf = O.convert(x, O.BF16, O.F32).astype(np.float64)
    s = np.repeat(sc.astype(np.float64), 128, axis=1)[:, :512].repeat(128, axis=0)[:128]
    deq = table[y] * s
    # relative step of E4M3 is 2^-3; subnormals (below 2^-6 of 448/amax scale) have an absolute step
    err = np.abs(deq - xf)
    bound = np.maximum(np.abs(xf) * 2.0**-4, s * 2.0**-10) * (1 + 1e-6)
    assert (err <= bound).all()


def test_nonfinite_block_flags_its_scale():
    x = np.ones((1, 256), np.float32)
    x[0, 3] = np.inf
    y, sc = O.fp8_quantize_blockwise(bf16(x), O.BF16, 1, 128)
    assert np.isinf(sc[0, 0]) and sc[0, 1] == np.float32(1.0) / np.float32(448.0)
    # r = 0: finite elements become zero and inf * 0 = NaN
    assert (y[0, :128][np.arange(128) != 3] == 0).all() and y[0, 3] == 0x7F


def test_nan_block_scale_is_the_quiet_nan():
    x = np.ones((1, 128), np.float32)
    x[0, 9] = np.nan
    y, sc = O.fp8_quantize_blockwise(bf16(x), O.BF16, 1, 128)
    assert sc.view(np.uint32)[0, 0] == 0x7FC00000 and y[0, 9] == 0x7F
