"""Pins for the oracle's MX block formats (32-element blocks, UE8M0 scales)."""
import numpy as np
import pytest
import torch

from tests.conftest import golden

import oracle as O

GRID = np.array(golden("nvfp4_format.json")["e2m1_magnitudes"])
EMAX = {O.E4M3: 8, O.E5M2: 15, O.E2M1: 2, O.E2M3: 2, O.E3M2: 4}

# FP6 magnitudes, codes 0..31 in order, written out from the bit layouts:
# E2M3 subnormals k/8, then 1.000..1.875 x 2^0..2^2; E3M2 subnormals k/16,
# then 1.00..1.75 x 2^-2..2^4.
E2M3_MAGS = [0, .125, .25, .375, .5, .625, .75, .875,
             1, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875,
             2, 2.25, 2.5, 2.75, 3, 3.25, 3.5, 3.75,
             4, 4.5, 5, 5.5, 6, 6.5, 7, 7.5]
E3M2_MAGS = [0, .0625, .125, .1875, .25, .3125, .375, .4375,
             .5, .625, .75, .875, 1, 1.25, 1.5, 1.75,
             2, 2.5, 3, 3.5, 4, 5, 6, 7,
             8, 10, 12, 14, 16, 20, 24, 28]
FP6 = {O.E2M3: E2M3_MAGS, O.E3M2: E3M2_MAGS}


def bf16(x):
    return O.convert(np.asarray(x, np.float32), O.F32, O.BF16)


def ue8m0_value(code):
    # library decode of the scale byte (torch's float8_e8m0fnu)
    return torch.tensor(np.asarray(code, np.uint8)).view(torch.float8_e8m0fnu).float().numpy()


@pytest.mark.parametrize("fmt", [O.E2M3, O.E3M2])
def test_fp6_decode_table(fmt):
    codes = np.arange(64, dtype=np.uint8)
    got = O.convert(codes, fmt, O.F32)
    mags = np.array(FP6[fmt], np.float32)
    np.testing.assert_array_equal(got[:32], mags)
    np.testing.assert_array_equal(got[32:], -mags)


@pytest.mark.parametrize("fmt", [O.E2M3, O.E3M2])
def test_fp6_encode_brute_force_every_bf16(fmt):
    """Nearest magnitude, ties to the even code, beyond the largest value
    saturating, sign kept (also on zero): every finite BF16 pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = O.convert(bits, O.BF16, O.F32)
    fin = np.isfinite(x)
    bits, x = bits[fin], x[fin]
    got = O.convert(bits, O.BF16, fmt)
    mags = np.array(FP6[fmt], np.float64)
    a = np.minimum(np.abs(x.astype(np.float64)), mags[-1])
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equidistant neighbours take the even code
    idx = np.where(cand.sum(axis=1) > 1, np.argmax(cand & (np.arange(32)[None, :] % 2 == 0), axis=1),
                   np.argmax(cand, axis=1))
    want = idx.astype(np.uint8) | np.where(np.signbit(x), 0x20, 0).astype(np.uint8)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2, O.E2M1, O.E2M3, O.E3M2])
def test_scale_exponent_closed_form(fmt):
    # each block's largest magnitude is a power of two 2^k (k from -20 to 20):
    # the scale is 2^(k - emax) and that element lands on 2^emax
    ks = np.arange(-20, 21)
    x = np.zeros((len(ks), 32), np.float32)
    rng = np.random.default_rng(0)
    for i, k in enumerate(ks):
        x[i] = rng.uniform(-1, 1, 32) * 2.0**k
        x[i, 5] = 2.0**k
    codes, scales, dq = O.mx_quantize(bf16(x), O.BF16, fmt)
    np.testing.assert_array_equal(scales[:, 0].astype(int) - 127, ks - EMAX[fmt])
    np.testing.assert_array_equal(ue8m0_value(scales[:, 0]), 2.0 ** (ks - EMAX[fmt]))
    # dequantised block maximum is exact
    np.testing.assert_array_equal(O.convert(dq[:, 5], O.BF16, O.F32), 2.0**ks)


def test_e2m1_elements_brute_force():
    rng = np.random.default_rng(3)
    x = bf16(rng.standard_normal((8, 64)) * 3)
    codes, scales, _ = O.mx_quantize(x, O.BF16, O.E2M1)
    xf = O.convert(x, O.BF16, O.F32)
    for r in range(8):
        for b in range(2):
            e = int(scales[r, b]) - 127
            for j in range(32):
                y = np.float32(xf[r, b * 32 + j]) * np.float32(2.0**-e)
                a = abs(float(y))
                d = np.abs(GRID - min(a, 7.0))
                cand = np.arange(8)[d == d.min()]
                c = 7 if a > 6 else int(cand[(cand & 1) == 0][0] if cand.size > 1 else cand[0])
                c |= 8 if np.signbit(y) else 0
                i = b * 32 + j
                got = (codes[r, i // 2] >> (4 * (i & 1))) & 0xF
                assert got == c


@pytest.mark.parametrize("fmt,dt", [(O.E4M3, torch.float8_e4m3fn), (O.E5M2, torch.float8_e5m2)])
def test_fp8_elements_match_torch(fmt, dt):
    rng = np.random.default_rng(4)
    x = bf16(rng.standard_normal((16, 128)) * rng.choice([1e-3, 1.0, 300.0], size=(16, 1)))
    codes, scales, _ = O.mx_quantize(x, O.BF16, fmt)
    xf = O.convert(x, O.BF16, O.F32).reshape(16, 4, 32)
    y = xf * (2.0 ** -(scales.astype(np.float32) - 127))[:, :, None].astype(np.float32)
    maxv = 448.0 if fmt == O.E4M3 else 57344.0
    y = np.clip(y.astype(np.float32), -maxv, maxv)  # values between max and 2^(emax+1) saturate
    ref = torch.from_numpy(y.reshape(16, 128)).to(dt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref)


def test_zero_and_nonfinite_blocks():
    x = np.zeros((1, 96), np.float32)
    x[0, 40] = np.inf
    x[0, 64:] = 1.0
    codes, scales, dq = O.mx_quantize(bf16(x), O.BF16, O.E4M3)
    assert list(scales[0]) == [0, 0xFF, 127 - 8]
    assert not codes[0, :64].any() and not dq[0, :64].any()


def test_nvfp4_blocks_are_finer_than_mxfp4():
    # [NVFP4] §2.1 / §3: 16-element E4M3-scaled blocks track the data more
    # closely than 32-element power-of-two blocks; on Gaussian data the
    # NVFP4 dequantisation error is smaller.
    rng = np.random.default_rng(7)
    x = bf16(rng.standard_normal((64, 1024)))
    xf = O.convert(x, O.BF16, O.F32).astype(np.float64)
    _, _, dq_mx = O.mx_quantize(x, O.BF16, O.E2M1)
    _, _, _, _, dq_nv = O.nvfp4_quantize(x, False, False)
    e_mx = np.mean((O.convert(dq_mx, O.BF16, O.F32) - xf) ** 2)
    e_nv = np.mean((O.convert(dq_nv, O.BF16, O.F32) - xf) ** 2)
    assert e_nv < e_mx


def test_block_sizes_and_scale_kinds_printed_on_the_pages():
    g = golden("mx_format.json")
    rng = np.random.default_rng(11)
    x = bf16(rng.standard_normal((4, 256)) * 5)
    _, scales, dq = O.mx_quantize(x, O.BF16, O.E2M1)
    assert scales.shape == (4, 256 // g["mx_block"])
    # every MX scale is a power of two: its dequantised element values divide
    # by 2^(byte - 127) into E2M1 magnitudes
    mags = set(golden("nvfp4_format.json")["e2m1_magnitudes"])
    dqf = O.convert(dq, O.BF16, O.F32).reshape(4, -1, g["mx_block"])
    for r in range(4):
        for b in range(scales.shape[1]):
            unit = 2.0 ** (int(scales[r, b]) - 127)
            assert set(np.abs(dqf[r, b]) / unit) <= mags
    # NVFP4 keeps one E4M3 scale per 16 elements: twice as many scales
    _, nv_scales, _, _, _ = O.nvfp4_quantize(x, False, False, 0, False, 0)
    assert nv_scales.shape == (4, 256 // g["nvfp4_block"])
    assert nv_scales.size == 2 * scales.size
