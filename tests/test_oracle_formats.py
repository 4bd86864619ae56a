"""Pins for the oracle's number formats (CPU only).

Each check ties the oracle to something other than itself: values printed on
the pages (golden fixtures), library conversions (numpy float16, torch
bfloat16 / float8), or a brute-force nearest-code search over every code.
"""
import numpy as np
import pytest
import torch

from tests.conftest import golden

import oracle as O


def f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def all_bf16_as_f32():
    b = np.arange(65536, dtype=np.uint32)
    return (b << 16).view(np.float32)


def random_f32(n, seed=0):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32)


# ---- FP16 ---------------------------------------------------------------------


def test_fp16_page_limits():
    g = golden("fp16_limits.json")
    enc = lambda v: O.lib().orc_f32_to_f16(float(v))
    dec = lambda h: O.lib().orc_f16_to_f32(h)
    assert enc(g["max_finite"]) == 0x7BFF and dec(0x7BFF) == g["max_finite"]
    assert enc(g["min_normal"]) == 0x0400 and dec(0x0400) == g["min_normal"]
    assert enc(g["min_subnormal"]) == 0x0001 and dec(0x0001) == g["min_subnormal"]
    # below 2^-24 it becomes zero: half of it is a tie that goes to even (0)
    assert enc(g["underflow_below"] / 2) == 0x0000
    assert enc(-g["underflow_below"] / 2) == 0x8000
    assert enc(np.nextafter(np.float32(2**-25), np.float32(1))) == 0x0001
    # the largest finite value plus half an ulp (16) is a tie to the even code,
    # which is past the top of the format: infinity
    assert enc(65519.99) == 0x7BFF
    assert enc(65520.0) == 0x7C00
    assert enc(-1e6) == 0xFC00


def test_fp16_encode_matches_numpy_library():
    x = np.concatenate([random_f32(400_000, 1), all_bf16_as_f32()])
    # add every f16 value and every midpoint between neighbours
    h = np.arange(0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, h.astype(np.float32), mids, -mids])
    x = x[~np.isnan(x)]
    ours = O.convert(x, O.F32, O.F16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_fp16_decode_matches_numpy_library():
    h = np.arange(65536, dtype=np.uint16)
    ours = O.convert(h, O.F16, O.F32)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def all_f32_nans():
    m = np.arange(1, 1 << 23, dtype=np.uint32)
    return np.concatenate([0x7F800000 | m, 0xFF800000 | m]).view(np.float32)


def test_16bit_nan_is_the_image_of_the_canonical_binary32_nan():
    """Reading R-NaN16: every binary32 NaN, whatever its sign and payload, is
    written as the 16-bit image of the canonical binary32 NaN 0x7FFFFFFF (the
    NaN a GPU's arithmetic returns, so a NaN's bits never depend on which
    operation made it).  That image is what numpy's and torch's CPU FP16
    casts write for 0x7FFFFFFF, and in BF16, whose values are the upper
    halves of binary32 values, the upper half 0x7FFF."""
    canon = np.array([0x7FFFFFFF], np.uint32).view(np.float32)
    f16_numpy = int(canon.astype(np.float16).view(np.uint16)[0])
    f16_torch = int(torch.from_numpy(canon).to(torch.float16).view(torch.int16).numpy().view(np.uint16)[0])
    bf16_upper_half = 0x7FFFFFFF >> 16
    assert f16_numpy == f16_torch == 0x7FFF
    nans = all_f32_nans()
    assert (O.convert(nans, O.F32, O.F16) == f16_numpy).all()
    assert (O.convert(nans, O.F32, O.BF16) == bf16_upper_half).all()
    # and both decode to a NaN again
    assert np.isnan(O.convert(np.array([f16_numpy], np.uint16), O.F16, O.F32)[0])
    assert np.isnan(O.convert(np.array([bf16_upper_half], np.uint16), O.BF16, O.F32)[0])


# ---- BF16 ---------------------------------------------------------------------


def test_bf16_encode_matches_torch_library():
    x = np.concatenate([random_f32(400_000, 2), all_bf16_as_f32()])
    b = np.arange(65536, dtype=np.uint32)
    lo = ((b << 16) | 0x8000).view(np.float32)  # exact midpoints
    x = np.concatenate([x, lo, ((b << 16) | 0x7FFF).view(np.float32), ((b << 16) | 0x8001).view(np.float32)])
    x = x[~np.isnan(x)]
    ours = O.convert(x, O.F32, O.BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_decode_is_upper_half_of_f32():
    h = np.arange(65536, dtype=np.uint16)
    ours = O.convert(h, O.BF16, O.F32)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# ---- FP8 ----------------------------------------------------------------------


def fp8_table_from_torch(fmt):
    dt = torch.float8_e4m3fn if fmt == O.E4M3 else torch.float8_e5m2
    return torch.arange(256, dtype=torch.uint8).view(dt).float().numpy()


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_decode_matches_torch_library(fmt):
    ours = np.array([O.lib().orc_fp8_to_f32(c, fmt) for c in range(256)], dtype=np.float32)
    ref = fp8_table_from_torch(fmt)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_fp8_page_ranges():
    g = golden("fp8_formats.json")
    L = O.lib()
    t = fp8_table_from_torch(O.E4M3)
    assert np.nanmax(t) == g["e4m3"]["max_finite"] == 448.0
    assert L.orc_f32_to_fp8_sat(448.0, O.E4M3) == 0x7E
    assert L.orc_f32_to_fp8_sat(-448.0, O.E4M3) == 0xFE
    # clip(x, -448, 448): anything larger saturates, infinities included
    for v in (449.0, 1e4, 3e38, float("inf")):
        assert L.orc_f32_to_fp8_sat(v, O.E4M3) == 0x7E
        assert L.orc_f32_to_fp8_sat(-v, O.E4M3) == 0xFE
    # E5M2 keeps IEEE infinities in its code space, so its largest finite
    # value is the one below the all-ones exponent: 1.75 * 2^15
    t5 = fp8_table_from_torch(O.E5M2)
    assert np.isinf(t5[0x7C]) and t5[0x7B] == 57344.0
    assert L.orc_f32_to_fp8_sat(float("inf"), O.E5M2) == 0x7B
    assert L.orc_f32_to_fp8_sat(float("nan"), O.E4M3) == 0x7F
    assert L.orc_f32_to_fp8_sat(float("nan"), O.E5M2) == 0x7F


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_encode_brute_force_all_bf16(fmt):
    table = fp8_table_from_torch(fmt)
    x = all_bf16_as_f32()
    x = x[~np.isnan(x)]
    ours = O.convert(x, O.F32, fmt).astype(np.int64)
    # vectorised brute force over the 128 non-negative codes
    pos = np.arange(128)
    pv = table[pos].astype(np.float64)
    ok = np.isfinite(pv)
    pv, pc = pv[ok], pos[ok]
    a = np.abs(x.astype(np.float64))
    a = np.where(np.isinf(a), pv.max() * 4, a)
    d = np.abs(a[:, None] - pv[None, :])
    best = d.min(axis=1, keepdims=True)
    is_best = d == best
    # prefer even codes among ties
    score = np.where(is_best, np.where((pc & 1) == 0, 2, 1), 0)
    c = pc[np.argmax(score, axis=1)]
    c = np.where(a > pv.max(), pc[np.argmax(pv)], c)
    ref = c | np.where(np.signbit(x), 128, 0)
    np.testing.assert_array_equal(ours, ref)


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_fp8_encode_matches_torch_in_range(fmt):
    dt = torch.float8_e4m3fn if fmt == O.E4M3 else torch.float8_e5m2
    maxv = 448.0 if fmt == O.E4M3 else 57344.0
    x = random_f32(300_000, 3)
    x = x[np.isfinite(x) & (np.abs(x) <= maxv)]
    x = np.concatenate([x, (np.random.default_rng(4).standard_normal(200_000) * 10).astype(np.float32)])
    x = x[np.abs(x) <= maxv]
    ours = O.convert(x, O.F32, fmt)
    ref = torch.from_numpy(x).to(dt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


# ---- E2M1 ----------------------------------------------------------------------


def test_e2m1_grid():
    g = golden("nvfp4_format.json")
    vals = [O.lib().orc_e2m1_to_f32(c) for c in range(16)]
    assert vals[:8] == g["e2m1_magnitudes"]
    assert vals[8:] == [-v for v in g["e2m1_magnitudes"]]
    assert np.signbit(vals[8])


def test_e2m1_ties_and_saturation():
    L = O.lib()
    enc = lambda v: L.orc_f32_to_e2m1(v)
    # ties go to the code with an even last bit
    assert [enc(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == [0, 2, 2, 4, 4, 6, 6]
    assert [enc(v) for v in (6.0, 7.0, 1e30)] == [7, 7, 7]
    assert enc(-0.0) == 8 and enc(-0.1) == 8 and enc(0.1) == 0


def test_e2m1_brute_force_all_bf16():
    g = np.array(golden("nvfp4_format.json")["e2m1_magnitudes"])
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    ours = O.convert(x, O.F32, O.E2M1).astype(np.int64)
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - g[None, :])
    best = d.min(axis=1, keepdims=True)
    codes = np.arange(8)
    score = np.where(d == best, np.where((codes & 1) == 0, 2, 1), 0)
    c = np.argmax(score, axis=1)
    c = np.where(a > 6.0, 7, c)
    ref = c | np.where(np.signbit(x), 8, 0)
    np.testing.assert_array_equal(ours, ref)


# ---- lost update and underflow ------------------------------------------------


def test_lost_update_threshold_fp16():
    g = golden("lost_update.json")
    L = O.lib()
    thr = 2.0 ** g["relative_threshold_log2"]
    spacing = 2.0 ** g["spacing_near_one_log2"]
    one = L.orc_f32_to_f16(1.0)
    # an update of half the threshold relative to w = 1 disappears in FP16
    assert L.orc_f32_to_f16(1.0 + thr / 2) == one
    assert L.orc_f32_to_f16(1.0 - thr / 2) == one  # tie, even code is 1.0
    # an update of one spacing survives
    assert L.orc_f16_to_f32(L.orc_f32_to_f16(1.0 + spacing)) == 1.0 + spacing
    # and the FP32 master keeps the small update
    assert np.float32(1.0) + np.float32(thr / 2) != np.float32(1.0)


def test_gradient_underflow_and_loss_scaling():
    g = golden("fp16_limits.json")
    L = O.lib()
    tiny = g["underflow_below"] / 2  # 2^-25: lost in FP16
    assert L.orc_f32_to_f16(tiny) == 0
    S = golden("gradscaler.json")["init_scale"]
    h = L.orc_f32_to_f16(tiny * S)  # 2^-9 after scaling: representable
    assert L.orc_f16_to_f32(h) == tiny * S
    # unscaling in FP32 restores it exactly
    assert np.float32(L.orc_f16_to_f32(h)) * np.float32(1.0 / S) == np.float32(tiny)
