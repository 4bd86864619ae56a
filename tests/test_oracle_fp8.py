"""Pins for the oracle's FP8 delayed-scaling cast (CPU).

The scale recurrence is checked against its closed form on tensors whose
amax is known by construction, including the eviction of an old amax from
the history window; amax against numpy; the cast against torch's float8
conversion inside the representable range.
"""
import numpy as np
import pytest
import torch

import oracle as O


def bf16(x):
    return O.convert(np.asarray(x, np.float32), O.F32, O.BF16)


@pytest.mark.parametrize("fmt", [O.F32, O.F16, O.BF16])
def test_amax_matches_numpy(fmt):
    rng = np.random.default_rng(fmt)
    x = (rng.standard_normal(100_001) * 3).astype(np.float32)
    xin = x if fmt == O.F32 else O.convert(x, O.F32, fmt)
    xf = O.convert(xin, fmt, O.F32)
    assert O.amax(xin, fmt) == np.abs(xf).max()
    xin2 = xin.copy()
    xin2[777] = 0x7FC1 if fmt != O.F32 else np.float32("nan")
    assert O.amax_f32_bits(xin2, fmt) == 0x7FC00000
    assert O.amax(np.zeros(5, np.float32), O.F32) == 0.0


def one_hot(n, pos, val):
    x = np.zeros(n, np.float32)
    x[pos] = val
    return bf16(x)


@pytest.mark.parametrize("fmt,fmax", [(O.E4M3, 448.0), (O.E5M2, 57344.0)])
def test_delayed_scale_closed_form_with_window_eviction(fmt, fmax):
    N = 4
    amaxes = [64.0, 2.0, 4.0, 8.0, 1.0, 0.5, 16.0, 0.25, 0.25, 0.25]
    meta = O.new_fp8_meta()
    hist = np.zeros(N, np.float32)
    scales_in_force = []
    for k, a in enumerate(amaxes):
        scales_in_force.append(meta.scale)
        O.fp8_cast_delayed(one_hot(1000, 3 * k + 1, a), O.BF16, fmt, meta, hist, 1.0)
        window = amaxes[max(0, k - N + 1):k + 1]
        assert meta.amax == a
        assert meta.scale == np.float32(fmax) / np.float32(max(window))
        assert meta.scale_inv == np.float32(1.0) / np.float32(meta.scale)
        assert meta.pos == (k + 1) % N
    # the first tensor is cast with the initial scale 1; 64 is evicted at k = 4
    assert scales_in_force[0] == 1.0
    assert scales_in_force[4] == np.float32(fmax) / np.float32(64.0)
    assert scales_in_force[5] == np.float32(fmax) / np.float32(8.0)


def test_margin_divides_the_scale():
    meta = O.new_fp8_meta()
    hist = np.zeros(8, np.float32)
    O.fp8_cast_delayed(one_hot(64, 5, 3.0), O.BF16, O.E4M3, meta, hist, 2.0)
    assert meta.scale == np.float32(448.0) / np.float32(6.0)


def test_cast_uses_the_scale_from_previous_steps():
    # Step 1 runs with scale 1, so 1000 clips to 448; step 2 runs with
    # 448 / 1000, so 500 lands on 224 exactly.
    meta = O.new_fp8_meta()
    hist = np.zeros(16, np.float32)
    y1 = O.fp8_cast_delayed(bf16([1000.0, -1000.0, 1.0]), O.BF16, O.E4M3, meta, hist, 1.0)
    assert list(y1) == [0x7E, 0xFE, 0x38]
    y2 = O.fp8_cast_delayed(bf16([500.0, 0.0, -3.0]), O.BF16, O.E4M3, meta, hist, 1.0)
    s = np.float32(448.0) / np.float32(1000.0)
    ref = torch.from_numpy(np.array([500.0, 0.0, -3.0], np.float32) * s).to(torch.float8_e4m3fn)
    assert list(y2) == list(ref.view(torch.uint8).numpy())
    assert y2[0] == 0x76  # 224 = 1.75 * 2^7


def test_zero_or_nonfinite_history_keeps_the_scale():
    meta = O.new_fp8_meta()
    hist = np.zeros(4, np.float32)
    O.fp8_cast_delayed(bf16(np.zeros(10)), O.BF16, O.E4M3, meta, hist, 1.0)
    assert meta.scale == 1.0 and meta.amax == 0.0
    x = np.zeros(10, np.uint16)
    x[2] = 0x7FC0  # NaN
    y = O.fp8_cast_delayed(x, O.BF16, O.E4M3, meta, hist, 1.0)
    assert np.isnan(meta.amax) and meta.scale == 1.0 and y[2] == 0x7F
    x[2] = 0x7F80  # +inf clips to the largest value
    y = O.fp8_cast_delayed(x, O.BF16, O.E5M2, O.new_fp8_meta(), np.zeros(4, np.float32), 1.0)
    assert y[2] == 0x7B


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_cast_matches_torch_inside_range(fmt):
    dt = torch.float8_e4m3fn if fmt == O.E4M3 else torch.float8_e5m2
    rng = np.random.default_rng(7)
    xb = bf16(rng.standard_normal(200_000).astype(np.float32))
    scale = np.float32(120.5 if fmt == O.E4M3 else 15000.0)
    y = O.fp8_cast_array(xb, O.BF16, fmt, scale)
    p = O.convert(xb, O.BF16, O.F32) * scale
    maxv = 448.0 if fmt == O.E4M3 else 57344.0
    inr = np.abs(p) <= maxv
    ref = torch.from_numpy(p[inr]).to(dt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(y[inr], ref)
    sat = ~inr
    assert sat.any()
    np.testing.assert_array_equal(y[sat], np.where(p[sat] > 0, 0x7E if fmt == O.E4M3 else 0x7B,
                                                   0xFE if fmt == O.E4M3 else 0xFB))


def test_ring_slot_is_taken_modulo_the_length():
    meta = O.new_fp8_meta()
    meta.pos = 9
    hist = np.zeros(4, np.float32)
    O.fp8_cast_delayed(one_hot(32, 0, 5.0), O.BF16, O.E4M3, meta, hist, 1.0)
    assert hist[1] == 5.0 and meta.pos == 2


@pytest.mark.parametrize("fmt,fmax", [(O.E4M3, 448.0), (O.E5M2, 57344.0)])
def test_most_recent_uses_only_the_latest_amax(fmt, fmax):
    # [FP8-TE] checklist: amax_compute_algo = most_recent follows fast changes.
    meta = O.new_fp8_meta()
    hist = np.zeros(8, np.float32)
    for k, a in enumerate([64.0, 2.0, 4.0, 0.5, 100.0, 1.0]):
        O.fp8_cast_delayed(one_hot(64, k, a), O.BF16, fmt, meta, hist, 2.0, O.AMAX_MOST_RECENT)
        assert meta.scale == np.float32(fmax) / (np.float32(2.0) * np.float32(a))
        assert hist[k] == a  # the ring is still recorded
    O.fp8_cast_delayed(bf16(np.zeros(16)), O.BF16, fmt, meta, hist, 2.0, O.AMAX_MOST_RECENT)
    assert meta.scale == np.float32(fmax) / np.float32(2.0)  # zero amax keeps the scale


def test_transpose_matches_numpy():
    y = np.random.default_rng(1).integers(0, 256, size=(48, 80)).astype(np.uint8)
    np.testing.assert_array_equal(O.transpose_u8(y), y.T)


def test_nan_bytes_match_torch():
    """Reading R1: a NaN becomes S.1111111 with its sign, the bytes torch's
    float8 casts produce for both signs; a NaN product (an infinity times a
    zero multiplier) takes the input element's sign."""
    import torch

    x = np.array([np.nan, -np.nan], np.float32)
    for fmt, dt in ((O.E4M3, torch.float8_e4m3fn), (O.E5M2, torch.float8_e5m2)):
        lib = torch.from_numpy(x).to(dt).view(torch.uint8).numpy()
        np.testing.assert_array_equal(O.convert(x, O.F32, fmt), lib)
        np.testing.assert_array_equal(lib, [0x7F, 0xFF])
        np.testing.assert_array_equal(O.fp8_cast_array(np.array([np.inf, -np.inf], np.float32), O.F32, fmt, 0.0),
                                      [0x7F, 0xFF])
        # 16-bit NaN inputs of both signs (every NaN payload) keep their sign too
        for src, tdt, fmt16 in ((np.arange(0x7F81, 0x7FFF + 1), torch.bfloat16, O.BF16),
                                (np.arange(0x7C01, 0x7FFF + 1), torch.float16, O.F16)):
            bits = np.concatenate([src, src | 0x8000]).astype(np.uint16)
            want = torch.from_numpy(bits.view(np.int16)).view(tdt).to(dt).view(torch.uint8).numpy()
            np.testing.assert_array_equal(O.fp8_cast_array(bits, fmt16, fmt, 1.0), want)


@pytest.mark.parametrize("fmt,fmax", [(O.E4M3, 448.0), (O.E5M2, 57344.0)])
def test_saturation_count_closed_form(fmt, fmax):
    """Integers 0..9999 at scale s: exactly those with k * s > fmax saturate
    (the products are exact here), infinities count, NaN does not; the count
    equals the number of saturated bytes in the cast."""
    k = np.arange(10000, dtype=np.float32)
    for s in (0.5, 1.0, 7.0):  # k * s exact in binary32: k > fmax / s saturates
        assert O.fp8_saturation_count(k, O.F32, fmt, s) == max(0, 9999 - int(np.floor(fmax / s)))
    x = np.array([np.inf, -np.inf, np.nan, 1.0, -1e9], np.float32)
    assert O.fp8_saturation_count(x, O.F32, fmt, 1.0) == 3
    y = O.fp8_cast_array(x[[0, 1, 3, 4]], O.F32, fmt, 1.0)
    maxcode = 0x7E if fmt == O.E4M3 else 0x7B
    assert int(np.sum((y & 0x7F) == maxcode)) == 3
