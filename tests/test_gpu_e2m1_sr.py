"""GPU parity: e2m1_stochastic_round, the stochastic rounding of the NVFP4
encode ([NVFP4] §2.2 item 4) on values and random bits the test supplies,
against the oracle's rule (round away from zero iff floor(frac * 2^16) + r16
>= 2^16) element by element: every value k * 2^-10 in (-7, 7) with a spread
of random words, both sides of every decision boundary floor(frac * 2^16) = m
for a sample of m in every grid gap, random values and bits, and the special
values."""
import numpy as np
import pytest
import torch

import oracle as O
import mixed_precision_numerics_gb300 as M
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def gpu_codes(y, r16):
    y = np.ascontiguousarray(y, np.float32)
    r16 = np.ascontiguousarray(r16, np.uint16)
    out = torch.empty((y.size + 1) // 2, dtype=torch.uint8, device="cuda")
    M.e2m1_stochastic_round(to_dev(y), to_dev(r16), out)
    b = to_host(out, np.uint8)
    codes = np.empty(2 * b.size, np.uint8)
    codes[0::2], codes[1::2] = b & 0xF, b >> 4
    return codes[: y.size], b


def check(y, r16):
    got, _ = gpu_codes(y, r16)
    want = O.e2m1_sr_with_bits(y, r16)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(float(y[k]), int(r16[k]), int(want[k]), int(got[k])) for k in bad[:8]]


def test_every_kth_1024th_in_the_range_with_a_spread_of_bits():
    v = (np.arange(-7 * 1024 + 1, 7 * 1024) * 2.0**-10).astype(np.float32)
    words = np.array([0, 1, 0x00FF, 0x0100, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFF00, 0xFFFE, 0xFFFF], np.uint16)
    rng = np.random.default_rng(11)
    words = np.concatenate([words, rng.integers(0, 1 << 16, 53).astype(np.uint16)])
    check(np.repeat(v, words.size), np.tile(words, v.size))


def test_both_sides_of_the_decision_boundaries():
    """x at floor(frac * 2^16) = m exactly rounds up with r16 = 2^16 - m; one ulp
    below it (floor = m - 1) it does not."""
    rng = np.random.default_rng(12)
    ys, rs = [], []
    for lo, hi in zip(GRID[:-1], GRID[1:]):
        ms = np.unique(np.concatenate([np.arange(1, 64), (1 << 16) - np.arange(1, 64),
                                       rng.integers(1, 1 << 16, 2000)]))
        for sgn in (1.0, -1.0):
            x = (sgn * (lo + (hi - lo) * ms / 65536.0)).astype(np.float32)
            below = np.nextafter(x, np.float32(sgn * lo)).astype(np.float32)
            r = ((1 << 16) - ms).astype(np.uint16)
            ys += [x, below, x, below]
            rs += [r, r, r - 1, r + 1]
    y = np.concatenate(ys)
    r16 = np.concatenate(rs).astype(np.uint16)
    check(y, r16)
    # the boundary itself: exactly half of these round up
    got, _ = gpu_codes(y, r16)
    assert 0 < np.mean((got & 7) != (O.e2m1_sr_with_bits(y, np.zeros_like(r16)) & 7)) < 1


def test_random_values_and_bits_and_odd_length():
    rng = np.random.default_rng(13)
    n = (1 << 20) + 1
    y = (rng.standard_normal(n) * np.exp(rng.uniform(-12, 3, n))).astype(np.float32)
    r16 = rng.integers(0, 1 << 16, n).astype(np.uint16)
    check(y, r16)
    _, b = gpu_codes(y, r16)
    assert b[-1] >> 4 == 0  # high nibble of the last byte of an odd count


def test_special_values():
    sp = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -np.nan, 6.0, -6.0, 6.5, 7.0, 1e30, -1e30,
                   1e-45, -1e-45, 2.0**-126, 5.9999995, -5.9999995, 0.25, -0.25, 0.24999999], np.float32)
    for r in (0, 1, 0x7FFF, 0x8000, 0xFFFF):
        check(sp, np.full(sp.size, r, np.uint16))


def test_empty_is_a_no_op():
    out = torch.full((4,), 0xAB, dtype=torch.uint8, device="cuda")
    M.e2m1_stochastic_round(torch.empty(0, device="cuda"), torch.empty(0, dtype=torch.int16, device="cuda"), out)
    assert (out.cpu() == 0xAB).all()
