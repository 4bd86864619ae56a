"""Pins for the oracle's gradient-norm clipping (CPU).

The norm is the plain definition (squares of the binary32 unscaled grads,
exact in binary64, summed in order in binary64).  It is checked where the
exact answer is known (integer-valued grads), against math.fsum's correctly
rounded sum and numpy's pairwise float64 norm within the binary64 summation
bound, and the clipped step against the closed form of Adam's first update.
"""
import math

import numpy as np
import pytest

import oracle as O


def f16(x):
    return O.convert(np.asarray(x, np.float32), O.F32, O.F16)


@pytest.mark.parametrize("sizes", [[1], [7, 16384, 16385], [40000, 3, 100001]])
def test_sum_of_squares_is_exact_for_integer_grads(sizes):
    rng = np.random.default_rng(len(sizes))
    grads = [rng.integers(-3, 4, size=n) for n in sizes]
    norm = O.grad_norm([f16(g) for g in grads], O.F16, 1.0)
    exact = sum(int((g.astype(np.int64) ** 2).sum()) for g in grads)
    assert norm == np.sqrt(float(exact))


U64 = 2.0 ** -53


@pytest.mark.parametrize("g_fmt", [O.F16, O.BF16])
def test_norm_matches_fsum_and_unscales_first(g_fmt):
    rng = np.random.default_rng(5)
    S = 1024.0
    sizes = (5, 20000, 70001)
    grads = [(rng.standard_normal(n) * 1e-2 * S).astype(np.float32) for n in sizes]
    g16 = [O.convert(g, O.F32, g_fmt) for g in grads]
    # S is a power of two: the binary32 unscale is exact, so the squares of
    # fp32(grad) / S are the exact terms; fsum rounds their sum once.
    terms = [float(x) ** 2 for g in g16 for x in (O.convert(g, g_fmt, O.F32).astype(np.float64) / S)]
    exact = math.fsum(terms)
    norm = O.grad_norm(g16, g_fmt, float(np.float32(1.0 / S)))
    n = sum(sizes)
    # n binary64 additions of non-negative terms, then one square root
    assert abs(norm * norm - exact) <= (n + len(sizes)) * U64 * exact * 1.01
    assert abs(norm - math.sqrt(exact)) <= ((n + len(sizes)) * U64 / 2 + U64) * math.sqrt(exact)
    pairwise = np.sqrt(sum(float(((O.convert(g, g_fmt, O.F32).astype(np.float64) / S) ** 2).sum()) for g in g16))
    assert norm == pytest.approx(pairwise, rel=n * U64)


def test_norm_squares_the_binary32_unscaled_grad():
    # S = 3: 1/S is not a power of two, so fp32(g) * fp32(1/S) rounds; the
    # norm of one element is the magnitude of that binary32 product, exactly.
    inv = float(np.float32(1.0 / 3.0))
    for v in (1.0, 7.0, -1000.0, 65504.0, 2.0 ** -24):
        g = f16([v])
        gu = np.float32(O.convert(g, O.F16, O.F32)[0]) * np.float32(inv)
        assert O.grad_norm([g], O.F16, inv) == abs(float(gu))


def test_norm_of_split_tensors_adds_their_sums():
    rng = np.random.default_rng(11)
    g = f16(rng.standard_normal(50000))
    whole = O.grad_norm([g], O.F16, 1.0)
    parts = O.grad_norm([g[:12345], g[12345:40000], g[40000:]], O.F16, 1.0)
    assert parts == pytest.approx(whole, rel=50000 * U64)
    assert O.grad_norm([], O.F16, 1.0) == 0.0
    assert O.grad_norm([g[:0]], O.F16, 1.0) == 0.0


def test_non_finite_grads_give_a_non_finite_norm():
    g = f16([1.0, 2.0, 3.0])
    inf = g.copy()
    inf[1] = 0x7C00
    nan = g.copy()
    nan[2] = 0x7E00
    assert O.grad_norm([g], O.F16, 1.0) == math.sqrt(14.0)
    assert math.isinf(O.grad_norm([g, inf], O.F16, 1.0))
    assert math.isnan(O.grad_norm([nan, g], O.F16, 1.0))


def test_clip_coefficient_closed_form():
    assert O.clip_coef(0.5, 1.0) == 1.0
    assert O.clip_coef(4.0, 1.0) == np.float32(1.0 / (4.0 + 1e-6))
    assert O.clip_coef(0.0, 1.0) == 1.0
    assert O.clip_coef(1e30, 1.0) == np.float32(1e-30)


def test_clipped_first_step_closed_form():
    # One element, g = 1, eps = 1e-3: Adam's first update is lr * gc / (|gc| + eps)
    # with gc the clipped grad.  Clipping to norm 1e-3 gives gc = 1e-3 / (1 + 1e-6).
    lr, eps, max_norm = 1e-2, 1e-3, 1e-3
    hp = O.AdamwHp(lr, 0.9, 0.999, eps, 0.0, max_norm)
    w, m, v = np.zeros(1, np.float32), np.zeros(1, np.float32), np.zeros(1, np.float32)
    w16 = np.zeros(1, np.uint16)
    st = O.new_scaler_state(1.0)
    found, norm, clip = O.adamw_step(hp, st, [(w, m, v, f16([1.0]), w16)], O.F16, O.F16)
    assert found == 0 and norm == 1.0 and clip == np.float32(max_norm / (1.0 + 1e-6))
    gc = float(np.float32(clip))
    np.testing.assert_allclose(w[0], -lr * gc / (gc + eps), rtol=1e-5)
    # without clipping the same step moves w by about lr
    w2 = np.zeros(1, np.float32)
    O.adamw_step(O.AdamwHp(lr, 0.9, 0.999, eps, 0.0, 0.0), O.new_scaler_state(1.0),
                 [(w2, np.zeros(1, np.float32), np.zeros(1, np.float32), f16([1.0]), w16)], O.F16, O.F16)
    np.testing.assert_allclose(w2[0], -lr / (1 + eps), rtol=1e-5)


def test_no_clip_below_the_threshold_is_bitwise_unclipped():
    rng = np.random.default_rng(9)
    g = f16(rng.standard_normal(3000) * 1e-3)
    w0 = rng.standard_normal(3000).astype(np.float32)
    outs = []
    for mx in (0.0, 1e6):
        w, m, v, w16 = w0.copy(), np.zeros(3000, np.float32), np.zeros(3000, np.float32), np.zeros(3000, np.uint16)
        O.adamw_step(O.AdamwHp(1e-3, 0.9, 0.999, 1e-8, 0.01, mx), O.new_scaler_state(1.0), [(w, m, v, g, w16)],
                     O.F16, O.F16)
        outs.append((w, m, v, w16))
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
