"""Pins for the oracle's gradient-norm clipping (CPU).

The fixed summation order is checked where the exact answer is known
(integer-valued grads, whose squares and partial sums are exact in binary32),
against numpy's float64 norm elsewhere, and the clipped step against the
closed form of Adam's first update.
"""
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


def test_norm_matches_float64_and_unscales_first():
    rng = np.random.default_rng(5)
    S = 1024.0
    grads = [(rng.standard_normal(n) * 1e-2 * S).astype(np.float32) for n in (5, 20000, 70001)]
    g16 = [f16(g) for g in grads]
    exact = np.sqrt(sum(float(((O.convert(g, O.F16, O.F32).astype(np.float64) / S) ** 2).sum()) for g in g16))
    norm = O.grad_norm(g16, O.F16, float(np.float32(1.0 / S)))
    assert norm == pytest.approx(exact, rel=2e-6)


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
