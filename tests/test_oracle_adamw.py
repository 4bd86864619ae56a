"""Pins for the oracle's mixed-precision optimizer step and loss scaler (CPU).

The AdamW checks compare the oracle against closed forms of Adam under
constant or zero gradients and against the exponential-moving-average sums
of the moments, which a dropped bias correction, a coupled weight decay, a
misplaced eps or a swapped beta would each break.  The scaler is checked
against the hand-traced schedule and the defaults printed on the pages.
"""
import numpy as np
import pytest

from tests.conftest import golden

import oracle as O


def hp(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8, wd=0.01):
    return O.AdamwHp(lr, b1, b2, eps, wd)


def run(hparams, w0, grads_f32, S=1.0, g_fmt=O.F16, w16_fmt=O.F16):
    """Apply len(grads) steps; grads are given unscaled in float32 and scaled
    by S into the 16-bit grad format.  Returns the list of (w, m, v, w16)."""
    n = w0.size
    w = w0.astype(np.float32).copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    w16 = np.zeros(n, np.uint16)
    st = O.new_scaler_state(S)
    out = []
    for g in grads_f32:
        g16 = O.convert((np.asarray(g, np.float64) * S).astype(np.float32), O.F32, g_fmt)
        O.adamw_step(hparams, st, [(w, m, v, g16, w16)], g_fmt, w16_fmt)
        out.append((w.copy(), m.copy(), v.copy(), w16.copy()))
    return out, st


def test_constant_gradient_closed_form():
    # With g constant, bias-corrected m_hat = g and v_hat = g^2 exactly, so each
    # step moves w by lr * g / (|g| + eps), whatever the step count.
    lr = 1e-3
    g = np.array([0.5, -0.25, 2.0, -4.0], np.float32)  # exact in FP16
    w0 = np.array([1.0, -2.0, 0.5, 3.0], np.float32)
    traj, st = run(hp(lr=lr, wd=0.0), w0, [g] * 6, S=1024.0)
    for k, (w, m, v, _) in enumerate(traj, start=1):
        expect = w0.astype(np.float64) - k * lr * g / (np.abs(g) + 1e-8)
        np.testing.assert_allclose(w, expect, rtol=0, atol=4e-7 * k)
    assert st.step == 6


def test_decoupled_weight_decay_closed_form():
    # g = 0 leaves m = v = 0 and the Adam term 0 / (0 + eps) = 0, so only the
    # decoupled decay acts: w_k = w_0 * (1 - lr * wd)^k.  A decay folded into
    # the gradient would instead move w by about lr per step.
    lr, wd = 1e-2, 0.1
    w0 = np.array([1.0, -3.0, 0.25, 7.0], np.float32)
    traj, _ = run(hp(lr=lr, wd=wd), w0, [np.zeros(4, np.float32)] * 5)
    for k, (w, m, v, _) in enumerate(traj, start=1):
        np.testing.assert_allclose(w, w0 * (1 - lr * wd) ** k, rtol=1e-6)
        assert not m.any() and not v.any()


def test_eps_is_added_after_the_square_root():
    # g = eps: update = lr * g / (|g| + eps) = lr / 2 on the first step.
    # eps inside the square root would give lr * 1e-8 / sqrt(1e-16 + 1e-8) ~ 1e-4 lr.
    eps = 1e-4
    g = np.full(4, eps, np.float32)
    w0 = np.zeros(4, np.float32)
    (w, _, _, _), = run(hp(lr=1e-3, eps=eps, wd=0.0), w0, [g], S=1.0, g_fmt=O.BF16)[0][:1]
    gb = O.convert(O.convert(g, O.F32, O.BF16), O.BF16, O.F32).astype(np.float64)
    np.testing.assert_allclose(w, -1e-3 * gb / (gb + eps), rtol=1e-6)


def test_moments_match_ema_sums():
    # m_t = (1-b1) sum_i b1^(t-i) g_i and v_t = (1-b2) sum_i b2^(t-i) g_i^2
    b1, b2 = 0.8, 0.95
    rng = np.random.default_rng(0)
    gs = [O.convert(O.convert(rng.standard_normal(8).astype(np.float32), O.F32, O.F16), O.F16, O.F32)
          for _ in range(7)]
    traj, _ = run(hp(b1=b1, b2=b2, wd=0.0), np.zeros(8, np.float32), gs)
    for t in range(1, 8):
        G = np.array(gs[:t], np.float64)
        wts1 = (1 - b1) * b1 ** np.arange(t - 1, -1, -1)
        wts2 = (1 - b2) * b2 ** np.arange(t - 1, -1, -1)
        np.testing.assert_allclose(traj[t - 1][1], wts1 @ G, rtol=2e-6, atol=1e-7)
        np.testing.assert_allclose(traj[t - 1][2], wts2 @ (G * G), rtol=2e-6, atol=1e-7)


def test_unscale_is_exact_for_power_of_two_scale():
    S = 65536.0
    st = O.new_scaler_state(S)
    s = O.adamw_begin(hp(), st, 0)
    assert s.inv_scale == 1.0 / S
    g = np.array([2.0**-25, 1e-4, -3e-3], np.float32)
    g16 = O.convert(g * np.float32(S), O.F32, O.F16)
    back = O.convert(g16, O.F16, O.F32) * np.float32(s.inv_scale)
    # 2^-25 is below FP16's range but survives the scaled round trip
    assert back[0] == np.float32(2.0**-25)


def test_working_copy_is_rounded_from_master():
    rng = np.random.default_rng(1)
    w0 = (rng.standard_normal(1000) * 0.02).astype(np.float32)
    gs = [rng.standard_normal(1000).astype(np.float32) * 1e-3 for _ in range(3)]
    for fmt in (O.F16, O.BF16):
        traj, _ = run(hp(), w0, gs, S=1.0, w16_fmt=fmt)
        for (w, _, _, w16) in traj:
            ref = w.astype(np.float16).view(np.uint16) if fmt == O.F16 else \
                __import__("torch").from_numpy(w).bfloat16().view(__import__("torch").int16).numpy().view(np.uint16)
            np.testing.assert_array_equal(w16, ref)


def test_lost_update_fp16_versus_fp32_master():
    # An update of lr = 2^-13 on w = 1 is below 2^-11 * w: in pure FP16 it is
    # lost every step, while the FP32 master accumulates it and the FP16 copy
    # moves once the accumulated change reaches half an FP16 spacing.
    lr = 2.0**-13
    g = np.array([1.0], np.float32)
    traj, _ = run(hp(lr=lr, wd=0.0), np.ones(1, np.float32), [g] * 4)
    L = O.lib()
    w16_pure = L.orc_f32_to_f16(1.0)
    for k in range(4):
        upd = lr * 1.0 / (1.0 + 1e-8)
        w16_pure = L.orc_f32_to_f16(np.float32(L.orc_f16_to_f32(w16_pure) - upd))
        assert w16_pure == L.orc_f32_to_f16(1.0)
    w_master = [t[0][0] for t in traj]
    np.testing.assert_allclose(w_master, [1 - k * lr for k in range(1, 5)], rtol=0, atol=1e-9)
    w16_master = [int(t[3][0]) for t in traj]
    # 1 - 2^-13 and 1 - 2^-12 round back to 1.0; 1 - 3*2^-13 and 1 - 2^-11 reach 0x3BFF
    assert w16_master == [0x3C00, 0x3C00, 0x3BFF, 0x3BFF]


def test_skipped_step_writes_nothing():
    w = np.ones(4, np.float32)
    m = np.full(4, 0.5, np.float32)
    v = np.full(4, 0.25, np.float32)
    w16 = np.full(4, 7, np.uint16)
    g = O.convert(np.array([1, 2, np.inf, 3], np.float32), O.F32, O.F16)
    st = O.new_scaler_state()
    found, _, _ = O.adamw_step(hp(), st, [(w, m, v, g, w16)], O.F16, O.F16)
    assert found == 1 and st.found_inf == 1 and st.step == 0
    assert st.beta1_pow == 1.0 and st.beta2_pow == 1.0
    assert (w == 1).all() and (m == 0.5).all() and (v == 0.25).all() and (w16 == 7).all()


@pytest.mark.parametrize("fmt,bad", [(O.F16, [0x7C00, 0xFC00, 0x7E00, 0x7C01]),
                                     (O.BF16, [0x7F80, 0xFF80, 0x7FC0, 0x7F81])])
def test_nonfinite_detection(fmt, bad):
    g = np.zeros(1000, np.uint16)
    g[:] = 0x7BFF if fmt == O.F16 else 0x7F7F  # largest finite
    assert O.nonfinite_any(g, fmt) == 0
    for b in bad:
        for pos in (0, 517, 999):
            h = g.copy()
            h[pos] = b
            assert O.nonfinite_any(h, fmt) == 1


def test_scaler_trajectory_hand_traced():
    t = golden("scaler_trajectory_tiny.json")
    cfg = O.ScalerCfg(t["growth_factor"], t["backoff_factor"], t["growth_interval"], 1)
    st = O.new_scaler_state(t["init_scale"])
    hp_ = hp()
    for k, step in enumerate(t["steps"]):
        assert st.scale == t["scale_used"][k]
        O.adamw_begin(hp_, st, t["found_inf"][k])
        O.loss_scale_update(st, cfg)
        assert st.growth_tracker == t["tracker_after"][k]
    assert st.scale == t["final_scale"]
    assert st.step == t["applied_steps"]
    assert st.skipped == t["skipped_steps"]
    # beta powers advance only on applied steps, from the float32 beta1
    assert st.beta1_pow == pytest.approx(float(np.float32(0.9)) ** 10, rel=1e-12)


def test_scaler_defaults_from_pages():
    g = golden("gradscaler.json")
    cfg = O.ScalerCfg(g["growth_factor"], g["backoff_factor"], g["growth_interval"], 1)
    st = O.new_scaler_state(g["init_scale"])
    assert st.scale == 2.0**16
    for _ in range(g["growth_interval"] - 1):
        O.loss_scale_update(st, cfg)
    assert st.scale == 65536.0
    O.loss_scale_update(st, cfg)
    assert st.scale == 131072.0 and st.growth_tracker == 0
    st.found_inf = 1
    O.loss_scale_update(st, cfg)
    assert st.scale == 65536.0 and st.skipped == 1


def test_scale_never_grows_to_infinity_and_has_no_floor():
    cfg = O.ScalerCfg(2.0, 0.5, 1, 1)
    st = O.new_scaler_state(float(np.float32(2.0**127)))
    O.loss_scale_update(st, cfg)
    assert st.scale == 2.0**127
    st = O.new_scaler_state(1.0)
    st.found_inf = 1
    for _ in range(3):
        O.loss_scale_update(st, cfg)
    assert st.scale == 0.125


def test_disabled_scaler_is_inert():
    cfg = O.ScalerCfg(2.0, 0.5, 1, 0)
    st = O.new_scaler_state(8.0)
    st.found_inf = 1
    O.loss_scale_update(st, cfg)
    assert st.scale == 8.0 and st.skipped == 0
