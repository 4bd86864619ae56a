"""The mixed-precision recipe's own claims, run through the kernels.

FP32 master weights keep updates smaller than the 16-bit spacing ([MPT-es]
"La receta de precisión mixta"; [MPT-ko] "FP32 마스터 가중치": near 1.0 an
FP16 update below 2^-11 is lost), so the working copy moves once enough of them
have accumulated; and the dynamic loss scale backs off on every overflowing
step without a floor ([MPT-es] "Limitaciones": a scale collapsing towards 1 is a
symptom to watch, not something the schedule prevents)."""
import numpy as np
import pytest
import torch

import oracle as O

import mixed_precision_numerics_gb300 as M  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def test_fp32_master_keeps_updates_below_the_fp16_spacing():
    n = 4096
    w = torch.ones(n, dtype=torch.float32, device="cuda")
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    w16 = torch.zeros(n, dtype=torch.float16, device="cuda")
    g = torch.full((n,), -1.0, dtype=torch.float16, device="cuda")  # constant gradient, scale 1
    lr = 2.0 ** -13  # Adam's step for a constant gradient is lr: a quarter of the FP16 spacing at 1.0
    hp = M.AdamwHparams(lr, 0.9, 0.999, 1e-8, 0.0)
    st = M.new_scaler_state(1.0)
    ow, om, ov, ow16 = np.ones(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    ohp, ost = O.AdamwHp(lr, 0.9, 0.999, 1e-8, 0.0), O.new_scaler_state(1.0)
    og = np.full(n, np.float16(-1.0)).view(np.uint16)
    moved_at = None
    for k in range(1, 17):
        M.mp_adamw_step([M.Param(w, m, v, g, w16)], hp, st)
        O.adamw_step(ohp, ost, [(ow, om, ov, og, ow16)], O.F16, O.F16)
        torch.cuda.synchronize()
        gw = w.cpu().numpy()
        np.testing.assert_array_equal(gw.view(np.uint32), ow.view(np.uint32))
        np.testing.assert_array_equal(w16.cpu().numpy().view(np.uint16), ow16)
        # an FP16 master would never move: 1.0 + lr rounds back to 1.0
        assert np.float16(np.float16(1.0) + np.float16(lr)) == np.float16(1.0)
        if moved_at is None and w16[0].item() != 1.0:
            moved_at = k
    assert gw[0] > 1.0 + 2.0 ** -11  # the FP32 master accumulated the small steps
    assert moved_at is not None and moved_at > 1  # the working copy moved once they added up


def test_loss_scale_backs_off_without_a_floor():
    n = 1024
    w = torch.zeros(n, dtype=torch.float32, device="cuda")
    g = torch.zeros(n, dtype=torch.float16, device="cuda")
    g[7] = float("inf")
    p = M.Param(w, torch.zeros_like(w), torch.zeros_like(w), g, torch.zeros(n, dtype=torch.float16, device="cuda"))
    hp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    st, ost = M.new_scaler_state(65536.0), O.new_scaler_state(65536.0)
    cfg, ocfg = M.ScalerCfg(2.0, 0.5, 2000, 1), O.ScalerCfg(2.0, 0.5, 2000, 1)
    ohp = O.AdamwHp(1e-3, 0.9, 0.999, 1e-8, 0.0)
    for k in range(24):
        M.mp_adamw_step([p], hp, st)
        M.loss_scale_update(st, cfg)
        O.adamw_begin(ohp, ost, 1)  # the oracle's step with found_inf set
        O.loss_scale_update(ost, ocfg)
    torch.cuda.synchronize()
    s = M.read_scaler_state(st)
    assert s.scale == ost.scale == 65536.0 * 2.0 ** -24  # halved 24 times, below 1 with no floor
    assert s.skipped == ost.skipped == 24 and s.step == 0
    assert not w.any()  # every step was skipped: nothing written
