"""CPU tests of the host side: the C ABI library loads and exports every
entry point declared in include/mpnum.h, its structs match the binding, its
host-only helpers and argument validation work without a GPU, and the
parallel oracle driver used by the GPU tests equals the plain oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O
import synth
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mpnum.h")


@pytest.fixture(scope="module")
def M():
    import __graft_entry__

    __graft_entry__._package_builder().build()
    import mixed_precision_numerics_gb300 as pkg

    return pkg


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MP_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(M):
    names = declared_functions()
    assert {"mp_adamw_step", "loss_scale_update", "fp8_cast_delayed", "nvfp4_quantize", "rht16"} <= set(names)
    raw = ctypes.CDLL(M.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in mpnum.h but not exported"


def test_struct_layouts(M):
    st = M.ScalerState()
    M.lib.mp_scaler_state_init(ctypes.byref(st), 65536.0)
    assert st.scale == 65536.0 and st.beta1_pow == 1.0 and st.beta2_pow == 1.0 and st.step == 0
    assert ctypes.sizeof(M.ScalerState) == 88 and M.ScalerState.internal_found.offset == 56
    m = M.Fp8Meta()
    M.lib.mp_fp8_meta_init(ctypes.byref(m))
    assert (m.scale, m.scale_inv, m.amax, m.pos) == (1.0, 1.0, 0.0, 0)
    assert M.nvfp4_workspace_size() >= 8
    for s in (0, -1, -2, -3, -4, -5):
        assert M.mp_status_str(s)


def test_argument_validation_without_gpu(M):
    L = M.lib
    launched0 = M.mp_launch_count()
    hp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    assert L.mp_adamw_step(None, 0, 9, M.MP_F16, ctypes.byref(hp), 16, None, 0, None) == M.MP_EINVAL
    assert L.mp_adamw_step(None, -1, M.MP_F16, M.MP_F16, ctypes.byref(hp), 16, None, 0, None) == M.MP_EINVAL
    assert L.mp_adamw_step(None, 0, M.MP_F16, M.MP_F16, ctypes.byref(hp), 12, None, 0, None) == M.MP_EALIGN
    bad = M.AdamwHparams(float("nan"), 0.9, 0.999, 1e-8, 0.0)
    assert L.mp_adamw_step(None, 0, M.MP_F16, M.MP_F16, ctypes.byref(bad), 16, None, 0, None) == M.MP_EINVAL
    p = (M.MpParam * 1)(M.MpParam(16, 16, 16, 24, 16, 5))
    assert L.mp_adamw_step(p, 1, M.MP_F16, M.MP_F16, ctypes.byref(hp), 16, None, 0, None) == M.MP_EALIGN
    # clipping needs a workspace of mp_adamw_workspace_size bytes
    clip = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1.0)
    p = (M.MpParam * 1)(M.MpParam(16, 16, 16, 16, 16, 40000))
    need = 32 * 8 + 4 * 3  # binary64 warp partials + one binary32 sum per 16384-element tile
    assert L.mp_adamw_workspace_size(p, 1) == need
    assert L.mp_adamw_workspace_size(None, 0) == 32 * 8
    assert L.mp_adamw_step(p, 1, M.MP_F16, M.MP_F16, ctypes.byref(clip), 16, None, 0, None) == M.MP_EWORKSPACE
    assert L.mp_adamw_step(p, 1, M.MP_F16, M.MP_F16, ctypes.byref(clip), 16, 16, need - 1, None) == M.MP_EWORKSPACE
    assert L.mp_adamw_step(p, 1, M.MP_F16, M.MP_F16, ctypes.byref(clip), 16, 20, need, None) == M.MP_EALIGN
    neg = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0, -1.0)
    assert L.mp_adamw_step(p, 1, M.MP_F16, M.MP_F16, ctypes.byref(neg), 16, None, 0, None) == M.MP_EINVAL
    cfg = M.ScalerCfg(2.0, 0.5, 0, 1)
    assert L.loss_scale_update(16, ctypes.byref(cfg), None) == M.MP_EINVAL
    assert L.fp8_cast_delayed(16, M.MP_BF16, 10, 16, M.MP_F16, 16, 16, 4, 1.0, 0, None) == M.MP_EINVAL
    assert L.fp8_cast_delayed(16, M.MP_BF16, 10, 16, M.MP_E4M3, 16, 16, 0, 1.0, 0, None) == M.MP_EINVAL
    assert L.fp8_cast_delayed(16, M.MP_BF16, 10, 16, M.MP_E4M3, 16, 16, 4, 0.0, 0, None) == M.MP_EINVAL
    assert L.fp8_cast_delayed(16, M.MP_BF16, 10, 16, M.MP_E4M3, 16, 16, 4, 1.0, 2, None) == M.MP_EINVAL
    assert L.fp8_cast_delayed(8, M.MP_BF16, 10, 16, M.MP_E4M3, 16, 16, 4, 1.0, 0, None) == M.MP_EALIGN
    c = L.fp8_cast_delayed_count
    assert c(16, M.MP_BF16, 10, 16, M.MP_E4M3, 16, 16, 4, 1.0, 0, None, None) == M.MP_EINVAL
    assert c(16, M.MP_BF16, 10, 16, M.MP_E4M3, 16, 16, 4, 1.0, 0, 12, None) == M.MP_EALIGN
    assert c(16, M.MP_BF16, 10, 16, M.MP_F16, 16, 16, 4, 1.0, 0, 16, None) == M.MP_EINVAL
    b = L.fp8_quantize_blockwise
    assert b(16, M.MP_BF16, 4, 128, 64, 64, 16, M.MP_E4M3, 16, None) == M.MP_ESHAPE
    assert b(16, M.MP_BF16, 4, 120, 1, 128, 16, M.MP_E4M3, 16, None) == M.MP_ESHAPE
    assert b(16, M.MP_BF16, 4, 128, 1, 128, 16, M.MP_E4M3, 18, None) == M.MP_EALIGN
    t = L.fp8_cast_transpose_delayed
    assert t(16, M.MP_BF16, 16, 24, 16, 16, M.MP_E4M3, 16, 16, 4, 1.0, 0, None) == M.MP_ESHAPE
    assert t(16, M.MP_BF16, 16, 32, 16, 8, M.MP_E4M3, 16, 16, 4, 1.0, 0, None) == M.MP_EALIGN
    e = L.e2m1_stochastic_round
    assert e(16, 16, -1, 16, None) == M.MP_EINVAL
    assert e(16, None, 4, 16, None) == M.MP_EINVAL
    assert e(16, 16, 4, 24, None) == M.MP_EALIGN
    assert e(None, None, 0, None, None) == M.MP_OK
    q = L.nvfp4_quantize
    assert q(16, 2, 24, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, 16, 256, None) == M.MP_ESHAPE
    assert q(16, 8, 32, 1, 0, 0, 0, 0, 16, 16, 16, 16, None, 16, 256, None) == M.MP_ESHAPE
    assert q(16, 2, 32, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, 16, 4, None) == M.MP_EWORKSPACE
    assert q(8, 2, 32, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, 16, 256, None) == M.MP_EALIGN
    # the no-alloc quantiser checks its arguments before it touches CUDA at
    # all: here, with no GPU, every argument error is reported as such
    qa = L.nvfp4_quantize_noalloc
    assert qa(16, 2, 24, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, None) == M.MP_ESHAPE
    assert qa(16, 8, 32, 1, 0, 0, 0, 0, 16, 16, 16, 16, None, None) == M.MP_ESHAPE
    assert qa(None, 2, 32, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, None) == M.MP_EINVAL
    assert qa(16, -1, 32, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, None) == M.MP_EINVAL
    assert qa(8, 2, 32, 0, 0, 0, 0, 0, 16, 16, 16, 16, None, None) == M.MP_EALIGN
    assert qa(16, 2, 32, 0, 0, 0, 0, 0, 16, 16, 16, 16, 24, None) == M.MP_EALIGN
    assert L.rht16(16, 2, 40, 0, 16, M.MP_F32, None) == M.MP_ESHAPE
    assert L.rht16(16, 2, 32, 0, 16, M.MP_E4M3, None) == M.MP_EINVAL
    mx = L.mx_quantize
    assert mx(16, M.MP_BF16, 2, 48, M.MP_E4M3, 16, 16, None, None) == M.MP_ESHAPE
    assert mx(16, M.MP_BF16, 2, 64, M.MP_F16, 16, 16, None, None) == M.MP_EINVAL
    assert mx(16, M.MP_E4M3, 2, 64, M.MP_E2M1, 16, 16, None, None) == M.MP_EINVAL
    assert mx(16, M.MP_BF16, 2, 64, 8, 16, 16, None, None) == M.MP_EINVAL
    assert mx(16, M.MP_BF16, 2, 48, M.MP_E3M2, 16, 16, None, None) == M.MP_ESHAPE
    assert mx(16, M.MP_BF16, 2, 64, M.MP_E2M1, 8, 16, None, None) == M.MP_EALIGN
    assert mx(16, M.MP_BF16, 2, 64, M.MP_E2M1, 16, 16, 40, None) == M.MP_EALIGN
    assert mx(None, M.MP_BF16, 2, 64, M.MP_E2M1, 16, 16, None, None) == M.MP_EINVAL
    assert mx(None, M.MP_BF16, 0, 64, M.MP_E2M1, None, None, None, None) == M.MP_OK
    assert M.mp_launch_count() == launched0  # every rejected call returned before launching


@pytest.mark.parametrize("b2,sr,rht", [(False, False, False), (False, True, True), (True, False, True), (True, True, False)])
def test_parallel_oracle_driver_equals_plain_oracle(b2, sr, rht):
    from tests.gpu_util import nvfp4_oracle

    x = synth.fill(synth.recipe(3, 0, 1.0, 0.01, 30.0, synth.OUT_SCALE), synth.BF16, 400 * 320, shape=(400, 320))
    x = x[:384] if b2 else x
    a = nvfp4_oracle(x, b2, sr, 42, rht, 0x1234)
    b = O.nvfp4_quantize(x, b2, sr, 42, rht, 0x1234)
    for u, v in zip(a, b):
        if isinstance(u, np.ndarray):
            np.testing.assert_array_equal(u, v)
        else:
            assert u == v


def test_generator_is_deterministic_and_reproducible_by_index():
    r = synth.recipe(9, 3, 2.0, 0.01, 10.0, synth.OUT_SCALE)
    a = synth.fill(r, synth.F16, 5000)
    b = synth.fill(r, synth.F16, 5000)
    np.testing.assert_array_equal(a, b)
    idx = np.array([0, 17, 4999])
    np.testing.assert_array_equal(synth.fill_at(r, synth.F16, idx), a[idx])
    np.testing.assert_array_equal(synth.fill(r, synth.F16, 10, start=17), a[17:27])


# ---- the Python binding checks tensors before their pointers cross the ABI ----------


def test_binding_rejects_host_tensors_before_any_launch():
    import torch

    import mixed_precision_numerics_gb300 as M

    x = torch.zeros(64, dtype=torch.bfloat16)
    y = torch.zeros(64, dtype=torch.uint8)
    n0 = M.mp_launch_count()
    with pytest.raises(ValueError, match="CUDA tensor"):
        M.fp8_cast_delayed(x, y, M.MP_E4M3, torch.zeros(32, dtype=torch.uint8), torch.zeros(4))
    with pytest.raises(ValueError, match="CUDA tensor"):
        M.mx_quantize(x.view(2, 32), y, torch.zeros(2, dtype=torch.uint8), M.MP_E4M3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        M.fp8_quantize_blockwise(x.view(1, 64), y, torch.zeros(1), 1, 128)
    with pytest.raises(ValueError, match="CUDA tensor"):
        M.nvfp4_quantize(x.view(4, 16), y, y, torch.zeros(1), torch.zeros(1, dtype=torch.int32),
                         torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        M.rht16(x.view(4, 16), torch.zeros(64), 0x5A5A)
    w = torch.zeros(8)
    g = torch.zeros(8, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        M.mp_adamw_step([M.Param(w, w, w, g, g)], M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0),
                        torch.zeros(88, dtype=torch.uint8))
    assert M.mp_launch_count() == n0


def test_binding_size_rule_follows_the_alignment_rule():
    """The size check steps aside where the library itself rejects the pointer
    (misaligned), and applies to an aligned pointer."""
    import mixed_precision_numerics_gb300 as M

    class FakeCuda:
        is_cuda = True

        def __init__(self, nbytes, ptr, device):
            self._n, self._p, self.device = nbytes, ptr, device

        def is_contiguous(self):
            return True

        def numel(self):
            return self._n

        def element_size(self):
            return 1

        def data_ptr(self):
            return self._p

    import torch

    dev = torch.device("cuda", 0)
    ref = FakeCuda(64, 4096, dev)
    M._dev(FakeCuda(10, 4096 + 3, dev), "y", 64, like=ref)  # misaligned: left to the library
    with pytest.raises(ValueError, match="bytes, the call needs 64"):
        M._dev(FakeCuda(10, 4096, dev), "y", 64, like=ref)
    with pytest.raises(ValueError, match="the call runs on"):
        M._dev(FakeCuda(64, 4096, torch.device("cuda", 1)), "y", 64, like=ref)
