"""GPU parity: mx_quantize (MXFP8 / MXFP4, 32-element blocks with UE8M0
scales) against the oracle, bit for bit: codes, scale bytes and the BF16
dequantised copy."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import synth.workloads as W
from tests.gpu_util import to_dev, to_host

import mixed_precision_numerics_gb300 as M  # noqa: E402

pytestmark = pytest.mark.gpu
XFMT = {torch.float32: O.F32, torch.float16: O.F16, torch.bfloat16: O.BF16}
EFMT = {M.MP_E4M3: O.E4M3, M.MP_E5M2: O.E5M2, M.MP_E2M1: O.E2M1, M.MP_E2M3: O.E2M3, M.MP_E3M2: O.E3M2}


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def gpu_mx(xt, elem, want_dq=True):
    rows, cols = xt.shape
    nbytes = rows * cols // (2 if elem == M.MP_E2M1 else 1)
    codes = torch.full((nbytes,), 0xCC, dtype=torch.uint8, device="cuda")
    sc = torch.full((rows, cols // 32), 0xCC, dtype=torch.uint8, device="cuda")
    dq = torch.full((rows, cols), -7.0, dtype=torch.bfloat16, device="cuda") if want_dq else None
    M.mx_quantize(xt, codes, sc, elem, dq)
    torch.cuda.synchronize()
    return (codes.cpu().numpy().reshape(rows, -1), sc.cpu().numpy(),
            dq.view(torch.int16).cpu().numpy().view(np.uint16) if want_dq else None)


def make_input(rows, cols, dtype, seed):
    xf = synth.fill(synth.recipe(110 + seed, rows, 2.0, 0.02, 60.0, synth.OUT_SCALE), synth.F32, rows * cols,
                    shape=(rows, cols))
    flat = xf.reshape(-1)
    if flat.size >= 512:
        flat[[5, 40, 77]] = [np.inf, np.nan, -np.inf]
        flat[256:320] = 0.0                       # two all-zero blocks
        flat[320:352] *= np.float32(2.0**-135)    # a block of tiny values (subnormal in FP32)
        flat[352:384] *= np.float32(2.0**100)     # a block near the top of the range
        flat[384:416] = -0.0
    if dtype == torch.float32:
        return xf, to_dev(xf)
    x = O.convert(xf, O.F32, XFMT[dtype])
    return x, to_dev(x, dtype)


def check(x, xfmt, xt, elem):
    c, s, d = gpu_mx(xt, elem)
    rc, rs, rd = O.mx_quantize(x, xfmt, EFMT[elem])
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(c, rc)
    np.testing.assert_array_equal(d, rd)


@pytest.mark.parametrize("elem", [M.MP_E4M3, M.MP_E5M2, M.MP_E2M1, M.MP_E2M3, M.MP_E3M2])
@pytest.mark.parametrize("shape", [(1, 32), (3, 96), (7, 544), (129, 1056), (257, 4096)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_small_shapes(elem, shape, dtype):
    x, xt = make_input(*shape, dtype, shape[0])
    check(x, XFMT[dtype], xt, elem)


def test_without_dequant():
    x, xt = make_input(64, 512, torch.bfloat16, 3)
    c, s, _ = gpu_mx(xt, M.MP_E2M1, want_dq=False)
    rc, rs, _ = O.mx_quantize(x, O.BF16, O.E2M1, want_dequant=False)
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(c, rc)


@pytest.mark.parametrize("elem", [M.MP_E2M1, M.MP_E4M3, M.MP_E2M3, M.MP_E3M2])
def test_full_size_activation(elem):
    c = W.NVFP4_RNE
    x = torch.empty((c.act_rows, c.act_cols), dtype=torch.bfloat16, device="cuda")
    synth.fill_device(c.act_recipe(), synth.BF16, x)
    gc, gs, gd = gpu_mx(x, elem)
    rc, rs, rd = O.mx_quantize(to_host(x, np.uint16).reshape(c.act_rows, c.act_cols), O.BF16, EFMT[elem])
    assert np.array_equal(gs, rs)
    assert np.array_equal(gc, rc)
    assert np.array_equal(gd, rd)


def test_full_size_gradient_e5m2():
    c = W.NVFP4_GRAD
    x = torch.empty((c.rows, c.cols), dtype=torch.bfloat16, device="cuda")
    synth.fill_device(c.recipe(), synth.BF16, x)
    gc, gs, _ = gpu_mx(x, M.MP_E5M2, want_dq=False)
    rc, rs, _ = O.mx_quantize(to_host(x, np.uint16).reshape(c.rows, c.cols), O.BF16, O.E5M2, want_dequant=False)
    assert np.array_equal(gs, rs)
    assert np.array_equal(gc, rc)


def test_fp6_every_bf16_magnitude_on_a_unit_scale():
    """Blocks whose maximum is 2^emax (scale 2^0) carry every BF16 value in
    [-2^(emax+1), 2^(emax+1)): the FP6 codes are the format's own rounding."""
    for elem, emax in ((M.MP_E2M3, 2), (M.MP_E3M2, 4)):
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        v = O.convert(bits, O.BF16, O.F32)
        v = v[np.isfinite(v) & (np.abs(v) < 2.0 ** (emax + 1))]
        n = -(-v.size // 31) * 31
        v = np.concatenate([v, np.zeros(n - v.size, np.float32)]).reshape(-1, 31)
        x = np.concatenate([np.full((v.shape[0], 1), 2.0 ** emax, np.float32), v], axis=1)
        xb = O.convert(x, O.F32, O.BF16)
        c, s, d = gpu_mx(to_dev(xb, torch.bfloat16), elem)
        rc, rs, rd = O.mx_quantize(xb, O.BF16, EFMT[elem])
        assert (rs == 127).all()
        np.testing.assert_array_equal(c, rc)
        np.testing.assert_array_equal(d, rd)


def test_errors():
    x = torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros(4 * 48, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MpError) as e:
        M.mx_quantize(x, codes, sc, M.MP_E4M3)
    assert e.value.status == M.MP_ESHAPE
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(M.MpError) as e:
        M.mx_quantize(x, codes, sc, M.MP_BF16)
    assert e.value.status == M.MP_EINVAL
    with pytest.raises(M.MpError) as e:
        M.mx_quantize(x, codes[1:], sc, M.MP_E4M3)
    assert e.value.status == M.MP_EALIGN
    # empty input: nothing launched, nothing written
    n0 = M.mp_launch_count()
    M.mx_quantize(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"), codes, sc, M.MP_E2M1)
    assert M.mp_launch_count() == n0
