"""GPU parity: fp8_quantize_blockwise (fine-grained FP8, online 1x128 and
128x128 block scales) against the oracle, bit for bit."""
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


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def gpu_blockwise(xt, br, bc, fmt=M.MP_E4M3):
    rows, cols = xt.shape
    y = torch.full((rows, cols), 0xCC, dtype=torch.uint8, device="cuda")
    sc = torch.full((-(-rows // br), -(-cols // bc)), -7.0, dtype=torch.float32, device="cuda")
    M.fp8_quantize_blockwise(xt, y, sc, br, bc, fmt)
    torch.cuda.synchronize()
    return y.cpu().numpy(), sc.cpu().numpy()


def make_input(rows, cols, dtype, seed):
    xf = synth.fill(synth.recipe(90 + seed, rows, 2.0, 0.02, 60.0, synth.OUT_SCALE), synth.F32, rows * cols,
                    shape=(rows, cols))
    if rows * cols >= 400:
        xf.reshape(-1)[[5, 9, 13]] = [np.inf, np.nan, -0.0]
        xf.reshape(-1)[256:384] = 0.0
    if dtype == torch.float32:
        return xf, to_dev(xf)
    f = XFMT[dtype]
    x = O.convert(xf, O.F32, f)
    return x, to_dev(x, dtype)


@pytest.mark.parametrize("block", [(1, 128), (128, 128)])
@pytest.mark.parametrize("shape", [(1, 128), (3, 256), (5, 144), (130, 272), (257, 1040)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_small_shapes(block, shape, dtype):
    x, xt = make_input(*shape, dtype, shape[0])
    y, sc = gpu_blockwise(xt, *block)
    ry, rsc = O.fp8_quantize_blockwise(x, XFMT[dtype], *block)
    np.testing.assert_array_equal(sc.view(np.uint32), rsc.view(np.uint32))
    np.testing.assert_array_equal(y, ry)


def test_e5m2_blocks():
    x, xt = make_input(200, 384, torch.bfloat16, 7)
    for block in ((1, 128), (128, 128)):
        y, sc = gpu_blockwise(xt, *block, M.MP_E5M2)
        ry, rsc = O.fp8_quantize_blockwise(x, O.BF16, *block, O.E5M2)
        np.testing.assert_array_equal(sc.view(np.uint32), rsc.view(np.uint32))
        np.testing.assert_array_equal(y, ry)


def test_full_size_activations_1x128():
    c = W.FP8
    x = torch.empty((c.rows, c.cols), dtype=torch.bfloat16, device="cuda")
    synth.fill_device(c.act_recipe(5), synth.BF16, x)
    y, sc = gpu_blockwise(x, 1, 128)
    ry, rsc = O.fp8_quantize_blockwise(to_host(x, np.uint16).reshape(c.rows, c.cols), O.BF16, 1, 128)
    np.testing.assert_array_equal(sc.view(np.uint32), rsc.view(np.uint32))
    assert np.array_equal(y, ry)


def test_full_size_weights_128x128():
    c = W.NVFP4_RNE
    x = torch.empty((c.w_rows, c.w_cols), dtype=torch.bfloat16, device="cuda")
    synth.fill_device(c.w_recipe(), synth.BF16, x)
    y, sc = gpu_blockwise(x, 128, 128)
    ry, rsc = O.fp8_quantize_blockwise(to_host(x, np.uint16).reshape(c.w_rows, c.w_cols), O.BF16, 128, 128)
    np.testing.assert_array_equal(sc.view(np.uint32), rsc.view(np.uint32))
    assert np.array_equal(y, ry)


def test_shape_errors():
    x = torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(96, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(4, device="cuda")
    for br, bc in ((1, 128), (64, 64)):
        with pytest.raises(M.MpError) as e:
            M.fp8_quantize_blockwise(x, y, sc, br, bc)
        assert e.value.status == M.MP_ESHAPE


def test_empty_tensor_launches_nothing():
    n0 = M.mp_launch_count()
    for br in (1, 128):
        x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
        M.fp8_quantize_blockwise(x, torch.empty(0, dtype=torch.uint8, device="cuda"),
                                 torch.empty(0, device="cuda"), br, 128)
    assert M.mp_launch_count() == n0


@pytest.mark.parametrize("shape,dtype", [((4000, 7184), torch.bfloat16), ((3000, 4112), torch.float32),
                                         ((2049, 6160), torch.float16)])
@pytest.mark.parametrize("block", [(1, 128), (128, 128)])
def test_many_blocks_per_cta_ragged(shape, dtype, block):
    """Enough 128 x 128 boxes that every CTA's ring of tile copies wraps several
    times, with partial boxes (and 1 x 128 tiles) on the right and bottom edges."""
    x, xt = make_input(*shape, dtype, 3)
    for fmt, ofmt in ((M.MP_E4M3, O.E4M3), (M.MP_E5M2, O.E5M2)):
        y, sc = gpu_blockwise(xt, *block, fmt)
        ry, rsc = O.fp8_quantize_blockwise(x, XFMT[dtype], *block, ofmt)
        np.testing.assert_array_equal(sc.view(np.uint32), rsc.view(np.uint32))
        assert np.array_equal(y, ry)
    assert M.mp_wait_failures() == 0


def test_no_wait_gave_up():
    assert M.mp_wait_failures() == 0


def test_random_shape_sweep_against_the_oracle():
    """Seeded random shapes (cols % 16 == 0, rows anything; a multiple of 16 for
    the transposed cast) in every input type and both formats, from one partial
    box up to several boxes per CTA: the tile casts match the oracle bit for bit."""
    rng = np.random.default_rng(2026)
    dts = [torch.bfloat16, torch.float16, torch.float32]
    for i in range(24):
        rows = int(rng.choice([int(rng.integers(1, 130)), int(rng.integers(130, 1500))]))
        cols = 16 * int(rng.integers(1, 200))
        dtype = dts[i % 3]
        fmt, ofmt = ((M.MP_E4M3, O.E4M3), (M.MP_E5M2, O.E5M2))[i % 2]
        x, xt = make_input(rows, cols, dtype, 200 + i)
        for br in (1, 128):
            y, sc = gpu_blockwise(xt, br, 128, fmt)
            ry, rsc = O.fp8_quantize_blockwise(x, XFMT[dtype], br, 128, ofmt)
            np.testing.assert_array_equal(sc.view(np.uint32), rsc.view(np.uint32), err_msg=f"{rows}x{cols} {br}")
            assert np.array_equal(y, ry), f"{rows}x{cols} {dtype} block {br}"
        r16 = max(16, rows // 16 * 16)
        xs, xts = make_input(r16, cols, dtype, 300 + i)
        meta, hist = M.new_fp8_meta(), torch.zeros(4, device="cuda")
        y = torch.empty(r16 * cols, dtype=torch.uint8, device="cuda")
        yt = torch.empty(r16 * cols, dtype=torch.uint8, device="cuda")
        M.fp8_cast_transpose_delayed(xts, y, yt, fmt, meta, hist)
        torch.cuda.synchronize()
        ref = O.fp8_cast_array(xs, XFMT[dtype], ofmt, 1.0).reshape(r16, cols)
        assert np.array_equal(y.cpu().numpy().reshape(r16, cols), ref), f"transpose {r16}x{cols} {dtype}"
        assert np.array_equal(yt.cpu().numpy().reshape(cols, r16), ref.T), f"transpose^T {r16}x{cols} {dtype}"
    assert M.mp_wait_failures() == 0
