"""No call writes outside its outputs: every output buffer sits between two
guard bands filled with a sentinel, and after each call on ragged shapes the
bands are unchanged (an out-of-bounds check that needs no sanitizer)."""
import numpy as np
import pytest
import torch

import synth

import mixed_precision_numerics_gb300 as M  # noqa: E402

pytestmark = pytest.mark.gpu
BAND = 4096  # bytes on each side, a multiple of 16 so the interior stays aligned
SENTINEL = 0xA5


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


class Guarded:
    """A device buffer of `shape`/`dtype` with sentinel bands before and after."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((BAND + n + BAND,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[BAND:BAND + n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        lo, hi = self.raw[:BAND], self.raw[-BAND:]
        assert bool((lo == SENTINEL).all()) and bool((hi == SENTINEL).all()), f"{what}: guard band written"


def bf16(rows, cols, seed):
    x = synth.fill(synth.recipe(seed, rows, 2.0, 0.01, 50.0, synth.OUT_SCALE), synth.BF16, rows * cols)
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda().reshape(rows, cols)


def typed(rows, cols, seed, dtype):
    """The bf16 input widened exactly to FP32, or rounded to FP16 (values in range)."""
    return bf16(rows, cols, seed).to(dtype)


@pytest.mark.parametrize("n", [1, 15, 16, 4097, 100_003])
def test_optimizer_outputs(n):
    w, m, v = (Guarded((n,), torch.float32) for _ in range(3))
    w16 = Guarded((n,), torch.bfloat16)
    g = torch.full((n,), 1.0, dtype=torch.float16, device="cuda")
    st = M.new_scaler_state(1.0)
    hp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 0.5)
    ws = Guarded((M.mp_adamw_workspace_size([M.Param(w.t, m.t, v.t, g, w16.t)]),), torch.uint8)
    M.mp_adamw_step([M.Param(w.t, m.t, v.t, g, w16.t)], hp, st, working_dtype=M.MP_BF16, workspace=ws.t)
    for b, name in ((w, "w"), (m, "m"), (v, "v"), (w16, "w16"), (ws, "workspace")):
        b.check(name)


@pytest.mark.parametrize("n", [1, 17, 4111, 1_000_003])
def test_fp8_cast(n):
    x = bf16(1, n, 1).reshape(-1)
    y = Guarded((n,), torch.uint8)
    M.fp8_cast_delayed(x, y.t, M.MP_E4M3, M.new_fp8_meta(), torch.zeros(4, device="cuda"))
    y.check("y")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(16, 16), (48, 1040), (272, 400)])
def test_fp8_cast_transpose(rows, cols, dtype):
    y, yt = Guarded((rows * cols,), torch.uint8), Guarded((rows * cols,), torch.uint8)
    M.fp8_cast_transpose_delayed(typed(rows, cols, 2, dtype), y.t, yt.t, M.MP_E5M2, M.new_fp8_meta(),
                                 torch.zeros(4, device="cuda"))
    y.check("y")
    yt.check("y_t")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("br", [1, 128])
@pytest.mark.parametrize("rows,cols", [(3, 144), (130, 272), (1000, 1040)])
def test_fp8_blockwise(br, rows, cols, dtype):
    y = Guarded((rows, cols), torch.uint8)
    sc = Guarded((-(-rows // br), -(-cols // 128)), torch.float32)
    M.fp8_quantize_blockwise(typed(rows, cols, 3, dtype), y.t, sc.t, br, 128)
    y.check("y")
    sc.check("scales")


@pytest.mark.parametrize("b2,sr,rht", [(False, False, False), (True, False, False), (False, True, True),
                                       (True, True, True)])
@pytest.mark.parametrize("rows,cols", [(16, 16), (48, 272)])
def test_nvfp4(b2, sr, rht, rows, cols):
    codes = Guarded((rows, cols // 2), torch.uint8)
    sc = Guarded((rows // 16 if b2 else rows, cols // 16), torch.uint8)
    dq = Guarded((rows, cols), torch.bfloat16)
    ts, nf = Guarded((1,), torch.float32), Guarded((1,), torch.int32)
    ws = Guarded((M.nvfp4_workspace_size(),), torch.uint8)
    ws.t.zero_()
    M.nvfp4_quantize(bf16(rows, cols, 4), codes.t, sc.t, ts.t, nf.t, ws.t, block_2d=b2, stochastic=sr, seed=5,
                     apply_rht=rht, sign_mask=0x1234, dequant=dq.t)
    for b, name in ((codes, "codes"), (sc, "scales"), (dq, "dequant"), (ts, "tensor scale"), (nf, "flag"),
                    (ws, "workspace")):
        b.check(name)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rht16(dtype):
    y = Guarded((37, 1024), dtype)
    M.rht16(bf16(37, 1024, 6), y.t, 0xE3BF)
    y.check("y")


@pytest.mark.parametrize("elem", [M.MP_E2M1, M.MP_E4M3, M.MP_E3M2])
@pytest.mark.parametrize("rows,cols", [(1, 32), (7, 544)])
def test_mx(elem, rows, cols):
    codes = Guarded((rows * cols // (2 if elem == M.MP_E2M1 else 1),), torch.uint8)
    sc = Guarded((rows, cols // 32), torch.uint8)
    dq = Guarded((rows, cols), torch.bfloat16)
    M.mx_quantize(bf16(rows, cols, 7), codes.t, sc.t, elem, dq.t)
    codes.check("codes")
    sc.check("scales")
    dq.check("dequant")
