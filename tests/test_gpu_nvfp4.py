"""GPU parity: nvfp4_quantize and rht16 (C ABI) against the oracle, bit for bit.

Small ragged shapes run every combination of block layout, transform,
rounding and dequant output; the three full-size workloads ([16384 x 5120]
1x16 RNE activations, [5120 x 5120] 16x16 RNE weights, [8192 x 12288]
RHT + 1x16 + SR gradients) are compared element by element against the
oracle (run on row chunks in parallel).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import synth.workloads as W
from tests.gpu_util import nvfp4_oracle, to_dev, to_host

pytestmark = pytest.mark.gpu

import mixed_precision_numerics_gb300 as M  # noqa: E402


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def gpu_quant(x_u16, block_2d, stochastic, seed, rht, mask, want_dequant=True, ws=None):
    rows, cols = x_u16.shape
    xt = to_dev(x_u16, torch.bfloat16) if x_u16.size else torch.empty((rows, cols), dtype=torch.bfloat16,
                                                                        device="cuda")
    codes = torch.full((rows, cols // 2), 0xAA, dtype=torch.uint8, device="cuda")
    srows = rows // 16 if block_2d else rows
    scales = torch.full((srows, cols // 16), 0xAA, dtype=torch.uint8, device="cuda")
    ts = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    nf = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dq = torch.full((rows, cols), 0x5555, dtype=torch.int16, device="cuda") if want_dequant else None
    ws = M.new_nvfp4_workspace() if ws is None else ws
    M.nvfp4_quantize(xt, codes, scales, ts, nf, ws, block_2d=block_2d, stochastic=stochastic, seed=seed,
                     apply_rht=rht, sign_mask=mask, dequant=dq, rows=rows, cols=cols)
    torch.cuda.synchronize()
    assert not ws.any().item(), "workspace must be left zero-filled"
    return (codes.cpu().numpy(), scales.cpu().numpy(), float(ts.item()), int(nf.item()),
            to_host(dq, np.uint16) if want_dequant else None)


def assert_same(got, ref, what=""):
    gc, gs, gts, gnf, gdq = got
    rc, rs, rts, rnf, rdq = ref
    assert np.array([gts], np.float32).view(np.uint32)[0] == np.array([rts], np.float32).view(np.uint32)[0], \
        f"{what} tensor scale {gts} vs {rts}"
    assert gnf == rnf, what
    bad = np.argwhere(gs != rs)
    assert bad.size == 0, f"{what}: {len(bad)} block scales differ, first at {bad[0]}: {gs[tuple(bad[0])]} vs {rs[tuple(bad[0])]}"
    bad = np.argwhere(gc != rc)
    assert bad.size == 0, f"{what}: {len(bad)} code bytes differ, first at {bad[0]}: 0x{gc[tuple(bad[0])]:02x} vs 0x{rc[tuple(bad[0])]:02x}"
    if gdq is not None:
        bad = np.argwhere(gdq != rdq)
        assert bad.size == 0, f"{what}: {len(bad)} dequant values differ, first at {bad[0]}"


def mixed_input(rows, cols, seed):
    x = synth.fill(synth.recipe(seed, 0, 1.0, 0.01, 40.0, synth.OUT_SCALE), synth.BF16, rows * cols, shape=(rows, cols))
    if x.size > 40:
        flat = x.reshape(-1)
        flat[[1, 5, 9]] = [0x8000, 0x0000, 0x0001]  # -0, +0, tiny subnormal
        if x.size >= 64:
            flat[32:48] = 0  # an all-zero block
    return x


@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (17, 272), (64, 4096), (33, 1040), (5, 5120)])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("sr", [False, True])
def test_1x16_small_shapes(shape, rht, sr):
    x = mixed_input(*shape, seed=40 + shape[0])
    mask = 0xB5E2
    got = gpu_quant(x, False, sr, 77, rht, mask)
    ref = O.nvfp4_quantize(x, False, sr, 77, rht, mask)
    assert_same(got, ref, f"1x16 {shape} rht={rht} sr={sr}")


@pytest.mark.parametrize("shape", [(16, 16), (32, 272), (48, 4112), (64, 512), (16, 5120)])
@pytest.mark.parametrize("rht", [False, True])
@pytest.mark.parametrize("sr", [False, True])
def test_16x16_small_shapes(shape, rht, sr):
    x = mixed_input(*shape, seed=60 + shape[0])
    mask = 0x1F0E
    got = gpu_quant(x, True, sr, 5, rht, mask)
    ref = O.nvfp4_quantize(x, True, sr, 5, rht, mask)
    assert_same(got, ref, f"16x16 {shape} rht={rht} sr={sr}")


def test_no_dequant_output_and_empty_tensor():
    x = mixed_input(32, 64, 3)
    got = gpu_quant(x, False, False, 0, False, 0, want_dequant=False)
    ref = O.nvfp4_quantize(x, False, False, 0, False, 0, want_dequant=False)
    assert_same(got, ref, "no dequant")
    got = gpu_quant(np.zeros((0, 32), np.uint16), False, False, 0, False, 0)
    assert got[2] == 0.0 and got[3] == 0


def test_every_bf16_value_on_a_unit_scale():
    """Blocks that each hold a 6.0 (so the block scale is 1 and r = 1) and an
    amax of 2688 (so s_t = 1) expose every BF16 magnitude in [0, 6] directly
    to the E2M1 rounding, RNE and stochastic."""
    vals = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = O.convert(vals, O.BF16, O.F32)
    vals = vals[np.isfinite(f) & (np.abs(f) <= 6.0)]
    per = 15
    nblk = (vals.size + per - 1) // per
    body = np.zeros(nblk * per, np.uint16)
    body[:vals.size] = vals
    blocks = np.concatenate([body.reshape(nblk, per), np.full((nblk, 1), 0x40C0, np.uint16)], axis=1)  # 6.0
    x = np.concatenate([blocks.reshape(-1), np.full(16, 0x4528, np.uint16)])  # 2688.0
    cols = 16 * 64
    x = np.concatenate([x, np.zeros((-x.size) % cols, np.uint16)]).reshape(-1, cols)
    for sr in (False, True):
        got = gpu_quant(x, False, sr, 99, False, 0)
        ref = O.nvfp4_quantize(x, False, sr, 99, False, 0)
        assert got[2] == 1.0
        assert_same(got, ref, f"unit scale sr={sr}")


def test_nonfinite_and_zero_inputs():
    x = mixed_input(16, 64, 8)
    x[3, 7] = 0x7F80
    for b2 in (False, True):
        got = gpu_quant(x, b2, False, 0, False, 0)
        ref = O.nvfp4_quantize(x, b2, False, 0, False, 0)
        assert got[3] == 1
        assert_same(got, ref, "inf input")
    x[3, 7] = 0xFFC1  # NaN
    got = gpu_quant(x, False, True, 0, True, 0x00FF)
    assert_same(got, O.nvfp4_quantize(x, False, True, 0, True, 0x00FF), "NaN input with RHT")
    z = np.zeros((32, 32), np.uint16)
    z[::3, ::5] = 0x8000
    for b2 in (False, True):
        got = gpu_quant(z, b2, True, 1, False, 0)
        assert_same(got, O.nvfp4_quantize(z, b2, True, 1, False, 0), "zeros")


def test_shape_and_alignment_errors():
    ws = M.new_nvfp4_workspace()
    x = torch.zeros((16, 48), dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros((16, 24), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((16, 3), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(1, dtype=torch.float32, device="cuda")
    nf = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MpError) as e:
        M.nvfp4_quantize(x, codes, sc, ts, nf, ws, rows=16, cols=40)
    assert e.value.status == M.MP_ESHAPE
    with pytest.raises(M.MpError) as e:
        M.nvfp4_quantize(x, codes, sc, ts, nf, ws, rows=8, cols=48, block_2d=True)
    assert e.value.status == M.MP_ESHAPE
    with pytest.raises(M.MpError) as e:
        M.nvfp4_quantize(x.view(-1)[1:], codes, sc, ts, nf, ws, rows=15, cols=48)
    assert e.value.status == M.MP_EALIGN
    with pytest.raises(M.MpError) as e:
        M.nvfp4_quantize(x, codes, sc, ts, nf, ws[:16], rows=16, cols=48)
    assert e.value.status == M.MP_EWORKSPACE


@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_rht16_standalone(out):
    x = mixed_input(37, 1024, 12)
    mask = 0x6A3C
    y = torch.empty((37, 1024), dtype=out, device="cuda")
    M.rht16(to_dev(x, torch.bfloat16), y, mask)
    torch.cuda.synchronize()
    ref = O.rht16(x, mask, O.F32 if out == torch.float32 else O.BF16)
    got = y.cpu().numpy() if out == torch.float32 else to_host(y, np.uint16)
    np.testing.assert_array_equal(got.view(np.uint32 if out == torch.float32 else np.uint16),
                                  ref.view(np.uint32 if out == torch.float32 else np.uint16))


def full_size_case(rows, cols, r, block_2d, sr, seed, rht, mask):
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    synth.fill_device(r, synth.BF16, x)
    x_host = to_host(x, np.uint16).reshape(rows, cols)
    np.testing.assert_array_equal(x_host.reshape(-1)[:4096], synth.fill(r, synth.BF16, 4096))
    got = gpu_quant(x_host, block_2d, sr, seed, rht, mask)
    ref = nvfp4_oracle(x_host, block_2d, sr, seed, rht, mask)
    return got, ref, x_host


def test_full_size_activations_1x16_rne():
    c = W.NVFP4_RNE
    got, ref, _ = full_size_case(c.act_rows, c.act_cols, c.act_recipe(), False, False, 0, False, 0)
    assert_same(got, ref, "activations [16384 x 5120] 1x16 RNE")


def test_full_size_weights_16x16_rne():
    c = W.NVFP4_RNE
    got, ref, _ = full_size_case(c.w_rows, c.w_cols, c.w_recipe(), True, False, 0, False, 0)
    assert_same(got, ref, "weights [5120 x 5120] 16x16 RNE")


def test_full_size_gradients_rht_sr():
    c = W.NVFP4_GRAD
    got, ref, x = full_size_case(c.rows, c.cols, c.recipe(), False, True, c.sr_seed, True, c.sign_mask())
    assert_same(got, ref, "gradients [8192 x 12288] RHT + 1x16 + SR")
    # stochastic rounding is unbiased: the mean error of the dequantised
    # values against x' is within a few standard errors of zero
    xp = O.nvfp4_prepare(x[:512], True, c.sign_mask()).astype(np.float64)
    dq = O.convert(got[4][:512], O.BF16, O.F32).astype(np.float64)
    err = (dq - xp).ravel()
    assert abs(err.mean()) < 5 * err.std() / np.sqrt(err.size)


def test_random_shape_sweep_2d_against_the_oracle():
    """Seeded random 16x16-block shapes (rows and cols multiples of 16, from one
    partial 16 x 256 strip to several strips per warp) with the transform and
    stochastic rounding on and off: codes, scales, tensor scale and dequantised
    values match the oracle bit for bit."""
    rng = np.random.default_rng(2027)
    for i in range(12):
        rows = 16 * int(rng.integers(1, 40))
        cols = 16 * int(rng.integers(1, 130))
        sr, rht = bool(i & 1), bool(i & 2)
        x = mixed_input(rows, cols, 500 + i)
        got = gpu_quant(x, True, sr, 77 + i, rht, 0x5A3C)
        ref = O.nvfp4_quantize(x, True, sr, 77 + i, rht, 0x5A3C)
        assert_same(got, ref, f"{rows}x{cols} sr={sr} rht={rht}")


# ---- the 1x16 encode's division-free block scale and its exact fallback -----------


def _bf16(v):
    return O.convert(np.asarray(v, np.float32), O.F32, O.BF16)


def midpoint_blocks(amax_bf16: int, count: int):
    """BF16 block maxima b whose block-scale quotient q = RN(RN(b / 6) / s_t)
    lies within a few units of an E4M3 rounding midpoint under the tensor
    scale s_t of a tensor with max |x| = amax: the blocks for which the
    encode's division-free estimate of the scale code cannot decide and the
    exact divisions run.  Found by the oracle's arithmetic in numpy."""
    f = np.float32
    a = O.convert(np.array([amax_bf16], np.uint16), O.BF16, O.F32)[0]
    s_t = f(a) / f(2688.0)
    b = O.convert(np.arange(1, amax_bf16 + 1, dtype=np.uint16), O.BF16, O.F32)
    qt = b * ((f(1) / f(6)) * (f(1) / s_t))
    lo, hi = qt * f(1 - 2.0 ** -21), qt * f(1 + 2.0 ** -21)
    undecided = O.convert(lo, O.F32, O.E4M3) != O.convert(hi, O.F32, O.E4M3)
    return np.arange(1, amax_bf16 + 1, dtype=np.uint16)[undecided][:count]


@pytest.mark.parametrize("sr", [False, True])
def test_1x16_blocks_whose_scale_code_needs_the_exact_divisions(sr):
    amax = int(_bf16([3.5])[0])  # a tensor max with many undecided block maxima (126)
    mids = midpoint_blocks(amax, 512)
    assert mids.size >= 100, "too few undecided block maxima for this tensor max"
    rng = np.random.default_rng(17)
    rows = mids.size + 1
    x = synth.fill(synth.recipe(80, 0, 0.05), synth.BF16, rows * 16, shape=(rows, 16))
    x[0, 5] = amax  # the tensor max
    for r, m in enumerate(mids, start=1):
        x[r, rng.integers(0, 16)] = m | (0x8000 if r % 3 == 0 else 0)  # the block max, some negative
        over = np.abs(O.convert(x[r], O.BF16, O.F32)) > O.convert(np.array([m], np.uint16), O.BF16, O.F32)[0]
        x[r] = np.where(over, x[r] & 0x8000, x[r]).astype(np.uint16)  # smaller than the block max
    got = gpu_quant(x, False, sr, 99, False, 0)
    ref = O.nvfp4_quantize(x, False, sr, 99, False, 0)
    assert_same(got, ref, f"undecided block scales sr={sr}")


@pytest.mark.parametrize("scale", [1e-30, 1e-26, 1e-25, 1e35, 1e36])
@pytest.mark.parametrize("rht,sr", [(False, False), (True, True), (True, False)])
def test_1x16_tensor_scales_outside_the_fast_range(scale, rht, sr):
    """Tensor scales below 2^-90 or above 2^110 run every block through the
    exact divisions and the two-step products; 1e-25 and 1e35 put s_t just
    inside the edges (s_t is about scale / 84 here)."""
    x = synth.fill(synth.recipe(81, 0, float(np.float32(scale)), 0.02, 8.0, synth.OUT_SCALE), synth.BF16, 64 * 512,
                   shape=(64, 512))
    got = gpu_quant(x, False, sr, 5, rht, 0x5A3C)
    ref = O.nvfp4_quantize(x, False, sr, 5, rht, 0x5A3C)
    assert_same(got, ref, f"scale {scale} rht={rht} sr={sr}")
    assert ref[3] == 0 and ref[2] != 0.0


@pytest.mark.parametrize("rht,sr", [(False, False), (False, True), (True, True)])
def test_1x16_blocks_of_subnormal_values_in_a_normal_tensor(rht, sr):
    """Blocks whose max is below 2^-120 take the exact path; their codes and
    scales are mostly zero, a few tiny values survive when the block is all
    that small and the tensor max is small too."""
    rows = 48
    x = synth.fill(synth.recipe(82, 0, 1.0), synth.BF16, rows * 64, shape=(rows, 64))
    tiny = (synth.fill(synth.recipe(83, 0, 1.0), synth.BF16, rows * 64, shape=(rows, 64)) & 0x807F).astype(np.uint16)
    x[::2, :32] = tiny[::2, :32]  # subnormals
    x[1::4] = tiny[1::4] | np.uint16(0x0080)  # the smallest normal binade
    got = gpu_quant(x, False, sr, 11, rht, 0x1357)
    ref = O.nvfp4_quantize(x, False, sr, 11, rht, 0x1357)
    assert_same(got, ref, f"subnormal blocks rht={rht} sr={sr}")
