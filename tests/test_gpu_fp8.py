"""GPU parity: fp8_cast_delayed (C ABI) against the oracle, bit for bit.

Covers every BF16 bit pattern at several scales, F16 and F32 inputs with
specials, ragged lengths, the tiny delayed-scaling workload (1024x1024 BF16,
history 16, 20 iterations) element by element, the FP8 workload at reduced
row count element by element, and the full [8192 x 4096] workload byte for
byte in every one of its 64 iterations, with the exact amax/scale recurrence.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synth
import synth.workloads as W
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

import mixed_precision_numerics_gb300 as M  # noqa: E402
FMT = {M.MP_E4M3: O.E4M3, M.MP_E5M2: O.E5M2}
XFMT = {torch.float32: O.F32, torch.float16: O.F16, torch.bfloat16: O.BF16}


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def set_meta(meta_t, scale=1.0, pos=0):
    m = M.read_fp8_meta(meta_t)
    m.scale = scale
    m.scale_inv = float(np.float32(1.0) / np.float32(scale))
    m.pos = pos
    meta_t.copy_(torch.frombuffer(bytearray(bytes(m)), dtype=torch.uint8).to(meta_t.device))


def gpu_cast(x_t, fmt, meta_t, hist_t, margin=1.0):
    y = torch.empty(x_t.numel(), dtype=torch.uint8, device="cuda")
    M.fp8_cast_delayed(x_t, y, fmt, meta_t, hist_t, margin)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def assert_meta_equal(g: "M.Fp8Meta", o: "O.Fp8Meta"):
    f = lambda v: np.array([v], np.float32).view(np.uint32)[0]
    assert f(g.scale) == f(o.scale), (g.scale, o.scale)
    assert f(g.scale_inv) == f(o.scale_inv)
    assert f(g.amax) == f(o.amax), (g.amax, o.amax)
    assert g.pos == o.pos
    assert g.internal_amax == 0 and g.internal_ticket == 0 and g.internal_hrest == 0


@pytest.mark.parametrize("fmt", [M.MP_E4M3, M.MP_E5M2])
@pytest.mark.parametrize("scale", [1.0, 3.0, 448.0 / 300.0, 2.0**-10, 2.0**20, 1e-30, 1e30])
def test_every_bf16_pattern(fmt, scale):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = np.concatenate([x, x[:13]])  # ragged tail
    xt = to_dev(x, torch.bfloat16)
    meta = M.new_fp8_meta()
    hist = torch.zeros(4, dtype=torch.float32, device="cuda")
    set_meta(meta, scale)
    y = gpu_cast(xt, fmt, meta, hist)
    ref = O.fp8_cast_array(x, O.BF16, FMT[fmt], scale)
    bad = np.nonzero(y != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x=0x{x[bad[0]]:04x} gpu=0x{y[bad[0]]:02x} oracle=0x{ref[bad[0]]:02x}"
    om = O.new_fp8_meta()
    om.scale = scale
    om.scale_inv = float(np.float32(1.0) / np.float32(scale))
    oh = np.zeros(4, np.float32)
    O.fp8_history_update(om, oh, 1.0, O.amax(x, O.BF16), FMT[fmt])
    assert_meta_equal(M.read_fp8_meta(meta), om)
    np.testing.assert_array_equal(hist.cpu().numpy().view(np.uint32), oh.view(np.uint32))


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
@pytest.mark.parametrize("fmt", [M.MP_E4M3, M.MP_E5M2])
def test_f16_f32_inputs_with_specials(dtype, fmt):
    rng = np.random.default_rng(5)
    n = 300_007
    xf = (rng.standard_normal(n) * rng.choice([1e-6, 1e-2, 1.0, 100.0, 1e4], n)).astype(np.float32)
    xf[[3, 77, 1000]] = [np.inf, -np.inf, 0.0]
    xf[5] = -0.0
    if dtype == torch.float16:
        x = O.convert(xf, O.F32, O.F16)
        x[[9, 11]] = [0x7E00, 0xFC01]  # NaNs
        xt = to_dev(x, torch.float16)
    else:
        x = xf.copy()
        x[[9, 11]] = np.float32("nan")
        xt = to_dev(x)
    for scale in (1.0, 7.5, 1e-3):
        meta = M.new_fp8_meta()
        hist = torch.zeros(8, dtype=torch.float32, device="cuda")
        set_meta(meta, scale)
        y = gpu_cast(xt, fmt, meta, hist)
        ref = O.fp8_cast_array(x, XFMT[dtype], FMT[fmt], scale)
        np.testing.assert_array_equal(y, ref)
        assert np.isnan(M.read_fp8_meta(meta).amax)
        assert M.read_fp8_meta(meta).scale == np.float32(scale)  # NaN history keeps the scale


@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 4095, 4096 * 2 + 3, 1_000_003])
def test_ragged_lengths(n):
    x = synth.fill(synth.recipe(11, n, 3.0), synth.BF16, n)
    xt = to_dev(x, torch.bfloat16) if n else torch.empty(0, dtype=torch.bfloat16, device="cuda")
    meta = M.new_fp8_meta()
    hist = torch.zeros(16, dtype=torch.float32, device="cuda")
    set_meta(meta, 17.0)
    y = gpu_cast(xt, M.MP_E4M3, meta, hist)
    ref = O.fp8_cast_array(x, O.BF16, O.E4M3, 17.0)
    np.testing.assert_array_equal(y, ref)
    om = O.new_fp8_meta()
    om.scale, om.scale_inv = 17.0, float(np.float32(1) / np.float32(17))
    oh = np.zeros(16, np.float32)
    O.fp8_history_update(om, oh, 1.0, O.amax(x, O.BF16) if n else 0.0, O.E4M3)
    assert_meta_equal(M.read_fp8_meta(meta), om)


def run_sequence(recipes, rows, cols, fmt, hist_len, margin):
    """GPU and oracle over a sequence of iterations, compared element by element."""
    meta = M.new_fp8_meta()
    hist = torch.zeros(hist_len, dtype=torch.float32, device="cuda")
    om, oh = O.new_fp8_meta(), np.zeros(hist_len, np.float32)
    for k, r in enumerate(recipes):
        x = synth.fill(r, synth.BF16, rows * cols)
        y = gpu_cast(to_dev(x, torch.bfloat16), fmt, meta, hist, margin)
        ref = O.fp8_cast_delayed(x, O.BF16, FMT[fmt], om, oh, margin)
        assert np.array_equal(y, ref), f"iteration {k}: {np.count_nonzero(y != ref)} bytes differ"
        assert_meta_equal(M.read_fp8_meta(meta), om)
        np.testing.assert_array_equal(hist.cpu().numpy().view(np.uint32), oh.view(np.uint32))
    return om


def test_tiny_delayed_scaling_workload():
    c = W.TINY_FP8
    om = run_sequence([c.recipe(k) for k in range(c.iters)], c.rows, c.cols, M.MP_E4M3, c.hist_len, c.margin)
    assert om.pos == c.iters % c.hist_len  # the ring wrapped


@pytest.mark.parametrize("which", ["act", "grad"])
def test_fp8_workload_reduced_rows(which):
    c = W.FP8
    rows = 64
    recipes = [c.act_recipe(k) if which == "act" else c.grad_recipe(k) for k in range(c.iters)]
    fmt = M.MP_E4M3 if which == "act" else M.MP_E5M2
    run_sequence(recipes, rows, c.cols, fmt, c.hist_len, c.margin)


def oracle_cast_parallel(x_host, x_fmt, fmt, scale):
    """The oracle's cast over row chunks on the host threads (its C calls
    release the GIL); the cast is element-wise, so chunking changes nothing."""
    import concurrent.futures as cf

    from tests.gpu_util import threads

    parts = np.array_split(x_host, threads() * 2)
    with cf.ThreadPoolExecutor(threads()) as ex:
        return np.concatenate(list(ex.map(lambda p: O.fp8_cast_array(p, x_fmt, fmt, scale), parts)))


@pytest.mark.parametrize("which", ["act", "grad"])
def test_fp8_workload_full_size(which):
    """[8192 x 4096] x 64 iterations: every output byte of every iteration
    against the oracle's cast of the same input under the scale in force, the
    amax of each iteration against torch's max |x| (exact), the scale
    recurrence against the oracle fed those amaxes, and the first 65536
    inputs of each iteration against the host generator."""
    c = W.FP8
    n = c.rows * c.cols
    fmt = M.MP_E4M3 if which == "act" else M.MP_E5M2
    meta = M.new_fp8_meta()
    hist = torch.zeros(c.hist_len, dtype=torch.float32, device="cuda")
    x = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(n, dtype=torch.uint8, device="cuda")
    om, oh = O.new_fp8_meta(), np.zeros(c.hist_len, np.float32)
    sat, scale_changes = 0, 0
    for k in range(c.iters):
        r = c.act_recipe(k) if which == "act" else c.grad_recipe(k)
        synth.fill_device(r, synth.BF16, x)
        scale_in_force = om.scale
        M.fp8_cast_delayed(x, y, fmt, meta, hist, c.margin)
        x_host = to_host(x, np.uint16)
        np.testing.assert_array_equal(x_host[:65536], synth.fill(r, synth.BF16, 65536))
        ref = oracle_cast_parallel(x_host, O.BF16, FMT[fmt], scale_in_force)
        got = y.cpu().numpy()
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, f"iteration {k}: {bad.size} bytes differ, first at {bad[:5]}"
        amax = float(x.float().abs().max().item())
        O.fp8_history_update(om, oh, c.margin, amax, FMT[fmt])
        assert_meta_equal(M.read_fp8_meta(meta), om)
        scale_changes += int(om.scale != scale_in_force)
        sat += int(((ref & 0x7F) == (0x7E if fmt == M.MP_E4M3 else 0x7B)).sum())
    assert scale_changes > 0
    if which == "act":
        assert sat > 0  # the drifting std makes the delayed scale lag: saturation happens


# ---- most_recent amax and the transposed output ----------------------------------


def test_most_recent_sequence():
    c = W.TINY_FP8
    meta = M.new_fp8_meta()
    hist = torch.zeros(c.hist_len, dtype=torch.float32, device="cuda")
    om, oh = O.new_fp8_meta(), np.zeros(c.hist_len, np.float32)
    for k in range(8):
        r = synth.recipe(c.seed, 100 + k, float(2.0 ** (k % 5 - 2)))
        x = synth.fill(r, synth.BF16, 65536 + 3)
        y = torch.empty(x.size, dtype=torch.uint8, device="cuda")
        M.fp8_cast_delayed(to_dev(x, torch.bfloat16), y, M.MP_E4M3, meta, hist, 1.5, amax_algo=M.MP_AMAX_MOST_RECENT)
        ref = O.fp8_cast_delayed(x, O.BF16, O.E4M3, om, oh, 1.5, O.AMAX_MOST_RECENT)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(y.cpu().numpy(), ref)
        assert_meta_equal(M.read_fp8_meta(meta), om)
        np.testing.assert_array_equal(hist.cpu().numpy().view(np.uint32), oh.view(np.uint32))


def cast_t(xt, fmt, meta, hist, algo=0):
    rows, cols = xt.shape
    y = torch.full((rows * cols,), 0xCC, dtype=torch.uint8, device="cuda")
    yt = torch.full((cols * rows,), 0xCC, dtype=torch.uint8, device="cuda")
    M.fp8_cast_transpose_delayed(xt, y, yt, fmt, meta, hist, 1.0, algo)
    torch.cuda.synchronize()
    return y.cpu().numpy().reshape(rows, cols), yt.cpu().numpy().reshape(cols, rows)


@pytest.mark.parametrize("shape", [(16, 16), (64, 64), (80, 144), (48, 1040), (1024, 1040)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("fmt", [M.MP_E4M3, M.MP_E5M2])
def test_cast_transpose_small(shape, dtype, fmt):
    rows, cols = shape
    xf = synth.fill(synth.recipe(80, rows, 3.0, 0.01, 100.0, synth.OUT_SCALE), synth.F32, rows * cols)
    xf[:3] = [np.inf, np.nan, -0.0]
    if dtype == torch.float32:
        x = xf
        xt = to_dev(x).reshape(rows, cols)
    else:
        fmt16 = O.BF16 if dtype == torch.bfloat16 else O.F16
        x = O.convert(xf, O.F32, fmt16)
        xt = to_dev(x, dtype).reshape(rows, cols)
    meta = M.new_fp8_meta()
    hist = torch.zeros(4, dtype=torch.float32, device="cuda")
    set_meta(meta, 13.0)
    y, yt = cast_t(xt, fmt, meta, hist)
    ref = O.fp8_cast_array(x, XFMT[dtype], FMT[fmt], 13.0).reshape(rows, cols)
    np.testing.assert_array_equal(y, ref)
    np.testing.assert_array_equal(yt, O.transpose_u8(ref))
    om = O.new_fp8_meta()
    om.scale, om.scale_inv = 13.0, float(np.float32(1) / np.float32(13))
    oh = np.zeros(4, np.float32)
    O.fp8_history_update(om, oh, 1.0, O.amax(x, XFMT[dtype]), FMT[fmt])
    assert_meta_equal(M.read_fp8_meta(meta), om)


@pytest.mark.parametrize("shape,dtype", [((2064, 4112), torch.bfloat16), ((1040, 6160), torch.float32),
                                         ((4112, 2064), torch.float16)])
def test_cast_transpose_many_tiles_per_cta(shape, dtype):
    """Enough 128 x 128 boxes that every CTA's ring of tile copies and its
    alternating transpose buffers wrap several times, with partial boxes on the
    right and bottom edges; the amax and the next scale still come out exact."""
    rows, cols = shape
    xf = synth.fill(synth.recipe(81, rows, 2.0, 0.01, 80.0, synth.OUT_SCALE), synth.F32, rows * cols)
    xf[[7, 100_003]] = [np.nan, -np.inf]
    x = xf if dtype == torch.float32 else O.convert(xf, O.F32, XFMT[dtype])
    xt = (to_dev(x) if dtype == torch.float32 else to_dev(x, dtype)).reshape(rows, cols)
    for fmt in (M.MP_E4M3, M.MP_E5M2):
        meta = M.new_fp8_meta()
        hist = torch.zeros(4, dtype=torch.float32, device="cuda")
        set_meta(meta, 0.37)
        y, yt = cast_t(xt, fmt, meta, hist)
        ref = O.fp8_cast_array(x, XFMT[dtype], FMT[fmt], 0.37).reshape(rows, cols)
        assert np.array_equal(y, ref)
        assert np.array_equal(yt, O.transpose_u8(ref))
        assert np.isnan(M.read_fp8_meta(meta).amax)
    assert M.mp_wait_failures() == 0


def test_cast_transpose_full_size_sequence():
    c = W.FP8
    meta = M.new_fp8_meta()
    hist = torch.zeros(c.hist_len, dtype=torch.float32, device="cuda")
    om, oh = O.new_fp8_meta(), np.zeros(c.hist_len, np.float32)
    x = torch.empty((c.rows, c.cols), dtype=torch.bfloat16, device="cuda")
    for k in range(3):
        synth.fill_device(c.act_recipe(k), synth.BF16, x)
        y, yt = cast_t(x, M.MP_E4M3, meta, hist)
        xh = to_host(x, np.uint16).reshape(c.rows, c.cols)
        ref = O.fp8_cast_delayed(xh, O.BF16, O.E4M3, om, oh, c.margin)
        assert np.array_equal(y, ref.reshape(c.rows, c.cols)), f"iteration {k}"
        assert np.array_equal(yt, ref.reshape(c.rows, c.cols).T), f"iteration {k} transposed"
        assert_meta_equal(M.read_fp8_meta(meta), om)


def test_cast_transpose_argument_errors():
    x = torch.zeros((16, 24), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(16 * 32, dtype=torch.uint8, device="cuda")
    meta, hist = M.new_fp8_meta(), torch.zeros(4, device="cuda")
    with pytest.raises(M.MpError) as e:
        M.fp8_cast_transpose_delayed(x, y, y, M.MP_E4M3, meta, hist)
    assert e.value.status == M.MP_ESHAPE


def test_cast_transpose_of_an_empty_tensor_still_records_the_step():
    """A [0, cols] cast is a step with amax 0: the ring slot is written and the
    position advances, as for an empty fp8_cast_delayed."""
    meta, hist = M.new_fp8_meta(), torch.full((3,), 5.0, device="cuda")
    om, oh = O.new_fp8_meta(), np.full(3, 5.0, np.float32)
    x = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.uint8, device="cuda")
    for _ in range(4):
        M.fp8_cast_transpose_delayed(x, y, y, M.MP_E4M3, meta, hist)
        O.fp8_cast_delayed(np.zeros(0, np.uint16), O.BF16, O.E4M3, om, oh, 1.0)
        torch.cuda.synchronize()
        assert_meta_equal(M.read_fp8_meta(meta), om)
        np.testing.assert_array_equal(hist.cpu().numpy().view(np.uint32), oh.view(np.uint32))


@pytest.mark.parametrize("fmt", [M.MP_E4M3, M.MP_E5M2])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_saturation_count_matches_the_oracle(fmt, dtype):
    """The counting cast writes the same bytes and state as the plain one and
    adds the oracle's saturation count; the counter accumulates over calls."""
    n = 1_000_003
    xf = synth.fill(synth.recipe(70, 1, 1.0, 0.01, 800.0, synth.OUT_T3), synth.F32, n)
    xf[[3, 5, 7]] = [np.inf, -np.inf, np.nan]
    x = xf if dtype == torch.float32 else O.convert(xf, O.F32, XFMT[dtype])
    xt = to_dev(x) if dtype == torch.float32 else to_dev(x, dtype)
    sat = torch.zeros(1, dtype=torch.int64, device="cuda")
    total = 0
    for scale in (1.0, 0.25, 40.0):
        m1, m2 = M.new_fp8_meta(), M.new_fp8_meta()
        set_meta(m1, scale)
        set_meta(m2, scale)
        h1, h2 = torch.zeros(4, device="cuda"), torch.zeros(4, device="cuda")
        y1 = torch.empty(n, dtype=torch.uint8, device="cuda")
        y2 = torch.empty(n, dtype=torch.uint8, device="cuda")
        M.fp8_cast_delayed(xt, y1, fmt, m1, h1)
        M.fp8_cast_delayed_count(xt, y2, fmt, m2, h2, sat)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2) and torch.equal(m1, m2)
        assert torch.equal(h1.view(torch.int32), h2.view(torch.int32))  # bits: the amax may be NaN
        total += O.fp8_saturation_count(x, XFMT[dtype], FMT[fmt], scale)
        assert int(sat.item()) == total


def test_chained_launches_see_the_previous_kernels_writes():
    """The quantisers are launched with programmatic stream serialization; each
    waits for the previous kernel before touching memory.  A torch kernel that
    rewrites the input right before every call must be seen by that call, and
    each FP8 cast must see the scale its predecessor left in the meta, with no
    synchronisation anywhere in the loop."""
    n = 1 << 20
    steps = 40
    x = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ys = torch.empty((steps, n), dtype=torch.uint8, device="cuda")
    codes = torch.empty((steps, n // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty((steps, n // 16), dtype=torch.uint8, device="cuda")
    ts = torch.empty(steps, dtype=torch.float32, device="cuda")
    nf = torch.empty(steps, dtype=torch.int32, device="cuda")
    ws = M.new_nvfp4_workspace()
    meta, hist = M.new_fp8_meta(), torch.zeros(4, device="cuda")
    vals = [float(2.0 ** (k % 7 - 3)) * (1 + (k % 3) / 8) for k in range(steps)]
    for k, v in enumerate(vals):
        x.fill_(v)  # a torch kernel writes the input
        M.fp8_cast_delayed(x, ys[k], M.MP_E4M3, meta, hist)
        M.nvfp4_quantize(x.view(1024, 1024), codes[k], sc[k], ts[k:k + 1], nf[k:k + 1], ws)
    torch.cuda.synchronize()
    om, oh = O.new_fp8_meta(), np.zeros(4, np.float32)
    for k, v in enumerate(vals):
        xb = O.convert(np.full(16, v, np.float32), O.F32, O.BF16)  # the same constant tensor, 16 elements
        want = O.fp8_cast_delayed(xb, O.BF16, O.E4M3, om, oh, 1.0)[0]
        assert bool((ys[k] == int(want)).all()), f"iteration {k}: the FP8 cast saw a stale input or scale"
        xv = (xb[:1].astype(np.uint32) << 16).view(np.float32)[0]
        assert np.float32(ts[k].item()) == np.float32(xv) / np.float32(2688.0), f"iteration {k}: tensor scale"
    assert_meta_equal(M.read_fp8_meta(meta), om)
