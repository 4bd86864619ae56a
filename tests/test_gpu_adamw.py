"""GPU parity: mp_adamw_step + loss_scale_update (C ABI) against the oracle.

The FP32 master, moments and step state must agree within 4 ulp (the order
of operations is fixed on both sides, so 0 is expected and reported); the
16-bit working copy and every scaler field bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import synth.workloads as W
from tests.conftest import golden
from tests.gpu_util import to_dev, to_host, ulp_diff

pytestmark = pytest.mark.gpu

import mixed_precision_numerics_gb300 as M  # noqa: E402
TD = {O.F16: torch.float16, O.BF16: torch.bfloat16}
MPD = {O.F16: M.MP_F16, O.BF16: M.MP_BF16}
MAX_ULP = 4


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def hp_of(c):
    return M.AdamwHparams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay), O.AdamwHp(c.lr, c.beta1, c.beta2, c.eps,
                                                                                     c.weight_decay)


def assert_state_equal(g, o):
    assert np.float32(g.scale) == np.float32(o.scale)
    assert g.growth_tracker == o.growth_tracker and g.found_inf == o.found_inf
    assert g.step == o.step and g.skipped == o.skipped
    assert g.beta1_pow == o.beta1_pow and g.beta2_pow == o.beta2_pow
    assert g.internal_found == 0 and g.internal_ticket == 0


class Tensors:
    def __init__(self, w0, g_fmt, w_fmt):
        n = w0.size
        self.w = to_dev(w0)
        self.m = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.v = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.g = torch.zeros(n, dtype=TD[g_fmt], device="cuda")
        self.w16 = torch.zeros(n, dtype=TD[w_fmt], device="cuda")
        self.ow, self.om, self.ov = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        self.ow16 = np.zeros(n, np.uint16)

    def param(self):
        return M.Param(self.w, self.m, self.v, self.g, self.w16)

    def oracle_tuple(self, g_host):
        return (self.ow, self.om, self.ov, g_host, self.ow16)

    def compare(self, what=""):
        for gt, ot, name in ((self.w, self.ow, "w"), (self.m, self.om, "m"), (self.v, self.ov, "v")):
            d = ulp_diff(gt.cpu().numpy(), ot)
            assert d.max(initial=0) <= MAX_ULP, f"{what} {name}: max ulp {d.max()}"
            assert d.max(initial=0) == 0, f"{what} {name}: max ulp {d.max()} (within tolerance but not exact)"
        np.testing.assert_array_equal(to_host(self.w16, np.uint16), self.ow16, err_msg=f"{what} working copy")


def test_tiny_step_twelve_steps():
    c = W.TINY
    t = golden("scaler_trajectory_tiny.json")
    ghp, ohp = hp_of(c)
    cfg = M.ScalerCfg(c.growth, c.backoff, c.interval, 1)
    ocfg = O.ScalerCfg(c.growth, c.backoff, c.interval, 1)
    w0 = synth.fill(c.master_recipe(), synth.F32, c.n)
    T = Tensors(w0, O.F16, O.F16)
    st = M.new_scaler_state(c.init_scale)
    ost = O.new_scaler_state(c.init_scale)
    for k in range(1, c.steps + 1):
        S = t["scale_used"][k - 1]
        assert M.read_scaler_state(st).scale == S
        g = synth.fill(c.grad_recipe(k, S), synth.F16, c.n)
        inj = c.injection(k)
        if inj:
            g[inj[0]] = inj[1]
        T.g.copy_(to_dev(g, torch.float16))
        M.mp_adamw_step([T.param()], ghp, st)
        M.loss_scale_update(st, cfg)
        O.adamw_step(ohp, ost, [T.oracle_tuple(g)], O.F16, O.F16)
        O.loss_scale_update(ost, ocfg)
        torch.cuda.synchronize()
        gs = M.read_scaler_state(st)
        assert gs.found_inf == t["found_inf"][k - 1]
        assert gs.growth_tracker == t["tracker_after"][k - 1]
        assert_state_equal(gs, ost)
        T.compare(f"step {k}")
    gs = M.read_scaler_state(st)
    assert gs.scale == t["final_scale"] and gs.step == t["applied_steps"] and gs.skipped == t["skipped_steps"]


@pytest.mark.parametrize("g_fmt,w_fmt", [(O.F16, O.F16), (O.F16, O.BF16), (O.BF16, O.BF16), (O.BF16, O.F16)])
def test_ragged_multi_tensor(g_fmt, w_fmt):
    sizes = [1, 7, 8, 9, 15, 4095, 4096, 4097, 8191, 100_003, 0, 3]
    ghp, ohp = M.AdamwHparams(3e-3, 0.8, 0.99, 1e-6, 0.1), O.AdamwHp(3e-3, 0.8, 0.99, 1e-6, 0.1)
    cfg, ocfg = M.ScalerCfg(2.0, 0.5, 2, 1), O.ScalerCfg(2.0, 0.5, 2, 1)
    S0 = 1024.0 if g_fmt == O.F16 else 1.0
    Ts = [Tensors(synth.fill(synth.recipe(20, i, 0.5), synth.F32, n), g_fmt, w_fmt) for i, n in enumerate(sizes)]
    st, ost = M.new_scaler_state(S0), O.new_scaler_state(S0)
    for k in range(1, 5):
        S = float(ost.scale)
        hosts = []
        for i, (T, n) in enumerate(zip(Ts, sizes)):
            g = synth.fill(synth.recipe(21, 100 * k + i, float(np.float32(0.01 * S))), synth.F16 if g_fmt == O.F16
                           else synth.BF16, n)
            if k == 2 and i == 5:
                g[17] = 0x7C00 if g_fmt == O.F16 else 0xFF80  # +inf / -inf
            hosts.append(g)
            if n:
                T.g.copy_(to_dev(g, TD[g_fmt]))
        M.mp_adamw_step([T.param() for T in Ts], ghp, st)
        M.loss_scale_update(st, cfg)
        O.adamw_step(ohp, ost, [T.oracle_tuple(g) for T, g in zip(Ts, hosts)], g_fmt, w_fmt)
        O.loss_scale_update(ost, ocfg)
        torch.cuda.synchronize()
        assert_state_equal(M.read_scaler_state(st), ost)
        for i, T in enumerate(Ts):
            T.compare(f"step {k} tensor {i}")
    assert ost.skipped == 1


def test_more_tensors_than_one_launch_table():
    rng = np.random.default_rng(3)
    sizes = rng.integers(1, 300, size=600).tolist()
    ghp, ohp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01), O.AdamwHp(1e-3, 0.9, 0.999, 1e-8, 0.01)
    Ts = [Tensors(synth.fill(synth.recipe(30, i, 0.02), synth.F32, n), O.BF16, O.BF16) for i, n in enumerate(sizes)]
    st, ost = M.new_scaler_state(1.0), O.new_scaler_state(1.0)
    for k in (1, 2):
        hosts = []
        for i, (T, n) in enumerate(zip(Ts, sizes)):
            g = synth.fill(synth.recipe(31, 1000 * k + i, 1e-3), synth.BF16, n)
            if k == 2 and i == 550:
                g[0] = 0x7FC0  # NaN in the second launch group
            hosts.append(g)
            T.g.copy_(to_dev(g, torch.bfloat16))
        M.mp_adamw_step([T.param() for T in Ts], ghp, st)
        O.adamw_step(ohp, ost, [T.oracle_tuple(g) for T, g in zip(Ts, hosts)], O.BF16, O.BF16)
        torch.cuda.synchronize()
        assert_state_equal(M.read_scaler_state(st), ost)
        for i in (0, 1, 511, 512, 513, 599):
            Ts[i].compare(f"step {k} tensor {i}")
    assert ost.found_inf == 1 and ost.step == 1


def test_empty_parameter_list_still_counts_the_step():
    ghp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    st = M.new_scaler_state(8.0)
    M.mp_adamw_step([], ghp, st, grad_dtype=M.MP_F16, working_dtype=M.MP_F16)
    s = M.read_scaler_state(st)
    assert s.step == 1 and s.found_inf == 0


def test_invalid_arguments_are_rejected_before_launch():
    ghp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    st = M.new_scaler_state()
    w = torch.zeros(9, dtype=torch.float32, device="cuda")
    g = torch.zeros(9, dtype=torch.float16, device="cuda")
    before = M.mp_launch_count()
    with pytest.raises(M.MpError) as e:
        M.mp_adamw_step([M.Param(w[1:], w[1:], w[1:], g[1:], g[1:])], ghp, st)
    assert e.value.status == M.MP_EALIGN
    with pytest.raises(M.MpError) as e:
        M.mp_adamw_step([M.Param(w, w, w, g, g)], M.AdamwHparams(1e-3, 1.0, 0.999, 1e-8, 0.0), st)
    assert e.value.status == M.MP_EINVAL
    with pytest.raises(M.MpError):
        M.loss_scale_update(st, M.ScalerCfg(2.0, 0.5, 0, 1))
    assert M.mp_launch_count() == before


def apply_parallel(s_orc, w, m, v, g, g_fmt, w16, w16_fmt):
    """The oracle's element-wise update over chunks of whole tensors on the
    host threads (its C calls release the GIL; chunks are contiguous views)."""
    import concurrent.futures as cf

    from tests.gpu_util import threads

    n = w.size
    edges = np.linspace(0, n, threads() * 2 + 1).astype(np.int64)

    def run(i):
        a, b = edges[i], edges[i + 1]
        O.adamw_apply(s_orc, w[a:b], m[a:b], v[a:b], g[a:b], g_fmt, w16[a:b], w16_fmt)

    with cf.ThreadPoolExecutor(threads()) as ex:
        list(ex.map(run, range(len(edges) - 1)))


def test_full_model_step():
    """Llama-3-8B-shaped list, 290 tensors, 8.03e9 params, 5 steps with an inf
    on step 3: found_inf per step against torch's isfinite over every grad;
    the embedding and lm_head (1.05e9 params) element by element; in every
    other tensor the elements on both sides of every 2816-element chunk edge
    of the update kernel, the first and last 8 and 96 random ones; and the
    working copy against torch's BF16 rounding of every master element."""
    c = W.FULL
    params = W.llama3_8b_params()
    total = sum(n for _, n in params)
    free, _ = torch.cuda.mem_get_info()
    need = total * 16 + (4 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, have {free / 2**30:.0f}")
    ghp, ohp = hp_of(c)
    cfg, ocfg = M.ScalerCfg(c.growth, c.backoff, c.interval, 1), O.ScalerCfg(c.growth, c.backoff, c.interval, 1)
    ws, ms, vs, gs, w16s = [], [], [], [], []
    for t, (name, n) in enumerate(params):
        w = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.fill_device(c.master_recipe(t), synth.F32, w)
        ws.append(w)
        ms.append(torch.zeros(n, dtype=torch.float32, device="cuda"))
        vs.append(torch.zeros(n, dtype=torch.float32, device="cuda"))
        gs.append(torch.empty(n, dtype=torch.float16, device="cuda"))
        w16s.append(torch.empty(n, dtype=torch.bfloat16, device="cuda"))
    plist = [M.Param(ws[i], ms[i], vs[i], gs[i], w16s[i]) for i in range(len(params))]
    rng = np.random.default_rng(7)
    inf_t = [nm for nm, _ in params].index(c.inf_tensor)
    whole = [t for t, (nm, _) in enumerate(params) if nm in ("embed_tokens", "lm_head")]
    assert len(whole) == 2
    chunk = 2816  # elements per stage of the update kernel's copy pipeline
    samples, host = {}, {}
    for t, (name, n) in enumerate(params):
        if t in whole:
            w0 = to_host(ws[t], np.float32)
            np.testing.assert_array_equal(w0[:4096], synth.fill(c.master_recipe(t), synth.F32, 4096))
            host[t] = [w0, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
            continue
        edges = np.arange(chunk, n, chunk, dtype=np.int64)
        idx = np.unique(np.concatenate([rng.integers(0, n, 96), np.arange(min(n, 8)), np.arange(max(0, n - 8), n),
                                        edges - 1, edges, [c.inject_index] if t == inf_t else []]).astype(np.int64))
        samples[t] = idx
        host[t] = [synth.fill_at(c.master_recipe(t), synth.F32, idx), np.zeros(idx.size, np.float32),
                   np.zeros(idx.size, np.float32), np.zeros(idx.size, np.uint16)]
    ostate = O.new_scaler_state(c.scale)
    st = M.new_scaler_state(c.scale)
    for step in range(1, c.steps + 1):
        for t, (name, n) in enumerate(params):
            synth.fill_device(c.grad_recipe(t, step), synth.F16, gs[t])
        if step == c.inf_step:
            gs[inf_t][c.inject_index] = float("inf")
        found = int(any(bool((~torch.isfinite(g)).any().item()) for g in gs))
        M.mp_adamw_step(plist, ghp, st)
        M.loss_scale_update(st, cfg)
        s_orc = O.adamw_begin(ohp, ostate, found)
        if not found:
            for t in range(len(params)):
                w, m, v, w16 = host[t]
                if t in whole:
                    g = to_host(gs[t], np.uint16)
                    apply_parallel(s_orc, w, m, v, g, O.F16, w16, O.BF16)
                else:
                    g_s = synth.fill_at(c.grad_recipe(t, step), synth.F16, samples[t])
                    O.adamw_apply(s_orc, w, m, v, g_s, O.F16, w16, O.BF16)
        O.loss_scale_update(ostate, ocfg)
        torch.cuda.synchronize()
        gst = M.read_scaler_state(st)
        assert gst.found_inf == found == int(step == c.inf_step)
        assert_state_equal(gst, ostate)
    for t, (name, n) in enumerate(params):
        w, m, v, w16 = host[t]
        if t in whole:
            got = [to_host(ws[t], np.float32), to_host(ms[t], np.float32), to_host(vs[t], np.float32),
                   to_host(w16s[t], np.uint16)]
        else:
            it = torch.from_numpy(samples[t]).cuda()
            got = [ws[t][it].cpu().numpy(), ms[t][it].cpu().numpy(), vs[t][it].cpu().numpy(),
                   to_host(w16s[t][it], np.uint16)]
        for gt, ot, nm in zip(got[:3], (w, m, v), ("w", "m", "v")):
            d = ulp_diff(gt, ot)
            assert d.max() <= MAX_ULP, f"{name} {nm}: {d.max()} ulp"
            assert d.max() == 0, f"{name} {nm}: {d.max()} ulp (within tolerance, not exact)"
        np.testing.assert_array_equal(got[3], w16, err_msg=f"{name} working copy")
        assert bool((ws[t].to(torch.bfloat16).view(torch.int16) == w16s[t].view(torch.int16)).all().item()), \
            f"{name}: working copy is not the RNE of the master"
    assert M.read_scaler_state(st).step == c.steps - 1


def test_check_then_apply_equals_fused_step():
    n = 50_001
    ghp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01)
    w0 = synth.fill(synth.recipe(40, 0, 0.02), synth.F32, n)
    A, B = Tensors(w0, O.F16, O.BF16), Tensors(w0, O.F16, O.BF16)
    sa, sb = M.new_scaler_state(512.0), M.new_scaler_state(512.0)
    for k in range(3):
        g = to_dev(synth.fill(synth.recipe(41, k, 5.0), synth.F16, n), torch.float16)
        A.g.copy_(g)
        B.g.copy_(g)
        M.mp_adamw_step([A.param()], ghp, sa)
        M.mp_adamw_check([B.param()], ghp, sb)
        M.mp_adamw_apply([B.param()], ghp, sb)
    torch.cuda.synchronize()
    for x, y in ((A.w, B.w), (A.m, B.m), (A.v, B.v), (A.w16, B.w16)):
        assert torch.equal(x.view(torch.int8) if x.dtype != torch.float32 else x, y.view(torch.int8) if y.dtype != torch.float32 else y)
    assert bytes(M.read_scaler_state(sa)) == bytes(M.read_scaler_state(sb))


# ---- gradient-norm clipping fused into the check pass -----------------------------


# The kernel sums squares in binary32 in tiles: a lane adds 64 squares, a warp
# folds 32 lanes in 5 steps and a tile its 8 warps in 3, so a tile sum of
# non-negative terms carries at most 72 roundings (71 additions and the square)
# of relative size 2^-24; the tiles are added in binary64 (error below 2^-40
# here).  The square root halves the relative error and the binary32 norm adds
# one rounding: |norm_gpu - norm| <= (36 + 1 + 1) * 2^-24 * norm.  The clip
# coefficient max_norm / (norm + 1e-6) inherits the same relative error.
NORM_REL = 38 * 2.0 ** -24


def assert_norm_close(g_norm, g_coef, o_norm, o_coef, what=""):
    """The kernel's norm and clip coefficient against the oracle's plain
    definition (binary64 sum in element order), within NORM_REL."""
    gn, on = float(np.float32(g_norm)), float(o_norm)
    if np.isfinite(on):
        assert abs(gn - on) <= NORM_REL * on, f"{what} norm {gn!r} vs {on!r} ({abs(gn - on) / on:.3g} rel)"
        gc, oc = float(np.float32(g_coef)), float(np.float32(o_coef))
        assert abs(gc - oc) <= NORM_REL * oc, f"{what} clip {gc!r} vs {oc!r}"
    else:
        assert not np.isfinite(gn) and np.isnan(gn) == np.isnan(on), f"{what} norm {gn} vs {on}"


def test_tiny_step_with_clipping():
    c = W.TINY
    t = golden("scaler_trajectory_tiny.json")
    max_norm = 0.05  # the unscaled grads have a norm near 0.1: clipping is active
    ghp = M.AdamwHparams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, max_norm)
    ohp = O.AdamwHp(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, max_norm)
    cfg, ocfg = M.ScalerCfg(c.growth, c.backoff, c.interval, 1), O.ScalerCfg(c.growth, c.backoff, c.interval, 1)
    w0 = synth.fill(c.master_recipe(), synth.F32, c.n)
    T = Tensors(w0, O.F16, O.F16)
    # An oracle run that forms its own coefficient from its own norm.  The two
    # coefficients differ by a relative delta <= NORM_REL, which scales every
    # clipped grad: a moment moves by at most delta times the sum of its terms'
    # magnitudes (Mabs), v by 2 delta (its terms are positive), and each update
    # step_size * m / den by at most 2 delta * step_size * Mabs / den (summed
    # over the steps in Uabs).  Master weights that an update brings near zero
    # lose their relative accuracy to that cancellation, so the master is
    # bounded in absolute terms by Uabs, not in ulps.
    pw, pm, pv, pw16 = w0.copy(), np.zeros(c.n, np.float32), np.zeros(c.n, np.float32), np.zeros(c.n, np.uint16)
    pst = O.new_scaler_state(c.init_scale)
    Mabs, Uabs = np.zeros(c.n), np.zeros(c.n)
    ws = torch.empty(M.mp_adamw_workspace_size([T.param()]), dtype=torch.uint8, device="cuda")
    st, ost = M.new_scaler_state(c.init_scale), O.new_scaler_state(c.init_scale)
    clipped = 0
    for k in range(1, c.steps + 1):
        S = t["scale_used"][k - 1]
        g = synth.fill(c.grad_recipe(k, S), synth.F16, c.n)
        inj = c.injection(k)
        if inj:
            g[inj[0]] = inj[1]
        T.g.copy_(to_dev(g, torch.float16))
        M.mp_adamw_step([T.param()], ghp, st, workspace=ws)
        M.loss_scale_update(st, cfg)
        torch.cuda.synchronize()
        gs = M.read_scaler_state(st)
        # the update given the kernel's coefficient: bit for bit
        found, norm, coef = O.adamw_step(ohp, ost, [T.oracle_tuple(g)], O.F16, O.F16, clip=gs.clip_coef)
        O.loss_scale_update(ost, ocfg)
        O.adamw_step(ohp, pst, [(pw, pm, pv, g, pw16)], O.F16, O.F16)
        O.loss_scale_update(pst, ocfg)
        assert_state_equal(gs, ost)
        assert_norm_close(gs.grad_norm, gs.clip_coef, norm, coef, f"step {k}")
        clipped += int(coef < 1.0)
        T.compare(f"step {k}")
        if not found:
            gu = O.convert(g, O.F16, O.F32).astype(np.float64) / S
            Mabs = c.beta1 * Mabs + (1 - c.beta1) * np.abs(gu * coef)
            tk = pst.step
            den = np.sqrt(pv.astype(np.float64)) / np.sqrt(1 - c.beta2 ** tk) + c.eps
            Uabs += c.lr / (1 - c.beta1 ** tk) * Mabs / den
        gw, gm, gv = (x.cpu().numpy().astype(np.float64) for x in (T.w, T.m, T.v))
        rnd = 16 * 2.0 ** -24  # the roundings of one update that the two runs take on different values
        for name, got, ref, tol in (
                ("w", gw, pw, 4 * np.spacing(np.abs(pw)) + (2 * NORM_REL + rnd) * 1.01 * Uabs),
                ("m", gm, pm, 4 * np.spacing(np.abs(pm)) + (NORM_REL + rnd) * 1.01 * Mabs),
                ("v", gv, pv, 4 * np.spacing(pv) + (2 * NORM_REL + rnd) * 1.01 * pv.astype(np.float64))):
            bad = np.abs(got - ref) > tol
            assert not bad.any(), f"step {k} {name} vs the independent oracle at {np.flatnonzero(bad)[:5]}"
        d16 = np.abs(T.w16.view(torch.int16).cpu().numpy().astype(np.int32) - pw16.view(np.int16).astype(np.int32))
        assert d16.max() <= 1, f"step {k}: working copy more than one code from the independent oracle"
    assert clipped >= 8


@pytest.mark.parametrize("g_fmt", [O.F16, O.BF16])
def test_ragged_multi_tensor_with_clipping(g_fmt):
    sizes = [1, 7, 16383, 16384, 16385, 40000, 0, 100_003]
    ghp = M.AdamwHparams(3e-3, 0.8, 0.99, 1e-6, 0.1, 0.5)
    ohp = O.AdamwHp(3e-3, 0.8, 0.99, 1e-6, 0.1, 0.5)
    S0 = 256.0 if g_fmt == O.F16 else 1.0
    Ts = [Tensors(synth.fill(synth.recipe(50, i, 0.5), synth.F32, n), g_fmt, O.BF16) for i, n in enumerate(sizes)]
    ws = torch.empty(M.mp_adamw_workspace_size([T.param() for T in Ts]), dtype=torch.uint8, device="cuda")
    st, ost = M.new_scaler_state(S0), O.new_scaler_state(S0)
    for k in range(1, 4):
        hosts = []
        for i, (T, n) in enumerate(zip(Ts, sizes)):
            g = synth.fill(synth.recipe(51, 100 * k + i, float(np.float32(0.01 * S0))),
                           synth.F16 if g_fmt == O.F16 else synth.BF16, n)
            hosts.append(g)
            if n:
                T.g.copy_(to_dev(g, TD[g_fmt]))
        M.mp_adamw_step([T.param() for T in Ts], ghp, st, workspace=ws)
        torch.cuda.synchronize()
        gs = M.read_scaler_state(st)
        found, norm, coef = O.adamw_step(ohp, ost, [T.oracle_tuple(g) for T, g in zip(Ts, hosts)], g_fmt, O.BF16,
                                         clip=gs.clip_coef)
        assert_state_equal(gs, ost)
        assert_norm_close(gs.grad_norm, gs.clip_coef, norm, coef, f"step {k}")
        assert coef < 1.0
        for i, T in enumerate(Ts):
            T.compare(f"step {k} tensor {i}")


def test_clipping_across_launch_groups():
    rng = np.random.default_rng(4)
    sizes = rng.integers(1, 20000, size=600).tolist()
    ghp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0)
    ohp = O.AdamwHp(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0)
    Ts = [Tensors(synth.fill(synth.recipe(60, i, 0.02), synth.F32, n), O.BF16, O.BF16) for i, n in enumerate(sizes)]
    ws = torch.empty(M.mp_adamw_workspace_size([T.param() for T in Ts]), dtype=torch.uint8, device="cuda")
    st, ost = M.new_scaler_state(1.0), O.new_scaler_state(1.0)
    hosts = []
    for i, (T, n) in enumerate(zip(Ts, sizes)):
        g = synth.fill(synth.recipe(61, i, 1e-3), synth.BF16, n)
        hosts.append(g)
        T.g.copy_(to_dev(g, torch.bfloat16))
    M.mp_adamw_check([T.param() for T in Ts], ghp, st, workspace=ws)
    M.mp_adamw_apply([T.param() for T in Ts], ghp, st)
    torch.cuda.synchronize()
    gs = M.read_scaler_state(st)
    found, norm, coef = O.adamw_step(ohp, ost, [T.oracle_tuple(g) for T, g in zip(Ts, hosts)], O.BF16, O.BF16,
                                     clip=gs.clip_coef)
    assert_norm_close(gs.grad_norm, gs.clip_coef, norm, coef)
    for i in (0, 511, 512, 599):
        Ts[i].compare(f"tensor {i}")


def test_full_model_clipping_norm_and_sampled_update():
    """Llama-3-8B list, 2 steps with max_grad_norm 1.0: the norm over all
    8.03e9 grads against the oracle's definition (each tensor's binary64 sum
    of squares on a host thread, from the generator's grads copied back), then
    sampled elements updated with the kernel's checked coefficient."""
    import concurrent.futures as cf

    c = W.FULL
    params = W.llama3_8b_params()
    total = sum(n for _, n in params)
    free, _ = torch.cuda.mem_get_info()
    if free < total * 16 + (8 << 30):
        pytest.skip("not enough device memory for the full model")
    max_norm = 1.0
    ghp = M.AdamwHparams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, max_norm)
    ohp = O.AdamwHp(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, max_norm)
    ws_, ms, vs, gs, w16s = [], [], [], [], []
    for t, (name, n) in enumerate(params):
        w = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.fill_device(c.master_recipe(t), synth.F32, w)
        ws_.append(w)
        ms.append(torch.zeros(n, dtype=torch.float32, device="cuda"))
        vs.append(torch.zeros(n, dtype=torch.float32, device="cuda"))
        gs.append(torch.empty(n, dtype=torch.float16, device="cuda"))
        w16s.append(torch.empty(n, dtype=torch.bfloat16, device="cuda"))
    plist = [M.Param(ws_[i], ms[i], vs[i], gs[i], w16s[i]) for i in range(len(params))]
    work = torch.empty(M.mp_adamw_workspace_size(plist), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(8)
    samples = [np.unique(rng.integers(0, n, 64)).astype(np.int64) for _, n in params]
    ow = [synth.fill_at(c.master_recipe(t), synth.F32, idx) for t, idx in enumerate(samples)]
    om = [np.zeros(i.size, np.float32) for i in samples]
    ov = [np.zeros(i.size, np.float32) for i in samples]
    ow16 = [np.zeros(i.size, np.uint16) for i in samples]
    st, ost = M.new_scaler_state(c.scale), O.new_scaler_state(c.scale)
    for step in (1, 2):
        for t in range(len(params)):
            synth.fill_device(c.grad_recipe(t, step), synth.F16, gs[t])
        M.mp_adamw_step(plist, ghp, st, workspace=work)
        s_orc = O.adamw_begin(ohp, ost, 0)
        inv = s_orc.inv_scale

        def sumsq(t):
            return O.grad_sumsq(to_host(gs[t], np.uint16), O.F16, inv)

        with cf.ThreadPoolExecutor(16) as ex:
            parts = list(ex.map(sumsq, range(len(params))))
        norm = O.norm_of_sumsqs(parts)
        torch.cuda.synchronize()
        gst = M.read_scaler_state(st)
        assert_norm_close(gst.grad_norm, gst.clip_coef, norm, O.clip_coef(norm, max_norm), f"step {step}")
        assert gst.clip_coef < 1.0
        s_orc.clip = gst.clip_coef
        for t, idx in enumerate(samples):
            O.adamw_apply(s_orc, ow[t], om[t], ov[t], synth.fill_at(c.grad_recipe(t, step), synth.F16, idx), O.F16,
                          ow16[t], O.BF16)
    for t, idx in enumerate(samples):
        it = torch.from_numpy(idx).cuda()
        for gt, ot in ((ws_[t], ow[t]), (ms[t], om[t]), (vs[t], ov[t])):
            assert ulp_diff(gt[it].cpu().numpy(), ot).max() == 0, params[t][0]
        np.testing.assert_array_equal(to_host(w16s[t][it], np.uint16), ow16[t])
