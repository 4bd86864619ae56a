"""Every entry point is stream-ordered, allocation-free and free of host
synchronisation, so a whole step can be captured in a CUDA graph.  A captured
step replayed over several steps (inputs refreshed between replays, an inf on
one step) must leave exactly the state the same calls leave when run eagerly."""
import numpy as np
import pytest
import torch

import synth
import synth.workloads as W

import mixed_precision_numerics_gb300 as M  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


SIZES = (300_001, 65_536, 17)
STEPS = 6
INF_STEP = 3


def grads(step):
    out = []
    for t, n in enumerate(SIZES):
        g = synth.fill(synth.recipe(70 + t, step, 1e-4 * 65536), synth.F16, n)
        if step == INF_STEP and t == 1:
            g[123] = np.float16(np.inf).view(np.uint16)
        out.append(torch.from_numpy(g.view(np.int16)).view(torch.float16).cuda())
    return out


class Step:
    """All state of one replica: optimizer, FP8 casts (delayed, transposed,
    blockwise), NVFP4 and MX outputs."""

    def __init__(self, clip: bool):
        self.params = []
        for t, n in enumerate(SIZES):
            w = torch.from_numpy(synth.fill(synth.recipe(60 + t, 0, 0.02), synth.F32, n)).cuda()
            self.params.append(M.Param(w, torch.zeros_like(w), torch.zeros_like(w),
                                       torch.zeros(n, dtype=torch.float16, device="cuda"),
                                       torch.zeros(n, dtype=torch.bfloat16, device="cuda")))
        self.hp = M.AdamwHparams(1e-3, 0.9, 0.999, 1e-8, 0.01, 0.05 if clip else 0.0)
        self.ws = torch.zeros(M.mp_adamw_workspace_size(self.params), dtype=torch.uint8, device="cuda")
        self.st = M.new_scaler_state(65536.0)
        self.cfg = M.ScalerCfg(2.0, 0.5, 2, 1)
        self.x = torch.zeros((256, 512), dtype=torch.bfloat16, device="cuda")
        self.y8 = torch.zeros(256 * 512, dtype=torch.uint8, device="cuda")
        self.meta, self.hist = M.new_fp8_meta(), torch.zeros(4, device="cuda")
        self.codes = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
        self.sc = torch.zeros((256, 32), dtype=torch.uint8, device="cuda")
        self.ts = torch.zeros(1, device="cuda")
        self.nf = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.nws = M.new_nvfp4_workspace()
        self.mxc = torch.zeros(256 * 256, dtype=torch.uint8, device="cuda")
        self.mxs = torch.zeros((256, 16), dtype=torch.uint8, device="cuda")
        # the tile casts read x through 2-D tensor copies (their tensor maps
        # travel as kernel parameters, so the graph holds them by value)
        self.yT, self.yTt = (torch.zeros(256 * 512, dtype=torch.uint8, device="cuda") for _ in range(2))
        self.metaT, self.histT = M.new_fp8_meta(), torch.zeros(3, device="cuda")
        self.yb1, self.yb2 = (torch.zeros(256 * 512, dtype=torch.uint8, device="cuda") for _ in range(2))
        self.sb1 = torch.zeros((256, 4), dtype=torch.float32, device="cuda")
        self.sb2 = torch.zeros((2, 4), dtype=torch.float32, device="cuda")

    def load_inputs(self, step):
        for p, g in zip(self.params, grads(step)):
            p.grad.copy_(g)
        x = synth.fill(synth.recipe(80, step, 2.0 ** (step % 3)), synth.BF16, 256 * 512)
        self.x.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).reshape(256, 512))

    def run(self):
        M.mp_adamw_step(self.params, self.hp, self.st, workspace=self.ws)
        M.loss_scale_update(self.st, self.cfg)
        M.fp8_cast_delayed(self.x, self.y8, M.MP_E4M3, self.meta, self.hist, 1.0)
        M.nvfp4_quantize(self.x, self.codes, self.sc, self.ts, self.nf, self.nws, stochastic=True, seed=99,
                         apply_rht=True, sign_mask=0xE3BF)
        M.mx_quantize(self.x, self.mxc, self.mxs, M.MP_E2M1)
        M.fp8_cast_transpose_delayed(self.x, self.yT, self.yTt, M.MP_E5M2, self.metaT, self.histT, 2.0)
        M.fp8_quantize_blockwise(self.x, self.yb1, self.sb1, 1, 128)
        M.fp8_quantize_blockwise(self.x, self.yb2, self.sb2, 128, 128)

    def snapshot(self):
        out = [self.st.clone(), self.meta.clone(), self.hist.clone(), self.y8.clone(), self.codes.clone(),
               self.sc.clone(), self.ts.clone(), self.mxc.clone(), self.mxs.clone(), self.yT.clone(),
               self.yTt.clone(), self.metaT.clone(), self.histT.clone(), self.yb1.clone(), self.yb2.clone(),
               self.sb1.clone(), self.sb2.clone()]
        for p in self.params:
            out += [p.master.clone(), p.exp_avg.clone(), p.exp_avg_sq.clone(), p.working.clone()]
        return [t.view(torch.uint8) if t.dtype != torch.uint8 else t for t in out]


@pytest.mark.parametrize("clip", [False, True])
def test_captured_step_replays_like_eager_calls(clip):
    # one throwaway eager step first: the library's one-time host queries
    # (device attributes, occupancy) happen outside the capture
    warm = Step(clip)
    warm.load_inputs(0)
    warm.run()
    torch.cuda.synchronize()
    eager, graphed = Step(clip), Step(clip)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        graphed.load_inputs(0)  # first touch outside the capture
        with torch.cuda.graph(g, stream=side):
            graphed.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for step in range(STEPS):
        eager.load_inputs(step)
        eager.run()
        graphed.load_inputs(step)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager.snapshot(), graphed.snapshot()):
            assert torch.equal(a.flatten(), b.flatten()), f"step {step}"
    st = M.read_scaler_state(graphed.st)
    assert st.step == STEPS - 1 and st.skipped == 1  # the inf step was skipped inside the graph
