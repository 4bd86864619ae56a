"""Checkpoint and resume: the optimizer and FP8 delayed-scaling state are plain
device buffers, so 12 steps in a row must equal 6 steps, a copy of every state
buffer to the host, a restore into fresh device buffers and 6 more steps -- bit
for bit, with an inf step on each side of the cut."""
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


SIZES = (200_003, 4096, 9)
INF_STEPS = {3: (0, 17), 8: (2, 4)}  # step -> (tensor, element)


class Replica:
    def __init__(self):
        self.w = [torch.from_numpy(synth.fill(synth.recipe(90 + t, 0, 0.02), synth.F32, n)).cuda()
                  for t, n in enumerate(SIZES)]
        self.m = [torch.zeros_like(w) for w in self.w]
        self.v = [torch.zeros_like(w) for w in self.w]
        self.w16 = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for n in SIZES]
        self.g = [torch.zeros(n, dtype=torch.float16, device="cuda") for n in SIZES]
        self.st = M.new_scaler_state(65536.0)
        self.meta, self.hist = M.new_fp8_meta(), torch.zeros(8, device="cuda")
        self.y = torch.zeros(128 * 256, dtype=torch.uint8, device="cuda")

    def buffers(self):
        return self.w + self.m + self.v + self.w16 + [self.st, self.meta, self.hist]

    def step(self, k, hp, cfg):
        for t, n in enumerate(SIZES):
            g = synth.fill(synth.recipe(95 + t, k, 1e-4 * 65536), synth.F16, n)
            if k in INF_STEPS and INF_STEPS[k][0] == t:
                g[INF_STEPS[k][1]] = np.float16(np.inf).view(np.uint16)
            self.g[t].copy_(torch.from_numpy(g.view(np.int16)).view(torch.float16))
        params = [M.Param(self.w[t], self.m[t], self.v[t], self.g[t], self.w16[t]) for t in range(len(SIZES))]
        M.mp_adamw_step(params, hp, self.st, working_dtype=M.MP_BF16)
        M.loss_scale_update(self.st, cfg)
        x = synth.fill(synth.recipe(99, k, 2.0 ** (k % 4)), synth.BF16, 128 * 256)
        xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        M.fp8_cast_delayed(xt, self.y, M.MP_E4M3, self.meta, self.hist, 1.0)


def test_resume_from_host_copies_is_bit_identical():
    c = W.TINY
    hp = M.AdamwHparams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay)
    cfg = M.ScalerCfg(2.0, 0.5, 3, 1)
    straight = Replica()
    for k in range(12):
        straight.step(k, hp, cfg)
    first = Replica()
    for k in range(6):
        first.step(k, hp, cfg)
    torch.cuda.synchronize()
    saved = [b.cpu().clone() for b in first.buffers()]  # the checkpoint
    del first
    resumed = Replica()
    for dst, src in zip(resumed.buffers(), saved):
        dst.copy_(src)
    for k in range(6, 12):
        resumed.step(k, hp, cfg)
    torch.cuda.synchronize()
    for a, b in zip(straight.buffers() + [straight.y], resumed.buffers() + [resumed.y]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    st = M.read_scaler_state(resumed.st)
    assert st.step == 10 and st.skipped == 2
