"""The five synthetic workloads: shapes, seeds and value distributions.

Every tensor is a recipe for ``synth`` (seed, stream, sigma, outliers), so the
tests and the benchmark build bit-identical inputs on the host or on the
device, and any element can be regenerated on its own.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import BF16, F16, F32, OUT_NONE, OUT_SCALE, OUT_T3, hash64, recipe

F16_POS_INF = 0x7C00
F16_NAN = 0x7E00


def f32(x: float) -> float:
    return float(np.float32(x))


# ---- tiny fused step (+ tiny FP8 cast) ------------------------------------------------
@dataclass(frozen=True)
class TinyStep:
    n: int = 1_048_576
    seed: int = 0
    w_sigma: float = 0.02
    g_sigma: float = 1e-4
    steps: int = 12
    inf_step: int = 3
    nan_step: int = 7
    inject_index: int = 12345
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    init_scale: float = 65536.0
    growth: float = 2.0
    backoff: float = 0.5
    interval: int = 4

    def master_recipe(self):
        return recipe(self.seed, 0x100, self.w_sigma)

    def grad_recipe(self, step: int, scale: float):
        return recipe(self.seed, 0x1000 + step, f32(f32(self.g_sigma) * f32(scale)))

    def injection(self, step: int):
        """(index, f16 bits) written over the generated grad on this step, or None."""
        if step == self.inf_step:
            return self.inject_index, F16_POS_INF
        if step == self.nan_step:
            return self.inject_index, F16_NAN
        return None


TINY = TinyStep()


@dataclass(frozen=True)
class TinyFp8:
    rows: int = 1024
    cols: int = 1024
    seed: int = 1
    iters: int = 20
    hist_len: int = 16
    margin: float = 1.0

    def recipe(self, k: int):
        return recipe(self.seed, k, 1.0)


TINY_FP8 = TinyFp8()


# ---- FP8 delayed-scaling cast ----------------------------------------------------------
@dataclass(frozen=True)
class Fp8Cast:
    rows: int = 8192
    cols: int = 4096
    iters: int = 64
    hist_len: int = 1024
    margin: float = 1.0
    drift: float = 1.05
    act_seed: int = 2
    grad_seed: int = 3
    act_outlier_p: float = 0.001
    act_outlier_mult: float = 50.0
    grad_sigma: float = 1e-3

    def act_recipe(self, k: int):
        return recipe(self.act_seed, k, f32(self.drift**k), self.act_outlier_p, self.act_outlier_mult, OUT_SCALE,
                      outlier_stream=0xACC)

    def grad_recipe(self, k: int):
        return recipe(self.grad_seed, k, f32(self.grad_sigma * self.drift**k))


FP8 = Fp8Cast()


# ---- NVFP4 RNE (activations 1x16, weights 16x16) -----------------------------------------
@dataclass(frozen=True)
class Nvfp4Rne:
    act_rows: int = 16384
    act_cols: int = 5120
    w_rows: int = 5120
    w_cols: int = 5120

    def act_recipe(self):
        return recipe(4, 0, 1.0, 0.005, 30.0, OUT_SCALE)

    def w_recipe(self):
        return recipe(5, 0, 0.02)


NVFP4_RNE = Nvfp4Rne()


# ---- NVFP4 gradient path (RHT + 1x16 + SR) ----------------------------------------------
@dataclass(frozen=True)
class Nvfp4Grad:
    rows: int = 8192
    cols: int = 12288
    sigma: float = 1e-3
    outlier_p: float = 0.001
    outlier_mult: float = 30.0
    sr_seed: int = 1234

    def recipe(self):
        return recipe(6, 0, self.sigma, self.outlier_p, self.outlier_mult, OUT_T3)

    def sign_mask(self) -> int:
        """Random signs of the Hadamard diagonal: 16 bits drawn from the generator."""
        return hash64(self.sr_seed, 0x52485400, 0) & 0xFFFF


NVFP4_GRAD = Nvfp4Grad()


# ---- full-model optimizer step (Llama-3-8B-shaped parameter list) -----------------------
def llama3_8b_params():
    """[(name, numel)] in model order: embedding, 32 decoder layers, lm_head."""
    h, kv, ff, vocab = 4096, 1024, 14336, 128256
    out = [("embed_tokens", vocab * h)]
    for i in range(32):
        p = f"layers.{i}."
        out += [(p + "attn.q", h * h), (p + "attn.k", kv * h), (p + "attn.v", kv * h), (p + "attn.o", h * h),
                (p + "mlp.gate", ff * h), (p + "mlp.up", ff * h), (p + "mlp.down", h * ff),
                (p + "input_norm", h), (p + "post_norm", h)]
    out.append(("lm_head", vocab * h))
    return out


@dataclass(frozen=True)
class FullStep:
    seed: int = 7
    steps: int = 5
    inf_step: int = 3
    inf_tensor: str = "layers.17.mlp.up"
    inject_index: int = 12345
    w_sigma: float = 0.02
    g_sigma: float = 1e-4
    scale: float = 65536.0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    growth: float = 2.0
    backoff: float = 0.5
    interval: int = 2000

    def master_recipe(self, t: int):
        return recipe(self.seed, 0x100000 + t, self.w_sigma)

    def grad_recipe(self, t: int, step: int):
        return recipe(self.seed, 0x200000 + t * 16 + step, f32(f32(self.g_sigma) * f32(self.scale)))


FULL = FullStep()
