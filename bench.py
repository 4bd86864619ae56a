#!/usr/bin/env python
"""Whole hot-path throughput of the mixed-precision machinery on GB300.

One step = one pass over every part of the hot path on one batch of
synthetic input, all of it resident in HBM before timing starts:
  * the fused optimizer step of a Llama-3-8B-shaped model (290 tensors,
    8,030,257,152 params, FP16 grads scaled by 65536, FP32 master/m/v, BF16
    working copy): inf/NaN check pass, AdamW update pass, loss-scale update;
  * FP8 delayed-scaling casts of a [8192 x 4096] BF16 activation to E4M3 and
    a [8192 x 4096] BF16 gradient to E5M2 (history 1024), each step on the
    next of 64 pre-generated inputs with drifting std;
  * NVFP4: [16384 x 5120] activations 1x16 RNE, [5120 x 5120] weights 16x16
    RNE, [8192 x 12288] gradients with the random Hadamard transform, 1x16
    blocks and stochastic rounding.
The metric is HBM GB/s of algorithmic bytes (minimum bytes each call must
move), whole step and per call, with the dominant call against the measured
HBM copy peak.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HBM GB/s and % of GB300 HBM roofline per kernel (AdamW step, FP8 cast, NVFP4)"
UNIT = "GB/s"
HBM_FALLBACK_GBS = 6800.0

# algorithmic bytes per unit (element or parameter)
B_CHECK = 2.0            # read the 16-bit grad once
B_APPLY = 28.0           # read g (2) + w, m, v (12); write w, m, v (12) + w16 (2)
B_FP8 = 3.0              # read 16-bit x (2); write 1 byte
B_NVFP4_1X16 = 2 + 2 + 0.5 + 1 / 16    # amax pass, encode pass, codes, 1x16 scales
B_NVFP4_2D = 2 + 2 + 0.5 + 1 / 256     # 16x16 scales


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--small", action="store_true",
                   help="profiling case: optimizer over decoder layer 0 only (218M params), 2 FP8 inputs")
    p.add_argument("--trace", metavar="PATH",
                   help="write one JSON line per timed step (loss scale, skip count, FP8 amax/scale, NVFP4 tensor "
                        "scales, per-call ms) to PATH; adds a few small device-to-host copies per step")
    return p.parse_args()


# ---------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; weak scaling, no collective on the data path)
# ---------------------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(world, backend: str = "nccl"):
    """One process per GPU over NCCL; the CPU tests use gloo."""
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend)


def _backend():
    import torch.distributed as dist

    return dist.get_backend()


def barrier(world):
    if world > 1:
        import torch
        import torch.distributed as dist

        if _backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if _backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: float, elapsed_ms: float, world: int):
    """Whole-job throughput: the bytes every rank processed over the slowest
    rank's time (weak scaling: each rank runs the same work).  Returns
    (GB/s, slowest rank's ms)."""
    slowest = max_over_ranks(elapsed_ms, world)
    return world * bytes_per_rank / (slowest * 1e-3) / 1e9, slowest


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(dev: int) -> str | None:
    import torch

    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------------------------------
# peaks, profile-derived traffic
# ---------------------------------------------------------------------------------------
def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("mp_adamw.cu", "mp_device.cuh"):
        with open(os.path.join(ROOT, "mixed_precision_numerics_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "adamw_update_traffic.json")


def profiled_traffic(params: int):
    """DRAM bytes of one update launch over `params` parameters, from the
    committed ncu record of a smaller capture of the same kernel, or None when
    that record was taken on different kernel source.  Reads scale with the
    parameters (the capture read exactly 14 B/param); writes are 14 B/param
    less the bytes the capture left dirty in L2 at kernel end (a constant of
    the cache, not of the parameter count).  Returns (read, write, residue)."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    n = rec["capture_params"]
    read = rec["dram_bytes_read"] / n * params
    residue = B_APPLY / 2 * n - rec["dram_bytes_write"]
    return read, B_APPLY / 2 * params - residue, residue


# ---------------------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------------------
class Workload:
    def __init__(self, small: bool):
        import torch

        import mixed_precision_numerics_gb300 as M
        import synth
        import synth.workloads as W

        self.M, self.torch = M, torch
        c = W.FULL
        params = W.llama3_8b_params()
        if small:
            params = [(n, k) for n, k in params if n.startswith("layers.0.")]
        self.param_names = [n for n, _ in params]
        self.P = sum(k for _, k in params)
        self.tensors = []
        for t, (name, n) in enumerate(params):
            w = torch.empty(n, dtype=torch.float32, device="cuda")
            synth.fill_device(c.master_recipe(t), synth.F32, w)
            g = torch.empty(n, dtype=torch.float16, device="cuda")
            synth.fill_device(c.grad_recipe(t, 1), synth.F16, g)
            self.tensors.append(M.Param(w, torch.zeros_like(w), torch.zeros_like(w), g,
                                        torch.empty(n, dtype=torch.bfloat16, device="cuda")))
        self.params = M.make_param_array(self.tensors)
        self.hp = M.AdamwHparams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay)
        self.cfg = M.ScalerCfg(c.growth, c.backoff, c.interval, 1)
        self.state = M.new_scaler_state(c.scale)

        f = W.FP8
        self.nbuf = 2 if small else f.iters
        self.fp8_n = f.rows * f.cols
        self.fp8_rows_cols = (f.rows, f.cols)
        self.act = [torch.empty(self.fp8_n, dtype=torch.bfloat16, device="cuda") for _ in range(self.nbuf)]
        self.grd = [torch.empty(self.fp8_n, dtype=torch.bfloat16, device="cuda") for _ in range(self.nbuf)]
        for k in range(self.nbuf):
            synth.fill_device(f.act_recipe(k), synth.BF16, self.act[k])
            synth.fill_device(f.grad_recipe(k), synth.BF16, self.grd[k])
        self.y_act = torch.empty(self.fp8_n, dtype=torch.uint8, device="cuda")
        self.y_grd = torch.empty(self.fp8_n, dtype=torch.uint8, device="cuda")
        self.meta_act, self.meta_grd = M.new_fp8_meta(), M.new_fp8_meta()
        self.hist_act = torch.zeros(f.hist_len, dtype=torch.float32, device="cuda")
        self.hist_grd = torch.zeros(f.hist_len, dtype=torch.float32, device="cuda")
        self.fp8_margin = f.margin

        r, g4 = W.NVFP4_RNE, W.NVFP4_GRAD
        self.q = []
        self.extra_bytes = {}
        for name, rows, cols, rec, b2, sr, rht, seed, mask in (
            ("nvfp4_act_1x16_rne", r.act_rows, r.act_cols, r.act_recipe(), False, False, False, 0, 0),
            ("nvfp4_w_16x16_rne", r.w_rows, r.w_cols, r.w_recipe(), True, False, False, 0, 0),
            ("nvfp4_grad_rht_1x16_sr", g4.rows, g4.cols, g4.recipe(), False, True, True, g4.sr_seed, g4.sign_mask()),
        ):
            x = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
            synth.fill_device(rec, synth.BF16, x)
            self.q.append(dict(
                name=name, x=x, rows=rows, cols=cols, b2=b2, sr=sr, rht=rht, seed=seed, mask=mask,
                codes=torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda"),
                scales=torch.empty((rows // 16 if b2 else rows, cols // 16), dtype=torch.uint8, device="cuda"),
                ts=torch.zeros(1, dtype=torch.float32, device="cuda"),
                nf=torch.zeros(1, dtype=torch.int32, device="cuda"),
                ws=M.new_nvfp4_workspace(),
                bytes=(B_NVFP4_2D if b2 else B_NVFP4_1X16) * rows * cols,
            ))
        torch.cuda.synchronize()

        # algorithmic bytes per call, in step order
        self.calls = ["adamw_check", "adamw_apply", "loss_scale_update", "fp8_act_e4m3", "fp8_grad_e5m2"] + \
                     [q["name"] for q in self.q]
        self.bytes = {"adamw_check": B_CHECK * self.P, "adamw_apply": B_APPLY * self.P, "loss_scale_update": 0.0,
                      "fp8_act_e4m3": B_FP8 * self.fp8_n, "fp8_grad_e5m2": B_FP8 * self.fp8_n}
        for q in self.q:
            self.bytes[q["name"]] = q["bytes"]
        self.step_bytes = sum(self.bytes.values())
        # units (parameters or elements) per call, for elements/s
        self.units = {"adamw_check": self.P, "adamw_apply": self.P, "loss_scale_update": 0,
                      "fp8_act_e4m3": self.fp8_n, "fp8_grad_e5m2": self.fp8_n}
        for q in self.q:
            self.units[q["name"]] = q["rows"] * q["cols"]
        self.units["fp8_act_e4m3_with_transpose"] = self.units["fp8_blockwise_1x128_act"] = self.fp8_n
        self.units["fp8_blockwise_128x128_w"] = r.w_rows * r.w_cols
        self.units["mxfp4_act"] = self.units["mxfp8_e4m3_act"] = self.units["mxfp6_e2m3_act"] = r.act_rows * r.act_cols
        self.units["rht16_bf16_grad"] = g4.rows * g4.cols

    def step(self, k: int, ev=None):
        """Enqueue one step on the current stream; ev: list of len(calls)+1 events."""
        M = self.M
        rec = (lambda i: ev[i].record()) if ev is not None else (lambda i: None)
        rec(0)
        M.mp_adamw_check(self.params, self.hp, self.state, grad_dtype=M.MP_F16)
        rec(1)
        M.mp_adamw_apply(self.params, self.hp, self.state, grad_dtype=M.MP_F16, working_dtype=M.MP_BF16)
        rec(2)
        M.loss_scale_update(self.state, self.cfg)
        rec(3)
        b = k % self.nbuf
        M.fp8_cast_delayed(self.act[b], self.y_act, M.MP_E4M3, self.meta_act, self.hist_act, self.fp8_margin)
        rec(4)
        M.fp8_cast_delayed(self.grd[b], self.y_grd, M.MP_E5M2, self.meta_grd, self.hist_grd, self.fp8_margin)
        rec(5)
        for i, q in enumerate(self.q):
            M.nvfp4_quantize(q["x"], q["codes"], q["scales"], q["ts"], q["nf"], q["ws"], block_2d=q["b2"],
                             stochastic=q["sr"], seed=q["seed"], apply_rht=q["rht"], sign_mask=q["mask"])
            rec(6 + i)

    # ---- per-step trace (optional) ---------------------------------------------------------
    def trace_buffers(self, steps: int):
        """Pinned host rows, one per step: scaler state, both FP8 metas, and the
        tensor scale and flag of each NVFP4 call."""
        torch = self.torch
        return {"state": torch.empty((steps, 88), dtype=torch.uint8, pin_memory=True),
                "meta": torch.empty((steps, 2, 32), dtype=torch.uint8, pin_memory=True),
                "ts": torch.empty((steps, len(self.q)), dtype=torch.float32, pin_memory=True),
                "nf": torch.empty((steps, len(self.q)), dtype=torch.int32, pin_memory=True)}

    def trace_copy(self, tr, k: int):
        """Stream-ordered copies of step k's state into row k (no synchronisation)."""
        tr["state"][k].copy_(self.state, non_blocking=True)
        tr["meta"][k, 0].copy_(self.meta_act, non_blocking=True)
        tr["meta"][k, 1].copy_(self.meta_grd, non_blocking=True)
        for i, q in enumerate(self.q):
            tr["ts"][k, i].copy_(q["ts"][0], non_blocking=True)
            tr["nf"][k, i].copy_(q["nf"][0], non_blocking=True)

    def trace_record(self, tr, k: int) -> dict:
        M = self.M
        st = M.ScalerState.from_buffer_copy(tr["state"][k].numpy().tobytes())
        metas = [M.Fp8Meta.from_buffer_copy(tr["meta"][k, j].numpy().tobytes()) for j in range(2)]
        return {"loss_scale": st.scale, "found_inf": st.found_inf, "skipped": st.skipped, "applied_steps": st.step,
                "growth_tracker": st.growth_tracker,
                "fp8": {name: {"amax": m.amax, "next_scale": m.scale, "pos": m.pos}
                        for name, m in zip(("act_e4m3", "grad_e5m2"), metas)},
                "nvfp4": {q["name"]: {"tensor_scale": float(tr["ts"][k, i]), "nonfinite": int(tr["nf"][k, i])}
                          for i, q in enumerate(self.q)}}

    def clipped_check_ms(self, reps: int = 5) -> float:
        """The check pass with gradient-norm clipping (max norm 1.0) on the same
        parameter list: tile sums of g*g plus the one-CTA fold."""
        torch, M = self.torch, self.M
        hp = M.AdamwHparams(self.hp.lr, self.hp.beta1, self.hp.beta2, self.hp.eps, self.hp.weight_decay, 1.0)
        ws = torch.empty(M.mp_adamw_workspace_size(self.params), dtype=torch.uint8, device="cuda")
        state = M.new_scaler_state(65536.0)
        M.mp_adamw_check(self.params, hp, state, grad_dtype=M.MP_F16, workspace=ws)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
        for k in range(reps):
            ev[2 * k].record()
            M.mp_adamw_check(self.params, hp, state, grad_dtype=M.MP_F16, workspace=ws)
            ev[2 * k + 1].record()
        torch.cuda.synchronize()
        return statistics.median(ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(reps))

    def isolated_call_times(self, reps: int = 16) -> dict:
        """Microseconds per call of each FP8 / NVFP4 / MX call, replayed from a
        CUDA graph.  Consecutive calls read different copies of their input and
        write different copies of their outputs (each set more than twice the
        L2), so no call finds its input in L2 and no output is rewritten while
        its lines still sit dirty in L2."""
        torch, M = self.torch, self.M
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size

        def rot(x, clone=True):
            nbytes = x.numel() * x.element_size()
            n = 1 if nbytes < (4 << 20) else min(reps, max(1, -(-2 * l2 // nbytes)))
            return [x] + [x.clone() if clone else torch.empty_like(x) for _ in range(n - 1)]

        def pick(lst, k):
            return lst[k % len(lst)]

        xs = {q["name"]: rot(q["x"]) for q in self.q}
        f = self.fp8_rows_cols
        n_fp8 = self.fp8_n
        y8 = rot(self.y_act, clone=False)
        y8g = rot(self.y_grd, clone=False)
        calls = {
            "fp8_act_e4m3": lambda k: M.fp8_cast_delayed(self.act[k % self.nbuf], pick(y8, k), M.MP_E4M3,
                                                         self.meta_act, self.hist_act, self.fp8_margin),
            "fp8_grad_e5m2": lambda k: M.fp8_cast_delayed(self.grd[k % self.nbuf], pick(y8g, k), M.MP_E5M2,
                                                          self.meta_grd, self.hist_grd, self.fp8_margin),
        }
        # calls outside the step, each with its algorithmic bytes per call
        yt = rot(torch.empty(n_fp8, dtype=torch.uint8, device="cuda"), clone=False)
        calls["fp8_act_e4m3_with_transpose"] = lambda k: M.fp8_cast_transpose_delayed(
            self.act[k % self.nbuf].view(*f), pick(y8, k), pick(yt, k), M.MP_E4M3, self.meta_act, self.hist_act,
            self.fp8_margin)
        self.extra_bytes["fp8_act_e4m3_with_transpose"] = (B_FP8 + 1.0) * n_fp8  # read 2, write y 1 and y_t 1
        sc128 = torch.empty(f[0] * (f[1] // 128), dtype=torch.float32, device="cuda")
        calls["fp8_blockwise_1x128_act"] = lambda k: M.fp8_quantize_blockwise(
            self.act[k % self.nbuf].view(*f), pick(y8, k), sc128, 1, 128)
        self.extra_bytes["fp8_blockwise_1x128_act"] = (3.0 + 4.0 / 128) * n_fp8
        wq = self.q[1]
        wr = xs[wq["name"]]
        yw = rot(torch.empty(wq["rows"] * wq["cols"], dtype=torch.uint8, device="cuda"), clone=False)
        scw = torch.empty(-(-wq["rows"] // 128) * -(-wq["cols"] // 128), dtype=torch.float32, device="cuda")
        calls["fp8_blockwise_128x128_w"] = lambda k: M.fp8_quantize_blockwise(pick(wr, k), pick(yw, k), scw, 128, 128)
        self.extra_bytes["fp8_blockwise_128x128_w"] = (3.0 + 4.0 / 16384) * wq["rows"] * wq["cols"]
        aq = self.q[0]
        n_a = aq["rows"] * aq["cols"]
        ar = xs[aq["name"]]
        mx_c = rot(torch.empty(n_a, dtype=torch.uint8, device="cuda"), clone=False)
        mx_s = rot(torch.empty(n_a // 32, dtype=torch.uint8, device="cuda"), clone=False)
        calls["mxfp4_act"] = lambda k: M.mx_quantize(pick(ar, k), pick(mx_c, k)[: n_a // 2], pick(mx_s, k), M.MP_E2M1)
        self.extra_bytes["mxfp4_act"] = (2.5 + 1.0 / 32) * n_a
        calls["mxfp8_e4m3_act"] = lambda k: M.mx_quantize(pick(ar, k), pick(mx_c, k), pick(mx_s, k), M.MP_E4M3)
        self.extra_bytes["mxfp8_e4m3_act"] = (3.0 + 1.0 / 32) * n_a
        calls["mxfp6_e2m3_act"] = lambda k: M.mx_quantize(pick(ar, k), pick(mx_c, k), pick(mx_s, k), M.MP_E2M3)
        self.extra_bytes["mxfp6_e2m3_act"] = (3.0 + 1.0 / 32) * n_a  # one FP6 code per byte
        gq = self.q[2]
        gr = xs[gq["name"]]
        ry = rot(torch.empty_like(gq["x"]), clone=False)
        calls["rht16_bf16_grad"] = lambda k: M.rht16(pick(gr, k), pick(ry, k), gq["mask"])
        self.extra_bytes["rht16_bf16_grad"] = 4.0 * gq["rows"] * gq["cols"]  # read 2, write 2
        for q in self.q:
            qc, qs = rot(q["codes"], clone=False), rot(q["scales"], clone=False)
            calls[q["name"]] = (lambda q, xr, qc, qs: lambda k: M.nvfp4_quantize(
                pick(xr, k), pick(qc, k), pick(qs, k), q["ts"], q["nf"], q["ws"], block_2d=q["b2"],
                stochastic=q["sr"], seed=q["seed"], apply_rht=q["rht"], sign_mask=q["mask"]))(q, xs[q["name"]], qc, qs)
        clean = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        out = {}
        for name, fn in calls.items():
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    for k in range(reps):
                        fn(k)
            torch.cuda.current_stream().wait_stream(side)
            clean.sum()  # read-only pass: leaves L2 holding clean lines
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            out[name] = a.elapsed_time(b) * 1e3 / reps
        return out

    # ---- end to end through host buffers -------------------------------------------------
    def e2e_setup(self):
        """Pinned host copies of every input, pinned host buffers for the
        results, and a second device input set so that a step's inputs can be
        copied in while the previous step runs.  One pinned buffer per tensor:
        the host allocator rounds each allocation up to a power of two, which
        costs less per tensor (about 20 GB for the step's 16.6 GB) than for one
        block holding them all (32 GB); the copy rate is the same either way."""
        torch, M = self.torch, self.M

        def pinned_copy(d):
            h = torch.empty(d.shape, dtype=d.dtype, pin_memory=True)
            h.copy_(d)
            return h

        self.h_grads = [pinned_copy(t.grad) for t in self.tensors]
        self.h_act = [pinned_copy(a) for a in self.act[:2]]
        self.h_grd = [pinned_copy(g) for g in self.grd[:2]]
        self.h_q = [pinned_copy(q["x"]) for q in self.q]
        self.h_out_fp8 = [torch.empty(self.fp8_n, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
        self.h_out_q = [(torch.empty(q["codes"].shape, dtype=torch.uint8, pin_memory=True),
                         torch.empty(q["scales"].shape, dtype=torch.uint8, pin_memory=True)) for q in self.q]
        self.h_small = torch.empty(88 + 64 + 3 * 8, dtype=torch.uint8, pin_memory=True)
        self.h2d = sum(h.numel() * h.element_size() for h in self.h_grads) + 2 * self.fp8_n * 2 + \
            sum(h.numel() * h.element_size() for h in self.h_q)
        self.d2h = 2 * self.fp8_n + sum(c.numel() + s.numel() for c, s in self.h_out_q) + 88 + 64 + 24
        # device input sets 0 and 1: the grads the parameter table points at, and the quantiser inputs
        grads1 = [torch.empty_like(t.grad) for t in self.tensors]
        tensors1 = [M.Param(t.master, t.exp_avg, t.exp_avg_sq, g, t.working) for t, g in zip(self.tensors, grads1)]
        self.in_sets = [
            dict(params=self.params, grads=[t.grad for t in self.tensors], qx=[q["x"] for q in self.q]),
            dict(params=M.make_param_array(tensors1), grads=grads1, qx=[torch.empty_like(q["x"]) for q in self.q]),
        ]
        self.copy_stream = torch.cuda.Stream()

    def h2d_link_gbs(self) -> float:
        """Host-to-device bandwidth of this machine: one 1 GiB pinned copy, best of 3."""
        torch = self.torch
        h = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
        d = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
        best = 0.0
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            d.copy_(h, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            best = max(best, (1 << 30) / (a.elapsed_time(b) * 1e-3) / 1e9)
        return best

    def e2e_copy_only_ms(self, reps: int = 3) -> float:
        """Milliseconds to copy one step's inputs in, with no kernels running:
        the floor of the pipelined end-to-end step on this machine."""
        torch = self.torch
        cur = torch.cuda.current_stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        for e in free:
            e.record(cur)
        self.copy_stream.wait_stream(cur)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.copy_stream)
        for k in range(reps):
            self.e2e_copy_in(k, copied, free)
        b.record(self.copy_stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def e2e_copy_in(self, k: int, copied, free):
        """On the copy stream: step k's inputs into device set k % 2, once the
        step that last read that set is done."""
        torch = self.torch
        cs, st = self.copy_stream, self.in_sets[k % 2]
        cs.wait_event(free[k % 2])
        with torch.cuda.stream(cs):
            for d, h in zip(st["grads"], self.h_grads):
                d.copy_(h, non_blocking=True)
            self.act[k % 2].copy_(self.h_act[k % 2], non_blocking=True)
            self.grd[k % 2].copy_(self.h_grd[k % 2], non_blocking=True)
            for d, h in zip(st["qx"], self.h_q):
                d.copy_(h, non_blocking=True)
        copied[k % 2].record(cs)

    def e2e_compute(self, k: int, copied, free):
        """On the current stream: step k on device set k % 2, results out."""
        M, torch = self.M, self.torch
        cur, st, b = torch.cuda.current_stream(), self.in_sets[k % 2], k % 2
        cur.wait_event(copied[b])
        M.mp_adamw_step(st["params"], self.hp, self.state, grad_dtype=M.MP_F16, working_dtype=M.MP_BF16)
        M.loss_scale_update(self.state, self.cfg)
        M.fp8_cast_delayed(self.act[b], self.y_act, M.MP_E4M3, self.meta_act, self.hist_act, self.fp8_margin)
        M.fp8_cast_delayed(self.grd[b], self.y_grd, M.MP_E5M2, self.meta_grd, self.hist_grd, self.fp8_margin)
        for q, x in zip(self.q, st["qx"]):
            M.nvfp4_quantize(x, q["codes"], q["scales"], q["ts"], q["nf"], q["ws"], block_2d=q["b2"],
                             stochastic=q["sr"], seed=q["seed"], apply_rht=q["rht"], sign_mask=q["mask"])
        free[b].record(cur)  # the inputs of set b are consumed
        self.h_out_fp8[0].copy_(self.y_act, non_blocking=True)
        self.h_out_fp8[1].copy_(self.y_grd, non_blocking=True)
        for q, (hc, hs) in zip(self.q, self.h_out_q):
            hc.copy_(q["codes"], non_blocking=True)
            hs.copy_(q["scales"], non_blocking=True)
        self.h_small[:88].copy_(self.state, non_blocking=True)
        self.h_small[88:120].copy_(self.meta_act, non_blocking=True)
        self.h_small[120:152].copy_(self.meta_grd, non_blocking=True)
        for i, q in enumerate(self.q):
            self.h_small[152 + 8 * i:156 + 8 * i].copy_(q["ts"].view(torch.uint8), non_blocking=True)
            self.h_small[156 + 8 * i:160 + 8 * i].copy_(q["nf"].view(torch.uint8), non_blocking=True)

    def e2e_run(self, steps: int):
        """steps end-to-end steps: every step's inputs are copied from pinned
        host memory and its results copied back; the copy of step k + 1's
        inputs (copy stream) overlaps step k's kernels (current stream)."""
        torch = self.torch
        cur = torch.cuda.current_stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        for e in free:
            e.record(cur)
        self.copy_stream.wait_stream(cur)
        self.e2e_copy_in(0, copied, free)
        for k in range(steps):
            if k + 1 < steps:
                self.e2e_copy_in(k + 1, copied, free)
            self.e2e_compute(k, copied, free)
        cur.wait_stream(self.copy_stream)


# ---------------------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------------------
class OracleSample:
    """Bounded samples of every part of the workload, run by the oracle as it
    stands (single thread).  A full step's time is projected from the measured
    per-part rates and the full step's algorithmic bytes."""

    def __init__(self, scale: float = 1.0):
        import numpy as np

        import oracle as O
        import synth
        import synth.workloads as W

        self.O, self.np = O, np
        n = int(1_000_000 * scale)
        c = W.FULL
        self.w = synth.fill(c.master_recipe(0), synth.F32, n)
        self.m = np.zeros(n, np.float32)
        self.v = np.zeros(n, np.float32)
        self.g = synth.fill(c.grad_recipe(0, 1), synth.F16, n)
        self.w16 = np.zeros(n, np.uint16)
        self.hp = O.AdamwHp(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay)
        self.st = O.new_scaler_state(c.scale)
        self.cfg = O.ScalerCfg(c.growth, c.backoff, c.interval, 1)
        f = W.FP8
        self.nf8 = int(1_000_000 * scale)
        self.xa = synth.fill(f.act_recipe(0), synth.BF16, self.nf8)
        self.xg = synth.fill(f.grad_recipe(0), synth.BF16, self.nf8)
        self.ma, self.mg = O.new_fp8_meta(), O.new_fp8_meta()
        self.ha, self.hg = np.zeros(f.hist_len, np.float32), np.zeros(f.hist_len, np.float32)
        r, g4 = W.NVFP4_RNE, W.NVFP4_GRAD
        ra = max(16, int(64 * scale) // 16 * 16)
        self.qa = synth.fill(r.act_recipe(), synth.BF16, ra * r.act_cols, shape=(ra, r.act_cols))
        self.qw = synth.fill(r.w_recipe(), synth.BF16, ra * r.w_cols, shape=(ra, r.w_cols))
        rg = max(16, int(32 * scale) // 16 * 16)
        self.qg = synth.fill(g4.recipe(), synth.BF16, rg * g4.cols, shape=(rg, g4.cols))
        self.mask, self.seed = g4.sign_mask(), g4.sr_seed
        self.n = n
        self.t = {"adamw": 0.0, "fp8": 0.0, "nvfp4_act": 0.0, "nvfp4_w": 0.0, "nvfp4_grad": 0.0}
        self.b = {k: 0.0 for k in self.t}

    def run_once(self):
        O, pc = self.O, time.perf_counter
        t0 = pc()
        O.adamw_step(self.hp, self.st, [(self.w, self.m, self.v, self.g, self.w16)], O.F16, O.BF16)
        O.loss_scale_update(self.st, self.cfg)
        t1 = pc()
        O.fp8_cast_delayed(self.xa, O.BF16, O.E4M3, self.ma, self.ha, 1.0)
        O.fp8_cast_delayed(self.xg, O.BF16, O.E5M2, self.mg, self.hg, 1.0)
        t2 = pc()
        O.nvfp4_quantize(self.qa, False, False, 0, False, 0, want_dequant=False)
        t3 = pc()
        O.nvfp4_quantize(self.qw, True, False, 0, False, 0, want_dequant=False)
        t4 = pc()
        O.nvfp4_quantize(self.qg, False, True, self.seed, True, self.mask, want_dequant=False)
        t5 = pc()
        for k, dt, by in (("adamw", t1 - t0, (B_CHECK + B_APPLY) * self.n), ("fp8", t2 - t1, B_FP8 * 2 * self.nf8),
                          ("nvfp4_act", t3 - t2, B_NVFP4_1X16 * self.qa.size),
                          ("nvfp4_w", t4 - t3, B_NVFP4_2D * self.qw.size),
                          ("nvfp4_grad", t5 - t4, B_NVFP4_1X16 * self.qg.size)):
            self.t[k] += dt
            self.b[k] += by
        return t5 - t0

    @staticmethod
    def combined(samples):
        """Per-part rates of concurrent samples add: returns an object whose
        projected() uses the summed rates."""
        class _Sum:
            pass

        out = _Sum()
        out.t = {k: 1.0 for k in samples[0].t}
        out.b = {k: sum(s.b[k] / s.t[k] for s in samples if s.t[k] > 0) for k in samples[0].t}
        out.projected = lambda full: OracleSample.projected(out, full)
        return out

    def sample_bytes(self):
        return sum(self.b.values())

    def projected(self, full_bytes: dict):
        """GB/s of the whole step projected from the per-part rates."""
        part = {"adamw": full_bytes["adamw_check"] + full_bytes["adamw_apply"],
                "fp8": full_bytes["fp8_act_e4m3"] + full_bytes["fp8_grad_e5m2"],
                "nvfp4_act": full_bytes["nvfp4_act_1x16_rne"], "nvfp4_w": full_bytes["nvfp4_w_16x16_rne"],
                "nvfp4_grad": full_bytes["nvfp4_grad_rht_1x16_sr"]}
        secs = sum(part[k] / (self.b[k] / self.t[k]) for k in part)
        return sum(part.values()) / secs / 1e9

    def describe(self):
        return (f"oracle, 1 thread: AdamW {self.n:,} params, FP8 2x{self.nf8:,} elems, NVFP4 "
                f"{self.qa.shape[0]}x{self.qa.shape[1]} 1x16 + {self.qw.shape[0]}x{self.qw.shape[1]} 16x16 + "
                f"{self.qg.shape[0]}x{self.qg.shape[1]} RHT+SR rows of the workload; full-step time projected "
                "from the per-part rates")


def full_step_bytes():
    import synth.workloads as W

    P = sum(n for _, n in W.llama3_8b_params())
    f, r, g = W.FP8, W.NVFP4_RNE, W.NVFP4_GRAD
    return {"adamw_check": B_CHECK * P, "adamw_apply": B_APPLY * P, "loss_scale_update": 0.0,
            "fp8_act_e4m3": B_FP8 * f.rows * f.cols, "fp8_grad_e5m2": B_FP8 * f.rows * f.cols,
            "nvfp4_act_1x16_rne": B_NVFP4_1X16 * r.act_rows * r.act_cols,
            "nvfp4_w_16x16_rne": B_NVFP4_2D * r.w_rows * r.w_cols,
            "nvfp4_grad_rht_1x16_sr": B_NVFP4_1X16 * g.rows * g.cols}


WORKLOAD_NAME = ("llama3-8b fused adamw step (290 tensors, 8,030,257,152 params, fp16 grads x65536, fp32 master/m/v,"
                 " bf16 working copy) + fp8 delayed cast [8192x4096] bf16->e4m3 and ->e5m2 (history 1024) + nvfp4 "
                 "[16384x5120] 1x16 rne + [5120x5120] 16x16 rne + [8192x12288] rht+1x16+sr")


def cpu_all_cores(full_bytes, seconds: float = 8.0):
    """The same oracle on every host core at once: one independent sample per
    thread (the oracle's C calls release the GIL); per-part rates add up."""
    import concurrent.futures as cf

    n = os.cpu_count() or 1
    samples = [OracleSample(scale=0.25) for _ in range(n)]
    for s in samples:
        s.run_once()
        s.t = {k: 0.0 for k in s.t}
        s.b = {k: 0.0 for k in s.b}
    deadline = time.perf_counter() + seconds

    def loop(s):
        while time.perf_counter() < deadline:
            s.run_once()

    with cf.ThreadPoolExecutor(n) as ex:
        list(ex.map(loop, samples))
    total = OracleSample.combined(samples)
    return {"value": round(total.projected(full_bytes), 4), "cores": n,
            "sample": f"{n} threads, each: " + samples[0].describe().replace("oracle, 1 thread: ", "")}


def cpu_baseline(full_bytes):
    """The oracle on every host core (as the reference arm runs it), plus the
    same on one core for context."""
    s = OracleSample(scale=1.0)
    s.run_once()  # warm
    s.t = {k: 0.0 for k in s.t}
    s.b = {k: 0.0 for k in s.b}
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < 8.0:
        s.run_once()
    allc = cpu_all_cores(full_bytes)
    return {"value": allc["value"], "unit": UNIT, "cores": allc["cores"], "kind": "oracle", "sample": allc["sample"],
            "one_core": {"value": round(s.projected(full_bytes), 4), "cores": 1, "sample": s.describe()}}


def run_reference(args):
    """The oracle as it stands, on every host core: one independent bounded
    sample of the workload per thread (its C calls release the GIL), every
    thread running each of the K timed steps; the full step's time is
    projected from the summed per-part rates."""
    import concurrent.futures as cf

    rank, world, _ = dist_env()
    if rank != 0:
        return
    full = full_step_bytes()
    n = os.cpu_count() or 1
    samples = [OracleSample(scale=0.25) for _ in range(n)]

    def run_all(ex):
        list(ex.map(lambda s: s.run_once(), samples))

    with cf.ThreadPoolExecutor(n) as ex:
        for _ in range(args.warmup):
            run_all(ex)
        for s in samples:
            s.t = {k: 0.0 for k in s.t}
            s.b = {k: 0.0 for k in s.b}
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run_all(ex)
        elapsed = time.perf_counter() - t0
    value = OracleSample.combined(samples).projected(full)
    sample = (f"{n} threads, each: " + samples[0].describe().replace("oracle, 1 thread: ", "") +
              f"; {args.steps} timed sample steps in {elapsed:.1f} s")
    # ms_per_step is the wall time of one timed sample step (every thread's
    # bounded sample); the full step's time at the measured rates is reported
    # under its own key.
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed / max(args.steps, 1) * 1e3, 3),
            "sample_bytes_per_step": int(sum(s.sample_bytes() for s in samples) / max(args.steps, 1)),
            "projected_ms_per_full_step": round(sum(full.values()) / (value * 1e9) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "arm": f"CPU oracle (scalar C, -O2) on {n} host threads"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world)
    import mixed_precision_numerics_gb300 as M

    wl = Workload(args.small)
    stream = torch.cuda.current_stream()

    for k in range(args.warmup):
        wl.step(k)
    torch.cuda.synchronize()

    ncalls = len(wl.calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ncalls + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(gpu_id_for_smi(local))
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    launches0 = M.mp_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    trace = wl.trace_buffers(args.steps) if args.trace else None
    t_start.record(stream)
    for k in range(args.steps):
        wl.step(args.warmup + k, evs[k])
        if trace is not None:
            wl.trace_copy(trace, k)
    t_stop.record(stream)
    torch.cuda.synchronize()
    launches = M.mp_launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()
    value, elapsed_ms = job_gbs(args.steps * wl.step_bytes, t_start.elapsed_time(t_stop), world)

    per_call_ms = {name: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps))
                   for i, name in enumerate(wl.calls)}
    if trace is not None and rank == 0:
        with open(args.trace, "w") as fh:
            for k in range(args.steps):
                rec = wl.trace_record(trace, k)
                rec["step"] = args.warmup + k
                rec["ms"] = {name: round(evs[k][i].elapsed_time(evs[k][i + 1]), 4) for i, name in enumerate(wl.calls)}
                fh.write(json.dumps(rec) + "\n")
    peak, peak_kind = hbm_peak()
    kernels = {}
    for name in wl.calls:
        ms = per_call_ms[name]
        gbs = wl.bytes[name] / (ms * 1e-3) / 1e9 if wl.bytes[name] else None
        kernels[name] = {"ms": round(ms, 4), "bytes": int(wl.bytes[name]),
                         "elems_per_s": float(f"{wl.units[name] / (ms * 1e-3):.4g}") if wl.units[name] else None,
                         "gbs": round(gbs, 1) if gbs else None,
                         "frac_of_" + peak_kind + "_hbm": round(gbs / peak, 4) if gbs else None}
    ms_per_step = elapsed_ms / args.steps
    if "nvfp4_grad_rht_1x16_sr" in kernels:
        kernels["nvfp4_grad_rht_1x16_sr"]["bound"] = "issue"
        kernels["nvfp4_grad_rht_1x16_sr"]["note"] = (
            "the encode pass runs about 17.2 instructions per element (Philox4x32-10 at one call per 8 elements, "
            "whose wide multiplies hold the FMA-heavy pipe, the Hadamard butterfly, stochastic rounding by the "
            "hardware conversion two elements at a time); ncu shows issue slots 65 % busy, the FMA-heavy and "
            "integer pipes 64 % and 58 % busy and DRAM about 35 %, so its HBM fraction is not its limit")
    if "fp8_act_e4m3" in kernels:
        kernels["fp8_act_e4m3"]["note"] = ("runs right after the update kernel and pays for the dirty L2 lines "
                                           "that kernel leaves; graph_isolated_* is the same call alone")

    apply_ms = per_call_ms["adamw_apply"]
    achieved = wl.bytes["adamw_apply"] / (apply_ms * 1e-3) / 1e9
    tr = profiled_traffic(wl.P)
    roofline = {"bound": "hbm", "kernel": "k_adamw_update (mp_adamw_apply, 28 B/param)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "traffic": round(tr[0] + tr[1]) if tr else None}
    if tr:
        roofline["traffic_read"] = round(tr[0])
        roofline["traffic_write"] = round(tr[1])
        roofline["traffic_note"] = (f"from {os.path.relpath(TRAFFIC_RECORD, ROOT)}: reads scaled by params "
                                    f"(the capture read {B_APPLY / 2:.0f} B/param); writes {B_APPLY / 2:.0f} B/param "
                                    f"less {tr[2] / 1e6:.1f} MB left dirty in L2 at kernel end (not scaled)")

    # Each quantiser call alone: 16 back-to-back calls captured in a CUDA
    # graph and replayed after an L2-clean point, so neither launch gaps nor
    # the previous kernel's dirty L2 lines are charged to it.
    isolated = wl.isolated_call_times(reps=2 if args.small else 16)
    for name, us in isolated.items():
        if name not in kernels:  # calls measured only in isolation
            wl.bytes[name] = wl.extra_bytes[name]
            kernels[name] = {"bytes": int(wl.bytes[name]), "note": "not in the step; graph-replayed only"}
        gbs = wl.bytes[name] / (us * 1e-6) / 1e9
        kernels[name]["graph_isolated_us"] = round(us, 2)
        kernels[name]["graph_isolated_elems_per_s"] = float(f"{wl.units[name] / (us * 1e-6):.4g}")
        kernels[name]["graph_isolated_gbs"] = round(gbs, 1)
        kernels[name]["graph_isolated_frac_of_" + peak_kind + "_hbm"] = round(gbs / peak, 4)

    clip_ms = wl.clipped_check_ms()
    gbs = wl.bytes["adamw_check"] / (clip_ms * 1e-3) / 1e9
    kernels["adamw_check_with_clipping"] = {"ms": round(clip_ms, 4), "bytes": int(wl.bytes["adamw_check"]),
                                            "gbs": round(gbs, 1), "frac_of_" + peak_kind + "_hbm": round(gbs / peak, 4),
                                            "note": "not in the step: max_grad_norm 1.0, timed after it"}

    e2e = None
    if not args.no_e2e:
        try:
            wl.e2e_setup()
            wl.e2e_run(2)
            torch.cuda.synchronize()
            barrier(world)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            wl.e2e_run(args.steps)
            b.record(stream)
            torch.cuda.synchronize()
            e_gbs, e_ms = job_gbs(args.steps * wl.step_bytes, a.elapsed_time(b), world)
            link = wl.h2d_link_gbs()
            copy_ms = wl.e2e_copy_only_ms()
            e2e = {"value": round(e_gbs, 1), "unit": UNIT, "ms_per_step": round(e_ms / args.steps, 3),
                   "h2d_bytes_per_step": int(wl.h2d), "d2h_bytes_per_step": int(wl.d2h),
                   "h2d_link_gbs": round(link, 1),
                   "h2d_ms_per_step_at_link_speed": round(wl.h2d / (link * 1e9) * 1e3, 2),
                   "h2d_ms_per_step_measured": round(copy_ms, 2),
                   "api": "mp_adamw_step + loss_scale_update + fp8_cast_delayed x2 + nvfp4_quantize x3 "
                          "with pinned host inputs copied in and outputs copied out every step; step k+1's "
                          "inputs are copied (second stream, second device input set) while step k runs"}
        except Exception as ex:  # host memory for the pinned buffers may be missing
            e2e = {"value": None, "unit": UNIT, "error": f"{type(ex).__name__}: {ex}"[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.small:
        cpu = cpu_baseline(wl.bytes)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": WORKLOAD_NAME + (" [small: decoder layer 0 only]" if args.small else ""),
                           "params": wl.P, "bytes_per_step": int(wl.step_bytes),
                           "l2": "inputs larger than L2: every step streams >=241 GB (>> 129 MB L2) and the FP8 "
                                 "inputs rotate over 64 buffers, so no buffer is L2-resident when reused",
                           "parallelism": f"replicas x{world} (no data-path collective)"},
                "roofline": roofline, "kernels": kernels, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
                "gpu_launches": int(launches)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
