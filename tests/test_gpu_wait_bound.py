"""The pipelines' waits are bounded: a wait on a barrier phase that nothing
completes gives up after its poll limit and says so, and the context stays
usable.  The probe kernel (tests/wait_probe.cu) uses the library's own wait
routine; it is built here with nvcc for sm_103a."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import mixed_precision_numerics_gb300 as M

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe(tmp_path_factory, cuda_ok):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = tmp_path_factory.mktemp("probe") / "libwaitprobe.so"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                        "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "mixed_precision_numerics_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "wait_probe.cu"), "-o", str(out)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    L = ctypes.CDLL(str(out))
    L.wait_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.wait_probe.restype = ctypes.c_int
    return L


def run_probe(L, arrive):
    ok = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert L.wait_probe(arrive, ok.data_ptr(), ns.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    return int(ok.item()), int(ns.item())


def test_completed_phase_is_seen_at_once(probe):
    ok, ns = run_probe(probe, 1)
    assert ok == 1
    assert ns < 10_000_000  # well under the limit


def test_wait_that_nothing_completes_gives_up_and_the_context_survives(probe):
    ok, ns = run_probe(probe, 0)
    assert ok == 0
    assert 1_000_000 <= ns <= 20_000_000_000  # the poll limit, not forever
    # the context still runs library work correctly afterwards
    x = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(4096, dtype=torch.uint8, device="cuda")
    meta, hist = M.new_fp8_meta(), torch.zeros(4, device="cuda")
    M.fp8_cast_delayed(x, y, M.MP_E4M3, meta, hist)
    torch.cuda.synchronize()
    assert np.all(y.cpu().numpy() == 0x38)  # 1.0 in E4M3
    assert M.mp_wait_failures() == 0  # the probe is not one of the library's kernels
