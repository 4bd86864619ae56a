"""nvfp4_quantize_noalloc, the entry point for callers that cannot allocate.

Some callers cannot allocate device memory where they call the quantiser (a
framework step whose memory pool must not grow, a plugin that is handed only
its inputs and outputs, host code that must not synchronise the device
through cudaMalloc).  This test calls the workspace-free entry point through
the C ABI twice in a row and checks that both calls give exactly what the
workspace entry point gives on the same inputs.  The file sorts last so that
a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import mixed_precision_numerics_gb300 as M

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def call_noalloc(x, rows, cols, block_2d, stochastic, rht, got):
    return M.lib.nvfp4_quantize_noalloc(
        ctypes.c_void_p(x.data_ptr()), rows, cols, int(block_2d), int(stochastic), 1234, int(rht), 0xE3BF,
        ctypes.c_void_p(got[0].data_ptr()), ctypes.c_void_p(got[1].data_ptr()),
        ctypes.c_void_p(got[2].data_ptr()), ctypes.c_void_p(got[3].data_ptr()),
        ctypes.c_void_p(got[4].data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def outputs(rows, cols, block_2d):
    return (torch.full((rows, cols // 2), 0xAA, dtype=torch.uint8, device="cuda"),
            torch.full((rows // 16 if block_2d else rows, cols // 16), 0xAA, dtype=torch.uint8, device="cuda"),
            torch.full((1,), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((rows, cols), 0x5555, dtype=torch.int16, device="cuda"))


@pytest.mark.parametrize("block_2d,stochastic,rht", [(False, True, True), (True, False, False)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(block_2d, stochastic, rht):
    assert M.lib.nvfp4_noalloc_scratch_bytes() >= M.nvfp4_workspace_size()
    rows, cols = 256, 1040
    ws = M.new_nvfp4_workspace()
    for call in range(2):
        r = synth.recipe(70 + call, call, 1.0 + call, 0.01, 30.0, synth.OUT_SCALE)
        x = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
        synth.fill_device(r, synth.BF16, x)
        ref = outputs(rows, cols, block_2d)
        got = outputs(rows, cols, block_2d)
        M.nvfp4_quantize(x, *ref[:4], ws, block_2d=block_2d, stochastic=stochastic, seed=1234, apply_rht=rht,
                         sign_mask=0xE3BF, dequant=ref[4])
        st = call_noalloc(x, rows, cols, block_2d, stochastic, rht, got)
        assert st == M.MP_OK, M.mp_status_str(st)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b), f"call {call}: outputs differ from the workspace entry point"
        assert int(got[3].item()) == 0 and float(got[2].item()) > 0.0


def test_noalloc_rejects_a_bad_shape_before_enqueueing_anything():
    """A shape the quantiser does not take (cols not a multiple of 16, or rows
    not a multiple of 16 for 16x16 blocks) returns MP_ESHAPE with no kernel
    launched, and the next call on the stream still gives the workspace entry
    point's results."""
    rows, cols = 64, 512
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    synth.fill_device(synth.recipe(75, 0, 1.0), synth.BF16, x)
    bad = outputs(rows, cols, True)
    before = M.mp_launch_count()
    assert call_noalloc(x, rows, cols - 8, False, False, False, bad) == M.MP_ESHAPE
    assert call_noalloc(x, rows - 8, cols, True, False, False, bad) == M.MP_ESHAPE
    assert M.mp_launch_count() == before
    torch.cuda.synchronize()
    for t, fill in zip(bad, (0xAA, 0xAA, -1.0, -1, 0x5555)):
        assert bool((t == fill).all().item()), "a rejected call wrote an output"
    got, ref = outputs(rows, cols, True), outputs(rows, cols, True)
    assert call_noalloc(x, rows, cols, True, False, False, got) == M.MP_OK
    M.nvfp4_quantize(x, *ref[:4], M.new_nvfp4_workspace(), block_2d=True, sign_mask=0xE3BF, seed=1234,
                     dequant=ref[4])
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
