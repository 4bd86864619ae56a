"""Pins for the oracle's NVFP4 quantiser, Hadamard transform, stochastic
rounding and Philox generator (CPU).

* The transform matrix equals scipy's Sylvester Hadamard / 4, is orthogonal,
  and maps signed one-hot inputs to signed columns in closed form.
* Block scales and element codes of small tensors (64 elements in 1x16
  blocks, one 16x16 tile) are re-derived by brute-force searches over every
  E4M3 scale code and every E2M1 code.
* Stochastic rounding is unbiased over 10^6 draws.
* Philox4x32-10 matches an independent library implementation.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import scipy.linalg
import torch

from tests.conftest import golden

import oracle as O

GRID = np.array(golden("nvfp4_format.json")["e2m1_magnitudes"])
E4M3_TABLE = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()


def bf16(x):
    return O.convert(np.asarray(x, np.float32), O.F32, O.BF16)


def f32_of_bf16(b):
    return O.convert(b, O.BF16, O.F32)


# ---- Hadamard ---------------------------------------------------------------


def transform_matrix(mask):
    cols = [O.rht16_tile(np.eye(16, dtype=np.float32)[j], mask) for j in range(16)]
    return np.stack(cols, axis=1).astype(np.float64)  # column j = T e_j


def test_hadamard_is_sylvester_over_four():
    T = transform_matrix(0)
    H = scipy.linalg.hadamard(16)
    np.testing.assert_array_equal(T * 4, H)
    np.testing.assert_array_equal(H @ H.T, 16 * np.eye(16))
    np.testing.assert_allclose(T @ T.T, np.eye(16), atol=0)


@pytest.mark.parametrize("mask", [0x0001, 0x8000, 0xA5C3, 0xFFFF])
def test_signed_one_hot_closed_form(mask):
    H = scipy.linalg.hadamard(16)
    for j in range(16):
        s = -1.0 if (mask >> j) & 1 else 1.0
        for a in (1.0, -3.5, 2.0**-20):
            e = np.zeros(16, np.float32)
            e[j] = a
            np.testing.assert_array_equal(O.rht16_tile(e, mask), (a * s / 4) * H[:, j])


def test_transform_is_orthogonal_on_random_rows():
    rng = np.random.default_rng(0)
    x = bf16(rng.standard_normal((64, 16 * 8)).astype(np.float32))
    mask = 0x3C5A
    y = O.rht16(x, mask).astype(np.float64)
    xf = f32_of_bf16(x).astype(np.float64)
    np.testing.assert_allclose(np.linalg.norm(y.reshape(-1, 16), axis=1),
                               np.linalg.norm(xf.reshape(-1, 16), axis=1), rtol=1e-6)
    T = transform_matrix(mask)
    back = (y.reshape(-1, 16) @ T)  # T^T applied per tile: rows are y^T
    np.testing.assert_allclose(back.reshape(xf.shape), xf, rtol=0, atol=1e-6)
    yb = O.rht16(x, mask, O.BF16)
    np.testing.assert_array_equal(yb, torch.from_numpy(y.astype(np.float32)).bfloat16()
                                  .view(torch.int16).numpy().view(np.uint16))


# ---- brute-force block scales and codes ------------------------------------------


def nearest_e4m3_code(q):
    pos = np.arange(127)  # 0x00 .. 0x7E, all non-negative finite codes
    vals = E4M3_TABLE[pos].astype(np.float64)
    if q > vals.max():
        return 0x7E
    d = np.abs(vals - q)
    cand = pos[d == d.min()]
    if cand.size > 1:
        cand = cand[(cand & 1) == 0]
    return int(cand[0])


def nearest_e2m1_code(y):
    a = abs(float(y))
    if a > 6.0:
        c = 7
    else:
        d = np.abs(GRID - a)
        cand = np.arange(8)[d == d.min()]
        if cand.size > 1:
            cand = cand[(cand & 1) == 0]
        c = int(cand[0])
    return c | (8 if np.signbit(y) else 0)


def brute_force_blocks(xp, blocks, s_t):
    """blocks: list of index arrays into xp (flat); returns dict of expected
    per-block scale code and per-element code and dequant bits."""
    codes = {}
    scales = []
    deq = {}
    for idx in blocks:
        vals = xp.ravel()[idx]
        bamax = np.float32(np.abs(vals).max())
        q = np.float32(np.float32(bamax / np.float32(6.0)) / np.float32(s_t))
        sc = nearest_e4m3_code(float(q))
        scales.append(sc)
        d = np.float32(np.float32(E4M3_TABLE[sc]) * np.float32(s_t))
        r = np.float32(0.0) if d == 0 else np.float32(np.float32(1.0) / d)
        for i, v in zip(idx, vals):
            c = nearest_e2m1_code(np.float32(v * r))
            codes[int(i)] = c
            val = (-1 if c & 8 else 1) * GRID[c & 7]
            deq[int(i)] = int(torch.tensor([np.float32(val) * d]).bfloat16().view(torch.int16).item()) & 0xFFFF
    return codes, scales, deq


def unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def make_64():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(16) * 2.0,          # ordinary block
        rng.standard_normal(16) * 1e-3,         # small block
        np.r_[rng.standard_normal(15) * 0.1, 40.0],  # one outlier
        np.zeros(16),                            # all-zero block
    ]).astype(np.float32)
    return bf16(x).reshape(1, 64)


@pytest.mark.parametrize("rht", [False, True])
def test_64_elements_1x16_brute_force(rht):
    x = make_64()
    mask = 0x9B17
    codes, scales, ts, nf, dq = O.nvfp4_quantize(x, block_2d=False, stochastic=False, apply_rht=rht,
                                                  sign_mask=mask)
    xp = O.rht16(x, mask) if rht else f32_of_bf16(x)
    assert nf == 0
    assert ts == np.float32(np.abs(xp).max()) / np.float32(2688.0)
    blocks = [np.arange(16 * b, 16 * b + 16) for b in range(4)]
    ec, es, ed = brute_force_blocks(xp, blocks, ts)
    np.testing.assert_array_equal(scales.ravel(), es)
    got = unpack(codes).ravel()
    np.testing.assert_array_equal(got, [ec[i] for i in range(64)])
    np.testing.assert_array_equal(dq.ravel(), [ed[i] for i in range(64)])
    if not rht:
        assert scales.ravel()[3] == 0 and (got[48:] == 0).all()  # zero block


def test_16x16_tile_brute_force():
    rng = np.random.default_rng(5)
    x = bf16((rng.standard_normal((16, 32)) * 0.02).astype(np.float32))
    x[7, 20] = bf16([0.9])[0]  # one large value in the second tile
    codes, scales, ts, nf, dq = O.nvfp4_quantize(x, block_2d=True, stochastic=False)
    xp = f32_of_bf16(x)
    assert scales.shape == (1, 2)
    blocks = []
    for b in range(2):
        rr, cc = np.meshgrid(np.arange(16), np.arange(16 * b, 16 * b + 16), indexing="ij")
        blocks.append((rr * 32 + cc).ravel())
    ec, es, ed = brute_force_blocks(xp, blocks, ts)
    np.testing.assert_array_equal(scales.ravel(), es)
    got = unpack(codes).ravel()
    np.testing.assert_array_equal(got, [ec[i] for i in range(512)])
    np.testing.assert_array_equal(dq.ravel(), [ed[i] for i in range(512)])


def test_rne_dequant_error_is_within_half_a_gap():
    rng = np.random.default_rng(11)
    x = bf16(rng.standard_normal((32, 256)).astype(np.float32))
    codes, scales, ts, nf, dq = O.nvfp4_quantize(x, block_2d=False, stochastic=False)
    xf = f32_of_bf16(x).reshape(-1, 16).astype(np.float64)
    q = unpack(codes).reshape(-1, 16)
    d = E4M3_TABLE[scales.ravel()].astype(np.float64) * ts
    val = np.where(q & 8, -1, 1) * GRID[q & 7] * d[:, None]
    y = np.abs(xf) / d[:, None]
    gap = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0)) * d[:, None]
    unsat = y <= 6
    assert (np.abs(val - xf)[unsat] <= gap[unsat] / 2 * (1 + 1e-6)).all()


def test_nonfinite_and_zero_tensors():
    x = bf16(np.ones((2, 32), np.float32))
    x[1, 5] = 0x7F80  # +inf
    codes, scales, ts, nf, dq = O.nvfp4_quantize(x, block_2d=False, stochastic=False)
    assert nf == 1 and np.isinf(ts)
    assert not codes.any() and not scales.any() and not dq.any()
    z = np.zeros((16, 16), np.uint16)
    z[3, 3] = 0x8000  # -0.0
    codes, scales, ts, nf, dq = O.nvfp4_quantize(z, block_2d=True, stochastic=True, seed=9)
    assert nf == 0 and ts == 0.0 and not codes.any() and not scales.any()


def test_shape_errors():
    with pytest.raises(ValueError):
        O.nvfp4_quantize(np.zeros((2, 24), np.uint16), block_2d=False, stochastic=False)
    with pytest.raises(ValueError):
        O.nvfp4_quantize(np.zeros((8, 32), np.uint16), block_2d=True, stochastic=False)


# ---- stochastic rounding ---------------------------------------------------------


@pytest.mark.parametrize("y,lo,hi", [(2.3, 2.0, 3.0), (0.1, 0.0, 0.5), (-1.2, 1.0, 1.5), (5.0, 4.0, 6.0)])
def test_sr_is_unbiased_over_1e6_draws(y, lo, hi):
    n = 1_000_000
    yv = np.full(n, y, np.float32)
    c = O.e2m1_sr_array(yv, seed=1234, i0=0)
    vals = np.where(c & 8, -1.0, 1.0) * GRID[c & 7]
    a = abs(float(np.float32(y)))
    p = (a - lo) / (hi - lo)
    assert set(np.unique(GRID[c & 7])) <= {lo, hi}
    phat = np.mean(GRID[c & 7] == hi)
    sigma_p = np.sqrt(p * (1 - p) / n)
    assert abs(phat - p) < 4 * sigma_p
    sigma = (hi - lo) * np.sqrt(p * (1 - p))
    assert abs(vals.mean() - float(np.float32(y))) < 4 * sigma / np.sqrt(n)


def test_sr_fixed_points_and_saturation():
    pts = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 7.5, -0.0, -4.0], np.float32)
    for seed in (0, 1, 99):
        c = O.e2m1_sr_array(np.repeat(pts, 50), seed=seed)
        expect = np.repeat([0, 1, 2, 3, 4, 5, 6, 7, 7, 8, 14], 50)
        np.testing.assert_array_equal(c, expect)


def test_sr_threshold_rule():
    L = O.lib()
    # 2.25 sits a quarter of the way from 2 to 3: it rounds up iff r16 >= 3/4 * 2^16
    assert L.orc_f32_to_e2m1_sr(2.25, 49151) == 4
    assert L.orc_f32_to_e2m1_sr(2.25, 49152) == 5
    # 0.125 is a quarter of the way from 0 to 0.5; the sign is applied after
    assert L.orc_f32_to_e2m1_sr(-0.125, 49151) == 8 | 0
    assert L.orc_f32_to_e2m1_sr(-0.125, 49152) == 8 | 1


# ---- Philox -------------------------------------------------------------------------

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def k(out, seed, c0p, c1p, c2p, c3p, N: tl.constexpr):
    o = tl.arange(0, N)
    c0 = tl.load(c0p + o); c1 = tl.load(c1p + o); c2 = tl.load(c2p + o); c3 = tl.load(c3p + o)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out + o * 4 + 0, a); tl.store(out + o * 4 + 1, b)
    tl.store(out + o * 4 + 2, c); tl.store(out + o * 4 + 3, d)

cases = json.loads(sys.stdin.read())
res = []
for seed, ctrs in cases:
    n = len(ctrs)
    cols = [torch.tensor([c[i] for c in ctrs], dtype=torch.int64).to(torch.uint32) for i in range(4)]
    out = torch.zeros(n * 4, dtype=torch.uint32)
    k[(1,)](out, seed, *cols, N=n)
    res.append(out.to(torch.int64).tolist())
print(json.dumps(res))
"""


def test_philox_matches_triton_reference():
    pytest.importorskip("triton")
    rng = np.random.default_rng(17)
    cases = []
    for seed in (0, 1234, 0xDEADBEEFCAFEF00D, 2**63 + 5):
        ctrs = [[0, 0, 0, 0], [1, 0, 0, 0], [0, 0, 0, 1], [0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF]]
        ctrs += rng.integers(0, 2**32, size=(12, 4), dtype=np.uint64).tolist()
        cases.append([seed, ctrs])
    env = dict(os.environ, TRITON_INTERPRET="1")
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(cases), capture_output=True,
                       text=True, env=env, timeout=300)
    if p.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + p.stderr.strip().splitlines()[-1][:200])
    ref = json.loads(p.stdout.strip().splitlines()[-1])
    for (seed, ctrs), r in zip(cases, ref):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i, c in enumerate(ctrs):
            np.testing.assert_array_equal(O.philox(c, key), np.array(r[4 * i:4 * i + 4], np.uint32))


def test_sr_bits_layout_and_uniformity():
    seed = 1234
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in (0, 1, 7, 8, 13, 2**33 + 5):
        w = O.philox([(i >> 3) & 0xFFFFFFFF, i >> 35, 0, 0], key)
        assert O.lib().orc_sr_bits(seed, i) == (int(w[(i >> 1) & 3]) >> (16 * (i & 1))) & 0xFFFF
    bits = O.sr_bits(seed, np.arange(1 << 16))
    counts = np.bincount(bits >> 12, minlength=16)
    chi2 = ((counts - 4096.0) ** 2 / 4096.0).sum()
    assert chi2 < 50  # 15 dof; p ~ 1e-5
