"""Pins of the oracle's NVFP4 training options ("Why FP8 training is stable" (magicnetworld.com),
sec 13; "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 3.2): the 16-point random
Hadamard transform, stochastic rounding of the E2M1 codes with one random byte per element, and
16x16 2-D weight blocks.

Pins: the transform against scipy's Hadamard matrix (a library routine) and its exact algebra on
integer inputs (orthogonality, involution, sign mask, preserved products); stochastic rounding's
support (only the two neighbours), its expectation (the page's E[Q(x) - x] = 0, exact when the
distance is a multiple of 1/256 of the step) and its probabilities; the composed quantizer
against the pinned NVFP4 recipe applied to the transformed values; 2-D block scales as the
maximum of the (pinned) 1x16 scales of their rows.
"""
import math

import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle as orc
from oracle import E2M1

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_transform_is_the_scaled_hadamard_matrix(golden):
    n = int(golden("nvfp4_training.txt")["rht_size"])
    H = hadamard(n).astype(np.float64) / 4.0
    rng = np.random.default_rng(1)
    for _ in range(20):
        v = rng.standard_normal(n).astype(np.float32)
        signs = int(rng.integers(0, 1 << 16))
        d = np.array([-1.0 if (signs >> i) & 1 else 1.0 for i in range(n)])
        ref = H @ (d * v.astype(np.float64))
        got = orc.fwht16(v, signs).astype(np.float64)
        assert np.allclose(got, ref, rtol=0, atol=16 * np.abs(v).max() * 2.0 ** -23)
    # small integers: every sum is exact, so the FP32 result equals the matrix product exactly
    vi = rng.integers(-8, 9, n).astype(np.float32)
    assert np.array_equal(orc.fwht16(vi, 0).astype(np.float64), H @ vi.astype(np.float64))


def test_transform_algebra_on_exact_inputs():
    rng = np.random.default_rng(2)
    v = rng.integers(-16, 17, 16).astype(np.float32)
    w = rng.integers(-16, 17, 16).astype(np.float32)
    t = orc.fwht16(v)
    assert np.array_equal(orc.fwht16(t), v)                       # 0.25 H16 is its own inverse
    assert float(np.dot(t, orc.fwht16(w))) == float(np.dot(v, w))  # products are preserved
    assert float(np.dot(t, t)) == float(np.dot(v, v))
    m = 0b1010000000000101
    vneg = v.copy()
    for i in range(16):
        if (m >> i) & 1:
            vneg[i] = -vneg[i]
    assert np.array_equal(orc.fwht16(v, m), orc.fwht16(vneg, 0))


@pytest.mark.parametrize("a", [0.1, 0.3, 0.5, 0.75, 1.2, 1.74, 2.5, 3.9, 5.0, 5.99])
def test_stochastic_rounding_support_and_expectation(golden, a):
    assert float(golden("nvfp4_training.txt")["sr_expected_error"]) == 0.0
    lo = max(g for g in GRID if g <= a)
    hi = min(g for g in GRID if g > a)
    vals = [orc.decode(E2M1, orc.e2m1_stochastic(a, r)) for r in range(256)]
    assert set(vals) <= {lo, hi}
    mean = sum(vals) / 256.0
    step = hi - lo
    assert -step / 256.0 < mean - a <= 0.0
    ups = sum(v == hi for v in vals)
    assert ups == math.floor(256 * (a - lo) / step)
    # negative inputs mirror
    assert [orc.e2m1_stochastic(-a, r) for r in range(256)] == [c | 0x8 for c in
                                                               (orc.e2m1_stochastic(a, r) for r in range(256))]


def test_stochastic_rounding_is_unbiased_on_the_fine_grid():
    # E[Q(x) - x] = 0 exactly whenever 256 (x - lo) / step is an integer
    for lo, hi in zip(GRID[:-1], GRID[1:]):
        for k in (1, 37, 128, 255):
            x = lo + (hi - lo) * k / 256.0
            mean = sum(orc.decode(E2M1, orc.e2m1_stochastic(x, r)) for r in range(256)) / 256.0
            assert mean == x
    assert orc.e2m1_stochastic(6.0, 0) == 7 and orc.e2m1_stochastic(7.5, 255) == 7 and orc.e2m1_stochastic(4.0, 0) == 6
    assert orc.e2m1_stochastic(-0.0, 0) == 0x8


def test_transformed_quantizer_follows_the_recipe():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(64, 128, generator=g) * 3).to(torch.bfloat16)
    signs = 0x5A3C
    q, s, sg = orc.nv_quantize_ex(bits(x), rht=True, signs=signs)
    xs = x.float().numpy()
    v = np.stack([orc.fwht16(xs[r, 16 * b:16 * b + 16], signs) for r in range(64) for b in range(8)])
    assert np.float32(sg) == np.float32(orc.nv_global_scale(float(np.abs(v).max())))
    for idx in range(0, v.shape[0], 5):
        r, b = divmod(idx, 8)
        code, sh = orc.nv_block_scale(sg, float(np.abs(v[idx]).max()))
        assert s[r, b] == code
        assert [int(c) for c in q[r, 16 * b:16 * b + 16]] == [orc.nv_encode(float(e), sh) for e in v[idx]]


def test_quantizer_without_options_equals_plain_nvfp4():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(32, 64, generator=g) * 2).to(torch.bfloat16)
    q, s, sg = orc.nv_quantize_ex(bits(x))
    qp, sp, sgp = orc.nv_quantize(bits(x))
    assert sg == sgp and np.array_equal(s, sp)
    assert np.array_equal(q[:, 0::2] | (q[:, 1::2] << 4), qp)


def test_stochastic_quantizer_picks_neighbours_of_the_quotient():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(32, 64, generator=g)).to(torch.bfloat16)
    rb = np.random.default_rng(6).integers(0, 256, (32, 64), dtype=np.uint8)
    q, s, sg = orc.nv_quantize_ex(bits(x), rbits=rb)
    qn, sn, _ = orc.nv_quantize_ex(bits(x))
    assert np.array_equal(s, sn)
    xs = x.float().numpy()
    for r in range(0, 32, 3):
        for c in range(0, 64, 5):
            _, sh = orc.nv_block_scale(sg, float(np.abs(xs[r, 16 * (c // 16):16 * (c // 16) + 16]).max()))
            y = float(np.float32(xs[r, c]) / np.float32(sh))
            assert orc.decode(E2M1, int(q[r, c])) in {math.copysign(v, y) for v in GRID
                                                      if abs(abs(y) - v) <= 2.0 or abs(y) >= 6}
            assert q[r, c] == orc.e2m1_stochastic(np.float32(y), int(rb[r, c]))


def test_2d16_scale_is_max_of_row_block_scales(golden):
    n = int(golden("nvfp4_training.txt")["weight_block_2d"])
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(64, 96, generator=g) * torch.logspace(-2, 2, 96)).to(torch.bfloat16)
    q, s, sg = orc.nv_quantize_2d16(bits(x))
    _, s1, sg1 = orc.nv_quantize(bits(x))                     # 1x16 scales, pinned elsewhere
    assert sg == sg1 and s.shape == (64 // n, 96 // n)
    for br in range(64 // n):
        for bc in range(96 // n):
            assert s[br, bc] == s1[n * br:n * br + n, bc].max()
    xs = x.float().numpy()
    for r in range(0, 64, 7):
        for c in range(0, 96, 5):
            _, sh = orc.nv_block_scale(sg, float(np.abs(xs[16 * (r // 16):16 * (r // 16) + 16,
                                                           16 * (c // 16):16 * (c // 16) + 16]).max()))
            assert q[r, c] == orc.nv_encode(float(xs[r, c]), sh)
