"""Pins of the oracle's Float8BlockScaling-to-MX path ("MXFP8 on SM120: software support"
(xuesongtap.github.io), sec 1.3): power-of-two FP32 block scales (1x128 tiles, 128x128 blocks),
their conversion to per-32 E8M0 scales reusing the FP8 codes, and 2-D 32x32 MX weight blocks.

Pins: the page's structure (tests/golden/float8_block_to_mx.txt), the DeepSeek tile's printed
scale (the power-of-two scale is the next power of two above it), minimality and no-saturation
of the scale rule, a brute-force nearest-code scan, exact equality of the dequantized values
before and after conversion, the product on converted scales against the block-scaled product,
and the 2-D block scale as the maximum of the (already pinned) 1x32 scales of its rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from oracle import E4M3, E5M2, E8M0


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def tile(rows, cols, seed, spread=4.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * torch.logspace(-spread, spread, cols)).to(torch.bfloat16)


def test_pow2_scale_against_printed_deepseek_scale(golden):
    g = golden("deepseek_tile_example.txt")
    s_page = float(g["scale"])                      # amax / 448 printed on the page
    amax = s_page * 448.0
    k = orc.pow2_scale_exp(amax)
    assert 1.0 <= 2.0 ** k / s_page < 2.0           # the next power of two at or above amax / 448
    assert k == -5


@pytest.mark.parametrize("amax", [448.0, 450.0, 224.0, 12.5, 1.0, 2.0 ** -100, 3.0e38, 2.0 ** -135])
def test_pow2_scale_is_minimal_and_never_saturates(amax):
    k = orc.pow2_scale_exp(amax)
    if -127 < k < 127:
        assert 448.0 * 2.0 ** k >= amax and 448.0 * 2.0 ** (k - 1) < amax
    assert -127 <= k <= 127
    assert orc.pow2_scale_exp(0.0) == 0


@pytest.mark.parametrize("which", ["1x128", "128x128"])
def test_pow2_quantize_matches_bruteforce(which):
    x = tile(128, 256, 3 if which == "1x128" else 4)
    q, s = (orc.ds_quantize_1x128_pow2 if which == "1x128" else orc.ds_quantize_128x128_pow2)(bits(x))
    xs = x.float().numpy().astype(np.float64)
    for r in range(0, 128, 7):
        for c in range(0, 256, 5):
            sc = float(s[r, c // 128]) if which == "1x128" else float(s[r // 128, c // 128])
            assert math.frexp(sc)[0] == 0.5                         # a power of two
            assert int(q[r, c]) == orc.encode_bruteforce(E4M3, xs[r, c] / sc)
    # nothing saturates: every block's amax / s lies in (224, 448]
    if which == "1x128":
        for r in range(128):
            for b in range(2):
                assert 224.0 < np.abs(xs[r, 128 * b:128 * b + 128]).max() / float(s[r, b]) <= 448.0
    else:
        for b in range(2):
            assert 224.0 < np.abs(xs[:, 128 * b:128 * b + 128]).max() / float(s[0, b]) <= 448.0


@pytest.mark.parametrize("block_rows", [1, 128])
def test_conversion_keeps_every_dequantized_value(golden, block_rows):
    g = golden("float8_block_to_mx.txt")
    assert int(g["block_1d"]) == int(g["sub_blocks"]) * int(g["mx_block"])
    x = tile(256, 384, 10 + block_rows)
    if block_rows == 1:
        q, s = orc.ds_quantize_1x128_pow2(bits(x))
        s_elem = np.repeat(s, 128, axis=1)
    else:
        q, s = orc.ds_quantize_128x128_pow2(bits(x))
        s_elem = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    e8 = orc.mx_scales_from_blocks(s, 256, 384, block_rows)
    assert e8.shape == (256, 384 // 32)
    dec = np.vectorize(lambda c: orc.decode(E4M3, int(c)))(q)
    mx_scale = np.repeat(np.vectorize(lambda c: orc.decode(E8M0, int(c)))(e8), 32, axis=1)
    assert np.array_equal(dec * mx_scale, dec * s_elem.astype(np.float64))
    # the four 32-blocks of a 128-block carry the same code
    assert (e8.reshape(256, -1, 4) == e8.reshape(256, -1, 4)[:, :, :1]).all()


def test_conversion_of_non_power_of_two_scales_is_nan():
    assert orc.e8m0_of_scale(0.25) == 125
    assert orc.e8m0_of_scale(2.0 ** -127) == 0
    assert orc.e8m0_of_scale(2.0 ** 127) == 254
    for bad in (0.0279018, 3.0, 0.0, -0.5, float("inf"), float("nan"), 2.0 ** -130):
        assert orc.e8m0_of_scale(bad) == 0xFF
    x = tile(128, 128, 21)
    _, s = orc.ds_quantize_1x128(bits(x))              # amax / 448: not powers of two
    e8 = orc.mx_scales_from_blocks(s, 128, 128, 1)
    pow2 = np.array([math.frexp(float(v))[0] == 0.5 for v in s.ravel()]).reshape(s.shape)
    assert (e8[~np.repeat(pow2, 4, axis=1)] == 0xFF).all()


def test_mx_product_on_converted_scales_equals_block_product():
    a = tile(128, 512, 30)
    b = (tile(256, 512, 31) * 0.02).to(torch.bfloat16)
    qa, sa = orc.ds_quantize_1x128_pow2(bits(a))
    qb, sb = orc.ds_quantize_128x128_pow2(bits(b))
    ea = orc.mx_scales_from_blocks(sa, 128, 512, 1)
    eb = orc.mx_scales_from_blocks(sb, 256, 512, 128)
    y_mx, ab_mx = orc.mx_gemm(qa, ea, E4M3, qb, eb, E4M3)
    y_ds, ab_ds = orc.ds_gemm(qa, sa, qb, sb)
    assert np.allclose(y_mx, y_ds, rtol=0, atol=1e-12 * ab_ds.max())
    assert np.allclose(ab_mx, ab_ds, rtol=1e-12)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_2d32_scale_is_max_of_row_block_scales(golden, fmt):
    g = golden("float8_block_to_mx.txt")
    n = int(g["weight_2d_block"])
    x = tile(128, 256, 40 + fmt, spread=6.0)
    q, s = orc.mx_quantize_2d32(bits(x), fmt)
    assert s.shape == (128 // n, 256 // n)
    _, srow = orc.mx_quantize_rowwise(bits(x), fmt)          # 1x32 scales, pinned elsewhere
    _, scol = orc.mx_quantize_colwise(bits(x), fmt)          # 32x1 scales (transposed)
    for br in range(128 // n):
        for bc in range(256 // n):
            assert s[br, bc] == srow[n * br:n * br + n, bc].max() == scol[n * bc:n * bc + n, br].max()
    xs = x.float().numpy().astype(np.float64)
    for r in range(0, 128, 9):
        for c in range(0, 256, 7):
            k = int(s[r // n, c // n]) - 127
            assert int(q[r, c]) == orc.encode_bruteforce(fmt, math.ldexp(xs[r, c], -k))


def test_2d32_nan_block():
    x = torch.ones(64, 64)
    x[40, 3] = float("nan")
    q, s = orc.mx_quantize_2d32(bits(x.to(torch.bfloat16)), E4M3)
    assert s.tolist() == [[127 - 8, 127 - 8], [0xFF, 127 - 8]]
    assert (q[32:, :32] == 0x7F).all() and (q[:32, :] != 0x7F).all()
