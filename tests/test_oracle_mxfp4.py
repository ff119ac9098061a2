"""Pins of the oracle's MXFP4 path: E2M1 elements, 32-element blocks, one E8M0 scale per block
("NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 5.5), with the OCP scale rule of the MX
format ("MXFP8 on SM120: software support" (xuesongtap.github.io), sec 0.1).

The pins come from the page's comparison table (tests/golden/mxfp4_format.txt), the E2M1 value
table, exact reconstruction of blocks that are representable, a brute-force nearest-value scan,
and exact rational sums for the product.
"""
import math
from fractions import Fraction

import numpy as np
import torch

import oracle as orc
from oracle import E2M1, E8M0

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16(values, shape):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).reshape(shape)


def test_mxfp4_format_facts(golden):
    g = golden("mxfp4_format.txt")
    n, eb, sb = int(g["block_size"]), int(g["element_bits"]), int(g["scale_bits"])
    assert (n * eb + sb) / n == float(g["bits_per_element"])
    nn = int(g["nvfp4_block_size"])
    assert (nn * eb + sb) / nn == float(g["nvfp4_bits_per_element"])
    # emax of E2M1: its largest value 6 = 1.5 * 2^2
    assert orc.emax(E2M1) == 2 == math.frexp(6.0)[1] - 1
    x = bf16([1.0] * 64, (1, 64))
    q, s = orc.mx_quantize_rowwise(bits(x), E2M1)
    assert q.shape == (1, 64) and s.shape == (1, 64 // n)


def test_mxfp4_scale_rule_and_saturation():
    assert orc.mx_scale_exp(6.0, E2M1) == 0          # [4, 8) -> k = 0
    assert orc.mx_scale_exp(4.0, E2M1) == 0
    assert orc.mx_scale_exp(3.99, E2M1) == -1
    assert orc.mx_scale_exp(8.0, E2M1) == 1
    assert orc.mx_scale_exp(2.0 ** -140, E2M1) == -127
    # amax 7.5 stays at k = 0 and saturates to 6; 0.7 in the same block rounds to 0.5 ([NV] sec 3.2)
    x = bf16([7.5, 0.7, -5.0, 5.0] + [0.0] * 28, (1, 32))
    q, s = orc.mx_quantize_rowwise(bits(x), E2M1)
    assert s[0, 0] == 127
    assert [orc.decode(E2M1, int(c)) for c in q[0, :4]] == [6.0, 0.5, -4.0, 4.0]  # 5 is a tie -> even (4)


def test_mxfp4_representable_blocks_reconstruct_exactly():
    rng = np.random.default_rng(7)
    for k in (-20, -3, 0, 5, 60):
        vals = rng.choice(E2M1_VALUES, 32) * rng.choice([-1.0, 1.0], 32)
        vals[rng.integers(0, 32)] = rng.choice([4.0, 6.0])      # block max in [4, 8)
        x = bf16(list(vals * 2.0 ** k), (1, 32))
        q, s = orc.mx_quantize_rowwise(bits(x), E2M1)
        assert int(s[0, 0]) == 127 + k
        rec = [orc.decode(E2M1, int(c)) * 2.0 ** k for c in q[0]]
        assert rec == [float(v) for v in x[0].float()]


def test_mxfp4_matches_bruteforce_scan():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(8, 256, generator=g) * torch.logspace(-6, 6, 256)).to(torch.bfloat16)
    q, s = orc.mx_quantize_rowwise(bits(x), E2M1)
    xs = x.float().numpy().astype(np.float64)
    for r in range(8):
        for b in range(8):
            blk = xs[r, 32 * b:32 * b + 32]
            amax = np.abs(blk).max()
            k = math.frexp(amax)[1] - 1 - 2                   # floor(log2 amax) - emax
            assert int(s[r, b]) == 127 + k
            for i, v in enumerate(blk):
                assert int(q[r, 32 * b + i]) == orc.encode_bruteforce(E2M1, math.ldexp(float(v), -k))


def test_mxfp4_nan_block_and_transpose():
    vals = [1.0] * 32 + [float("nan")] + [1.0] * 31
    x = bf16(vals, (1, 64))
    q, s = orc.mx_quantize_rowwise(bits(x), E2M1)
    assert list(s[0]) == [127 - 2, 0xFF]
    assert set(q[0, 32:].tolist()) == {0x7}
    g = torch.Generator().manual_seed(12)
    y = (torch.randn(64, 96, generator=g) * 3).to(torch.bfloat16)
    qT, sT = orc.mx_quantize_colwise(bits(y), E2M1)
    q2, s2 = orc.mx_quantize_rowwise(bits(y.t().contiguous()), E2M1)
    assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_mxfp4_gemm_exact_on_tiny_inputs():
    # E2M1 values have at most two significant bits; with scales in a narrow window every
    # partial sum is exact in double, so the oracle equals exact rational arithmetic
    rng = np.random.default_rng(21)
    M, N, K = 4, 6, 96
    qa = rng.integers(0, 16, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 16, (N, K), dtype=np.uint8)
    sa = rng.integers(120, 134, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 134, (N, K // 32), dtype=np.uint8)
    y, ab = orc.mx_gemm(qa, sa, E2M1, qb, sb, E2M1)
    tab = {c: Fraction(v) for c, v in enumerate(E2M1_VALUES + [-v for v in E2M1_VALUES])}
    e8 = lambda c: Fraction(2) ** (int(c) - 127)
    for m in range(M):
        for n in range(N):
            exact = sum(tab[int(qa[m, k])] * e8(sa[m, k // 32]) * tab[int(qb[n, k])] * e8(sb[n, k // 32])
                        for k in range(K))
            assert Fraction(y[m, n]) == exact
            assert ab[m, n] >= abs(y[m, n])


def test_mxfp4_gemm_one_hot_scale():
    rng = np.random.default_rng(22)
    M, N, K = 5, 4, 128
    qa = rng.integers(0, 16, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 16, (N, K), dtype=np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    y0, _ = orc.mx_gemm(qa, sa, E2M1, qb, sb, E2M1)
    sb2 = sb.copy()
    sb2[1, 3] = 129                      # B row 1, k-block 3 scaled by 4
    y1, _ = orc.mx_gemm(qa, sa, E2M1, qb, sb2, E2M1)
    d = y1 - y0
    assert not np.delete(d, 1, axis=1).any()
    dec = np.vectorize(lambda c: orc.decode(E2M1, int(c)))
    assert np.array_equal(d[:, 1], 3 * (dec(qa[:, 96:128]) @ dec(qb[1, 96:128])))
