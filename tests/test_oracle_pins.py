"""Pins of the oracle's quantizers and reference products.

Values come from the worked examples printed on the pages (tests/golden/),
exact rational arithmetic on tiny inputs, library matmuls of dequantized
operands, and structural properties (transpose, one-hot scale changes).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as orc
from oracle import E2M1, E4M3, E5M2, E8M0


def bf16(values, shape=None):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    if shape is not None:
        t = t.reshape(shape)
    return t


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ MX
def test_mx_64_element_example(golden):
    g = golden("mx_64_element_example.txt")
    n = int(g["block_size"])
    v0, v1 = float(g["block0_value"]), float(g["block1_value"])
    x = bf16([v0] * n + [v1] * n, (1, 2 * n))
    q, s = orc.mx_quantize_rowwise(bits(x), E4M3)
    scales = [orc.decode(E8M0, int(c)) for c in s[0]]
    assert scales == [float(g["scale0"]), float(g["scale1"])]
    qv = [orc.decode(E4M3, int(c)) for c in q[0]]
    assert set(qv) == {float(g["q_both_blocks"])}
    # exact reconstruction
    recon = [qv[i] * scales[i // n] for i in range(2 * n)]
    assert recon == [v0] * n + [v1] * n
    # the OCP rule reproduces the page's choice: floor(log2 amax) - emax
    assert orc.mx_scale_exp(v0, E4M3) == 2 and orc.mx_scale_exp(v1, E4M3) == -20
    # one shared scale s = 4: small values underflow to zero, large ones stay exact
    s4 = float(g["shared_scale"])
    assert orc.decode(E4M3, orc.encode(E4M3, v0 / s4)) == float(g["q_both_blocks"])
    assert orc.decode(E4M3, orc.encode(E4M3, v1 / s4)) == float(g["shared_small_q"])


def test_mx_scale_rule_edges():
    assert orc.mx_scale_exp(0.0, E4M3) == -127
    assert orc.mx_scale_exp(448.0, E4M3) == 0          # amax exactly at MAX -> q = 448
    assert orc.mx_scale_exp(511.0, E4M3) == 0          # [256, 512) -> k = 0, 511 saturates
    assert orc.mx_scale_exp(512.0, E4M3) == 1
    assert orc.mx_scale_exp(2.0 ** -133, E4M3) == -127  # clamp
    assert orc.mx_scale_exp(57344.0, E5M2) == 0
    assert orc.mx_scale_exp(2.0 ** 100, E5M2) == 85


def test_mx_saturation_between_448_and_512():
    # amax/2^k lands in (448, 512): the code saturates to 448 (satfinite)
    x = bf16([480.0] + [1.0] * 31, (1, 32))
    q, s = orc.mx_quantize_rowwise(bits(x), E4M3)
    assert s[0, 0] == 127 and q[0, 0] == 0x7E


def test_mx_nan_inf_block_and_zero_block():
    vals = [1.0] * 32 + [float("nan")] + [1.0] * 31 + [float("inf")] + [2.0] * 31 + [0.0] * 16 + [-0.0] * 16
    x = bf16(vals, (1, 128))
    q, s = orc.mx_quantize_rowwise(bits(x), E4M3)
    assert list(s[0]) == [127 - 8, 0xFF, 0xFF, 0]   # amax 1 -> k = 0 - emax
    assert set(q[0, 32:96].tolist()) == {0x7F}
    assert q[0, 96:112].tolist() == [0x00] * 16 and q[0, 112:128].tolist() == [0x80] * 16


def test_mx_bf16_subnormals_scaled_exactly():
    # bf16 subnormals are not flushed: amax = 3*2^-133 -> k = -127, x*2^127 exact
    tiny = [3 * 2.0 ** -133, 2.0 ** -133] + [0.0] * 30
    x = bf16(tiny, (1, 32))
    assert float(x[0, 0]) == 3 * 2.0 ** -133
    q, s = orc.mx_quantize_rowwise(bits(x), E4M3)
    assert s[0, 0] == 0
    assert orc.decode(E4M3, int(q[0, 0])) == 3 * 2.0 ** -6
    assert orc.decode(E4M3, int(q[0, 1])) == 2.0 ** -6


def test_colwise_is_rowwise_of_transpose():
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(96, 64, generator=g) * torch.logspace(-3, 3, 64)).to(torch.bfloat16)
    for fmt in (E4M3, E5M2):
        qT, sT = orc.mx_quantize_colwise(bits(x), fmt)
        q2, s2 = orc.mx_quantize_rowwise(bits(x.t().contiguous()), fmt)
        assert np.array_equal(qT, q2) and np.array_equal(sT, s2)


def test_mx_reconstruction_error_bound():
    # relative error <= 2^-p for elements that stay in the normal range after scaling; with the
    # floor rule the block maximum can land in (MAX, 2^(emax+1)) and saturate, which the
    # page's bound (stated for s = amax/MAX, no overflow) excludes
    g = torch.Generator().manual_seed(5)
    x = torch.randn(64, 256, generator=g).to(torch.bfloat16)
    for fmt, p in ((E4M3, 4), (E5M2, 3)):
        q, s = orc.mx_quantize_rowwise(bits(x), fmt)
        xs = x.float().numpy().astype(np.float64)
        dq = np.vectorize(lambda c: orc.decode(fmt, int(c)))(q)
        sc = np.repeat(np.vectorize(lambda c: orc.decode(E8M0, int(c)))(s), 32, axis=1)
        rec = dq * sc
        min_normal = 2.0 ** -6 if fmt == E4M3 else 2.0 ** -14
        top = 448.0 if fmt == E4M3 else 57344.0
        normal = (np.abs(xs) / sc >= min_normal) & (np.abs(xs) / sc <= top)
        rel = np.abs(rec - xs)[normal] / np.abs(xs)[normal]
        assert rel.max() <= 2.0 ** -p


# ------------------------------------------------------------------ DeepSeek
def test_deepseek_tile_example(golden):
    g = golden("deepseek_tile_example.txt")
    a = float(g["amax"])
    s = orc.ds_scale(a)
    assert abs(s - float(g["scale"])) < 5e-5
    assert abs(a / 28672 - float(g["threshold_full"])) < 5e-7
    xb = float(bf16([float(g["x"])])[0])
    ratio = np.float32(xb) / np.float32(s)
    assert abs(ratio - float(g["ratio"])) < 2e-3
    c = orc.ds_encode(xb, s)
    recon = orc.decode(E4M3, c) * s
    # error within half an ulp (1.74e-3) and within the relative bound 1.88e-3
    assert abs(recon - xb) <= float(g["half_ulp_abs"]) + 1e-6
    assert float(g["half_ulp_abs"]) <= float(g["rel_bound_abs"])
    # the 128-element tile through the full quantizer: outlier 12.5 plus 0.02..0.05 values
    vals = np.linspace(0.02, 0.05, 128)
    vals[17] = a
    vals[3] = float(g["x"])
    x = bf16(vals.tolist(), (1, 128))
    q, sc = orc.ds_quantize_1x128(bits(x))
    assert sc[0, 0] == np.float32(s)
    assert q[0, 3] == c
    # every non-outlier element stays in the normal range (code exponent field != 0)
    assert all((int(cc) >> 3) & 0xF for cc in q[0])


def test_deepseek_subnormal_example(golden):
    g = golden("deepseek_tile_example.txt")
    s = orc.ds_scale(float(g["amax_tensor"]))
    assert abs(s - float(g["scale_tensor"])) < 5e-4
    assert abs(float(g["amax_tensor"]) / 28672 - float(g["threshold_tensor"])) < 5e-5
    xb = float(bf16([float(g["x_small"])])[0])
    assert abs(xb / s - float(g["scaled_small"])) < 5e-5
    c = orc.ds_encode(xb, s)
    assert (c >> 3) & 0xF == 0 and c & 0x7 != 0      # subnormal code on the 2^-9 grid
    recon = orc.decode(E4M3, c) * s
    rel = abs(recon - xb) / xb
    assert abs(rel - float(g["rel_err_small"])) < 0.01
    assert rel <= float(g["rel_bound_small"])


def test_underflow_thresholds(golden):
    g = golden("underflow_thresholds.txt")
    a = 448.0                       # s = 1 exactly, so x/s = x
    s = orc.ds_scale(a)
    assert s == 1.0
    full = a / float(g["full_mantissa_den"])     # = 2^-6: smallest normal
    assert orc.ds_encode(full, s) == 0x08
    assert orc.ds_encode(float(np.nextafter(np.float32(full), np.float32(0))), s) == 0x08  # rounds up
    zero = a / float(g["zero_den"])             # = 2^-10: tie -> even -> 0
    assert orc.ds_encode(zero, s) == 0x00
    assert orc.ds_encode(float(np.nextafter(np.float32(zero), np.float32(1))), s) == 0x01


def test_deepseek_128x128_block_scale():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(256, 256, generator=g) * 0.02)
    x[130, 200] = 7.0
    x = x.to(torch.bfloat16)
    q, s = orc.ds_quantize_128x128(bits(x))
    amax = x.float().abs().reshape(2, 128, 2, 128).amax(dim=(1, 3)).numpy()
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    assert orc.decode(E4M3, int(q[130, 200])) == 448.0
    # 1x128 of the same rows differs from the 128x128 block result (different grouping)
    q1, s1 = orc.ds_quantize_1x128(bits(x))
    assert not np.array_equal(q1, q)


def test_deepseek_zero_tile():
    x = bf16([0.0] * 128, (1, 128))
    q, s = orc.ds_quantize_1x128(bits(x))
    assert s[0, 0] == 1.0 and not q.any()


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_worked_example(golden):
    g = golden("nvfp4_worked_example.txt")
    sg = orc.nv_global_scale(float(g["global_amax"]))
    assert abs(sg - float(g["s_global"])) < 5e-6
    t = (np.float32(float(g["block_amax"])) / np.float32(6)) / np.float32(sg)
    assert abs(t - float(g["s_block_raw"])) < 0.05
    code, s_hat = orc.nv_block_scale(sg, float(g["block_amax"]))
    assert orc.decode(E4M3, code) == float(g["s_block_e4m3"])
    y = np.float32(float(g["block_amax"])) / np.float32(s_hat)
    assert abs(y - float(g["scaled_element"])) < 5e-3
    qc = orc.nv_encode(float(g["block_amax"]), s_hat)
    assert orc.decode(E2M1, qc) == float(g["q_element"])
    recon = orc.decode(E2M1, qc) * s_hat
    assert abs(recon - float(g["reconstruction"])) < float(g["reconstruction_tol"])
    assert abs(recon - 2.41607) < 1e-4     # exact FP32 arithmetic


def test_nvfp4_quantize_structure():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(32, 64, generator=g)
    x[5, 7] = 40.0
    x = x.to(torch.bfloat16)
    qp, s, sg = orc.nv_quantize(bits(x))
    xs = x.float().numpy()
    assert sg == np.float32(np.abs(xs).max()) / np.float32(2688.0)
    # the block holding the global amax gets scale code 448 (t = 448 exactly) and q = 6
    assert orc.decode(E4M3, int(s[5, 0])) == 448.0
    lo = qp & 0xF
    hi = qp >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(32, 64)
    assert orc.decode(E2M1, int(codes[5, 7])) == 6.0
    # reconstruction error: at most half of the E2M1 step at that magnitude, times s_hat
    dq = np.vectorize(lambda c: orc.decode(E2M1, int(c)))(codes)
    sh = np.vectorize(lambda c: orc.decode(E4M3, int(c)))(s).astype(np.float64) * sg
    rec = dq * np.repeat(sh, 16, axis=1)
    err = np.abs(rec - xs)
    step = np.where(np.abs(dq) < 2, 0.5, np.where(np.abs(dq) < 4, 1.0, 2.0))
    assert (err <= 0.5 * step * np.repeat(sh, 16, axis=1) * 1.001 + 1e-12).all()


def test_nvfp4_zero_tensor():
    x = bf16([0.0] * 64, (2, 32))
    qp, s, sg = orc.nv_quantize(bits(x))
    assert sg == 1.0 and not qp.any() and not s.any()


# ------------------------------------------------------------------ products
def _exact_mx(qa, sa, fa, qb, sb, fb):
    M, K = qa.shape
    N = qb.shape[0]
    out = np.empty((M, N), dtype=object)
    da = [[Fraction(orc.decode(fa, int(c))) for c in row] for row in qa]
    db = [[Fraction(orc.decode(fb, int(c))) for c in row] for row in qb]
    ea = [[Fraction(orc.decode(E8M0, int(c))) for c in row] for row in sa]
    eb = [[Fraction(orc.decode(E8M0, int(c))) for c in row] for row in sb]
    for m in range(M):
        for n in range(N):
            out[m, n] = sum(da[m][k] * ea[m][k // 32] * db[n][k] * eb[n][k // 32] for k in range(K))
    return out


@pytest.mark.parametrize("K", [32, 64, 128])
def test_mx_gemm_exact_on_tiny_inputs(K):
    # codes and scales drawn from a window narrow enough that every partial sum is exact in
    # double, so the oracle must agree with exact rational arithmetic bit for bit
    rng = np.random.default_rng(K)
    M, N = 5, 7
    sign = lambda shape: rng.integers(0, 2, shape, dtype=np.uint8) << 7
    qa = rng.integers(0x28, 0x58, (M, K), dtype=np.uint8) | sign((M, K))
    qb = rng.integers(0x30, 0x48, (N, K), dtype=np.uint8) | sign((N, K))
    sa = rng.integers(124, 131, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(124, 131, (N, K // 32), dtype=np.uint8)
    y, ab = orc.mx_gemm(qa, sa, E4M3, qb, sb, E5M2)
    exact = _exact_mx(qa, sa, E4M3, qb, sb, E5M2)
    for m in range(M):
        for n in range(N):
            assert Fraction(y[m, n]) == exact[m, n]
    assert (ab >= np.abs(y)).all()


def test_mx_gemm_wide_range_within_double_rounding():
    rng = np.random.default_rng(99)
    M, N, K = 4, 6, 64
    qa = rng.integers(0, 256, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x11        # no NaN codes
    qb[(qb & 0x7C) == 0x7C] = 0x22        # no E5M2 Inf/NaN codes
    sa = rng.integers(100, 150, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(100, 150, (N, K // 32), dtype=np.uint8)
    y, ab = orc.mx_gemm(qa, sa, E4M3, qb, sb, E5M2)
    exact = _exact_mx(qa, sa, E4M3, qb, sb, E5M2)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(y[m, n]) - exact[m, n]) <= Fraction(K * 2.0 ** -52) * Fraction(ab[m, n])


def test_mx_gemm_matches_matmul_of_dequantized():
    rng = np.random.default_rng(2)
    M, N, K = 16, 24, 128
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8) | (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7)
    qb = rng.integers(0, 0x7E, (N, K), dtype=np.uint8)
    sa = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 135, (N, K // 32), dtype=np.uint8)
    dec = np.vectorize(lambda c: orc.decode(E4M3, int(c)))
    e8 = np.vectorize(lambda c: orc.decode(E8M0, int(c)))
    A = dec(qa) * np.repeat(e8(sa), 32, axis=1)
    B = dec(qb) * np.repeat(e8(sb), 32, axis=1)
    y, ab = orc.mx_gemm(qa, sa, E4M3, qb, sb, E4M3)
    assert np.allclose(y, A @ B.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(ab, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    # row subset returns the same rows
    ysub, _ = orc.mx_gemm(qa, sa, E4M3, qb, sb, E4M3, rows=[3, 11])
    assert np.array_equal(ysub, y[[3, 11]])


def test_mx_gemm_one_hot_scale():
    rng = np.random.default_rng(4)
    M, N, K = 6, 5, 128
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 0x7E, (N, K), dtype=np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    y0, _ = orc.mx_gemm(qa, sa, E4M3, qb, sb, E4M3)
    sa2 = sa.copy()
    sa2[2, 1] = 128                     # one scale doubled: row 2, k-block 1
    y1, _ = orc.mx_gemm(qa, sa2, E4M3, qb, sb, E4M3)
    d = y1 - y0
    assert not d[np.arange(M) != 2].any()
    dec = np.vectorize(lambda c: orc.decode(E4M3, int(c)))
    block = dec(qa[2, 32:64]) @ dec(qb[:, 32:64]).T
    assert np.array_equal(d[2], block)


def test_nv_gemm_scale_outside_sum(golden):
    g = golden("scale_outside_sum.txt")
    qv = [float(v) for v in g["q"].split(",")]
    pv = [float(v) for v in g["p"].split(",")]
    s = float(g["s"])
    enc = lambda v: orc.encode(E2M1, v)
    # one 16-element block, zero padded
    ca = [enc(v) for v in qv] + [0] * 12
    cb = [enc(v) for v in pv] + [0] * 12
    pack = lambda c: np.array([[c[i] | (c[i + 1] << 4) for i in range(0, 16, 2)]], np.uint8)
    sa = np.array([[orc.encode(E4M3, s)]], np.uint8)
    sb = np.array([[orc.encode(E4M3, 1.0)]], np.uint8)
    assert sa[0, 0] == 0x44 and sb[0, 0] == 0x38
    y, ab = orc.nv_gemm(pack(ca), sa, 1.0, pack(cb), sb, 1.0)
    assert y[0, 0] == float(g["result"])
    assert sum(a * b for a, b in zip(qv, pv)) == float(g["raw_dot"])
    # dequantize-then-sum gives the same value
    assert sum(s * a * b for a, b in zip(qv, pv)) == float(g["result"])
    # the global scales multiply the whole result
    y2, _ = orc.nv_gemm(pack(ca), sa, 0.5, pack(cb), sb, 4.0)
    assert y2[0, 0] == 2.0 * float(g["result"])


def test_nv_gemm_matches_matmul_of_dequantized():
    rng = np.random.default_rng(8)
    M, N, K = 8, 12, 64
    qa = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x20, 0x60, (M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x20, 0x60, (N, K // 16), dtype=np.uint8)
    dec2 = np.vectorize(lambda c: orc.decode(E2M1, int(c)))
    dec8 = np.vectorize(lambda c: orc.decode(E4M3, int(c)))
    unpack = lambda q: np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)
    A = dec2(unpack(qa)) * np.repeat(dec8(sa), 16, axis=1)
    B = dec2(unpack(qb)) * np.repeat(dec8(sb), 16, axis=1)
    y, _ = orc.nv_gemm(qa, sa, 0.25, qb, sb, 3.0)
    assert np.allclose(y, 0.75 * (A @ B.T), rtol=1e-12, atol=1e-12)


def test_ds_gemm_matches_matmul_of_dequantized():
    rng = np.random.default_rng(6)
    M, N, K = 8, 256, 256
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 0x7E, (N, K), dtype=np.uint8)
    sa = rng.uniform(0.01, 2, (M, K // 128)).astype(np.float32)
    sb = rng.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
    dec = np.vectorize(lambda c: orc.decode(E4M3, int(c)))
    A = dec(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    B = dec(qb) * np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0), 128, axis=1)
    y, _ = orc.ds_gemm(qa, sa, qb, sb)
    assert np.allclose(y, A @ B.T, rtol=1e-12, atol=1e-12)


def test_ds_gemm_tracks_fp64_of_unquantized_inputs():
    # K = 4096 random matrices: the quantized product stays close to the fp64 product of the
    # unquantized inputs (error from E4M3 rounding only, no accumulation loss in the oracle).
    g = torch.Generator().manual_seed(21)
    a = torch.randn(4, 4096, generator=g).to(torch.bfloat16)
    b = (torch.randn(128, 4096, generator=g) * 0.02).to(torch.bfloat16)
    qa, sa = orc.ds_quantize_1x128(bits(a))
    qb, sb = orc.ds_quantize_128x128(bits(b))
    y, ab = orc.ds_gemm(qa, sa, qb, sb)
    ref = a.double().numpy() @ b.double().numpy().T
    absref = np.abs(a.double().numpy()) @ np.abs(b.double().numpy()).T
    rel = np.abs(y - ref) / absref
    assert rel.max() < 2.0 ** -4          # per-product relative error <= 2^-4 bounds the sum
    assert np.median(rel) < 5e-3


# ------------------------------------------------------------------ MX quantization of FP32 values
def test_mx_rowwise_f32_equals_bf16_path_on_bf16_values():
    g = torch.Generator().manual_seed(13)
    x = (torch.randn(64, 256, generator=g) * torch.logspace(-9, 9, 256)).to(torch.bfloat16)
    for fmt in (E4M3, E5M2):
        q1, s1 = orc.mx_quantize_rowwise(bits(x), fmt)
        q2, s2 = orc.mx_quantize_rowwise_f32(x.float().numpy(), fmt)
        assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_mx_rowwise_f32_full_mantissa_matches_bruteforce():
    # FP32 values with 24-bit mantissas (not bf16): scale by the floor rule, codes by a scan
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((8, 128)) * np.exp2(rng.integers(-30, 30, (8, 128)))).astype(np.float32)
    x[3, 40] = np.inf
    q, s = orc.mx_quantize_rowwise_f32(x, E4M3)
    for r in range(8):
        for b in range(4):
            blk = x[r, 32 * b:32 * b + 32].astype(np.float64)
            if not np.isfinite(blk).all():
                assert s[r, b] == 0xFF and (q[r, 32 * b:32 * b + 32] == 0x7F).all()
                continue
            k = math.frexp(np.abs(blk).max())[1] - 1 - 8
            k = max(k, -127)
            assert s[r, b] == 127 + k
            for i in range(32):
                assert q[r, 32 * b + i] == orc.encode_bruteforce(E4M3, math.ldexp(float(blk[i]), -k))
