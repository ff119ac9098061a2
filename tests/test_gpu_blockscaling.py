"""GPU parity of Float8BlockScaling in MX form and of 2-D 32x32 MX weight blocks ("MXFP8 on SM120:
software support" (xuesongtap.github.io), sec 1.3) against the CPU oracle.

Power-of-two 1x128 / 128x128 quantizers and the 2-D 32x32 quantizer: codes and scales bit for
bit.  The scale conversion: E8M0 bytes bit for bit (NaN code for scales that are not powers of
two).  The product: converted scales through mx_gemm against the oracle's block-scaled product
(Σ_kb sA sB Σ qA qB), within |y - y_ref| <= 1e-5 * sum_k |a_k b_k| (+ one bf16 ulp for bf16).
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests import quantized
from tests.layouts import chunked_to_plain, plain_to_chunked
from tests.test_gpu_gemm import assert_close

pytestmark = pytest.mark.gpu

MXFMT = {orc.E4M3: mx.E4M3, orc.E5M2: mx.E5M2}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def edge_rows(x):
    x = x.clone().float()
    x[0, :128] = 0.0
    x[1, :128] = 2.0 ** -130                  # bf16 subnormals: the scale clamps at 2^-127
    x[2, :128] = -448.0                       # amax exactly 448 -> s = 1
    x[3, 5] = 3.0e38                          # near the bf16 maximum
    x[4, :128] = torch.linspace(-1, 1, 128)
    return x.to(torch.bfloat16)


# ------------------------------------------------------------------ power-of-two quantizers
@pytest.mark.parametrize("shape", [(128, 128), (256, 640), (4096, 7168)])
def test_pow2_1x128_quantize(shape):
    x = edge_rows(synthetic.normal(*shape, 1.0, 5400))
    oq, osc = orc.ds_quantize_1x128_pow2(x)
    q, s, _, _ = mx.mx_quantize(x.cuda(), block=128, block_rows=1, sfmt=mx.SCALE_FP32_POW2, layout=mx.ROWWISE)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().T.view(np.uint32), osc.view(np.uint32))
    assert mx.mx_check() == mx.MX_OK


@pytest.mark.parametrize("shape", [(128, 128), (384, 256), (2048, 7168)])
def test_pow2_128x128_quantize(shape):
    x = edge_rows(synthetic.normal(*shape, 0.02, 5401))
    oq, osc = orc.ds_quantize_128x128_pow2(x)
    q, s, _, _ = mx.mx_quantize(x.cuda(), block=128, block_rows=128, sfmt=mx.SCALE_FP32_POW2, layout=mx.ROWWISE)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), osc.view(np.uint32))


# ------------------------------------------------------------------ scale conversion
@pytest.mark.parametrize("block_rows", [1, 128])
def test_scale_conversion_bit_exact(block_rows):
    rows, cols = 384, 640
    x = synthetic.normal(rows, cols, 1.0, 5410 + block_rows)
    q, s, _, _ = mx.mx_quantize(x.cuda(), block=128, block_rows=block_rows, sfmt=mx.SCALE_FP32_POW2,
                                layout=mx.ROWWISE)
    e8 = mx.mx_scales_from_fp32_blocks(s, rows, cols, block_rows)
    s_plain = s.cpu().numpy().T.copy() if block_rows == 1 else s.cpu().numpy()
    ref = orc.mx_scales_from_blocks(s_plain, rows, cols, block_rows)
    assert np.array_equal(chunked_to_plain(e8.cpu().numpy(), rows, cols // 32), ref)


def test_scale_conversion_marks_non_powers_of_two():
    rows, cols = 128, 256
    vals = np.array([0.25, 2.0 ** -127, 2.0 ** 127, 0.0279018, 3.0, 0.0, -0.5, np.inf, np.nan, 2.0 ** -130],
                    np.float32)
    s = np.resize(vals, (cols // 128, rows)).astype(np.float32)          # [cols/128][rows]
    e8 = mx.mx_scales_from_fp32_blocks(torch.from_numpy(s).cuda(), rows, cols, 1)
    ref = orc.mx_scales_from_blocks(s.T.copy(), rows, cols, 1)
    assert np.array_equal(chunked_to_plain(e8.cpu().numpy(), rows, cols // 32), ref)
    assert {0xFF, 125, 0, 254} <= set(np.unique(ref).tolist())


def block_scaled_through_mx(a, b, out_dtype):
    M, K = a.shape
    N = b.shape[0]
    qa, sa, oqa, osa = quantized.ds(a, 1, pow2=True)
    qb, sb, oqb, osb = quantized.ds(b, 128, pow2=True)
    ea = mx.mx_scales_from_fp32_blocks(sa, M, K, 1)
    eb = mx.mx_scales_from_fp32_blocks(sb, N, K, 128)
    y = mx.mx_gemm(qa, ea, mx.E4M3, qb, eb, mx.E4M3, M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    return y, oqa, osa, oqb, osb


@pytest.mark.parametrize("M,N,K", [(128, 384, 256), (256, 256, 512), (512, 768, 1024)])
@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_block_scaled_product_through_mx_gemm(M, N, K, out_dtype):
    a = synthetic.normal(M, K, 1.0, 5420 + K)
    b = synthetic.normal(N, K, 0.02, 5421 + K)
    y, qa, sa, qb, sb = block_scaled_through_mx(a, b, out_dtype)
    ref, ab = orc.ds_gemm(qa, sa, qb, sb)
    assert_close(y.float().cpu().numpy(), ref, ab, bf16=out_dtype == mx.OUT_BF16, what="float8 blocks via mx")


def test_block_scaled_product_through_mx_gemm_full_size():
    a, b = synthetic.deepseek_pair()               # 4096 x 7168, 2048 x 7168
    M, K = a.shape
    N = b.shape[0]
    y, qa, sa, qb, sb = block_scaled_through_mx(a, b, mx.OUT_BF16)
    rows = np.array([0, 7, 128, 2049, 4095])
    ref, ab = orc.ds_gemm(qa, sa, qb, sb, rows=rows)
    assert_close(y[torch.from_numpy(rows).cuda()].float().cpu().numpy(), ref, ab, bf16=True, what="full size")


# ------------------------------------------------------------------ 2-D 32x32 blocks
def check_2d(x, fmt, layouts=(mx.BOTH, mx.ROWWISE, mx.COLWISE)):
    rows, cols = x.shape
    oq, os2 = orc.mx_quantize_2d32(x, fmt)
    srow = np.repeat(os2, 32, axis=0)                 # [rows][cols/32]: row r -> block row r / 32
    scol = np.repeat(os2.T, 32, axis=0)               # [cols][rows/32]: column c -> block column c / 32
    for layout in layouts:
        qr, sr, qc, sc = mx.mx_quantize(x.cuda(), block=32, block_rows=32, elem=MXFMT[fmt], layout=layout)
        if layout & mx.ROWWISE:
            assert np.array_equal(qr.cpu().numpy(), oq)
            assert np.array_equal(chunked_to_plain(sr.cpu().numpy(), rows, cols // 32), srow)
        if layout & mx.COLWISE:
            assert np.array_equal(qc.cpu().numpy(), oq.T)
            assert np.array_equal(chunked_to_plain(sc.cpu().numpy(), cols, rows // 32), scol)
    assert mx.mx_check() == mx.MX_OK


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (1152, 640)])
def test_2d32_quantize(fmt, shape):
    g = torch.Generator().manual_seed(shape[0] + 3 * shape[1] + fmt)
    x = (torch.randn(*shape, generator=g) * torch.logspace(-12, 12, shape[1])).to(torch.bfloat16)
    check_2d(x, fmt)


def test_2d32_edge_blocks():
    x = torch.randn(128, 256, generator=torch.Generator().manual_seed(9))
    x[:32, :32] = 0.0
    x[40, 70] = float("nan")                  # block (1, 2)
    x[100, 200] = float("inf")                # block (3, 6)
    x[64:96, 128:160] = 2.0 ** -130
    x[5, 250] = 480.0                         # saturation inside block (0, 7)
    for fmt in (orc.E4M3, orc.E5M2):
        check_2d(x.to(torch.bfloat16), fmt)


def test_2d32_full_size_weight():
    _, w, _ = synthetic.mxfp8_linear()        # 14336 x 4096
    check_2d(w, orc.E4M3, layouts=(mx.BOTH,))


def test_2d32_weights_in_fprop_and_dgrad():
    M, N, K = 256, 512, 384
    x = synthetic.normal(M, K, 1.0, 5430)
    w = synthetic.normal(N, K, 0.02, 5431)
    g = synthetic.normal(M, N, 1e-3, 5432)
    qx, sx, oqx, osx = quantized.mx_rowwise(x, orc.E4M3)
    (qw, sw, qwT, swT), (oqw, osw, oqwT, oswT) = quantized.mx_both(w, orc.E4M3, block_rows=32)
    qg, sg, oqg, osg = quantized.mx_rowwise(g, orc.E5M2)
    y = mx.mx_gemm(qx, sx, mx.E4M3, qw, sw, mx.E4M3, M, N, K, out_dtype=mx.OUT_F32)          # fprop
    dx = mx.mx_gemm(qg, sg, mx.E5M2, qwT, swT, mx.E4M3, M, K, N, out_dtype=mx.OUT_F32)      # dgrad
    assert mx.mx_check() == mx.MX_OK
    for out, ref_args in ((y, (oqx, osx, orc.E4M3, oqw, osw, orc.E4M3)),
                          (dx, (oqg, osg, orc.E5M2, oqwT, oswT, orc.E4M3))):
        ref, ab = orc.mx_gemm(*ref_args)
        assert_close(out.cpu().numpy(), ref, ab, what="2-D weights")
