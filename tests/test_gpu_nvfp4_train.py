"""GPU parity of the NVFP4 training options ("Why FP8 training is stable" (magicnetworld.com),
sec 13; "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 3.2) against the CPU oracle:
the 16-point random Hadamard transform, stochastic rounding with one random byte per element
(both through nvfp4_quantize_ex) and 16x16 2-D blocks (nvfp4_quantize_2d).  Codes, block scales
and the global scale bit for bit; the FP4 product of transformed operands within the product
tolerance against the oracle's product of the same quantized operands.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests import quantized
from tests.layouts import chunked_to_plain, pack_fp4, unpack_fp4
from tests.test_gpu_gemm import assert_close

pytestmark = pytest.mark.gpu

SIGNS = 0xB4D2


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def rand_bytes(shape, seed):
    return np.random.default_rng(seed).integers(0, 256, shape, dtype=np.uint8)


def check_ex(x, rht, sr, seed=0):
    rows, cols = x.shape
    rb = rand_bytes((rows, cols), seed) if sr else None
    oq, osc, og = orc.nv_quantize_ex(x, rht=rht, signs=SIGNS if rht else 0, rbits=rb)
    q, s, g = mx.nvfp4_quantize_ex(x.cuda(), rht=rht, signs=SIGNS if rht else 0,
                                   rbits=None if rb is None else torch.from_numpy(rb).cuda())
    assert mx.mx_check() == mx.MX_OK
    assert np.float32(g.item()).view(np.uint32) == np.float32(og).view(np.uint32)
    qn = unpack_fp4(q.cpu().numpy())
    bad = np.argwhere(qn != oq)
    assert bad.size == 0, f"codes differ at {bad[:5].tolist()}: gpu {qn[tuple(bad[0])]} oracle {oq[tuple(bad[0])]}"
    assert np.array_equal(chunked_to_plain(s.cpu().numpy(), rows, cols // 16), osc)
    return q, s, g, (pack_fp4(oq), osc, og)


@pytest.mark.parametrize("rht,sr", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("shape", [(128, 64), (128, 192), (256, 512)])
def test_nvfp4_options_small(rht, sr, shape):
    x = synthetic.with_sparse_outliers(*shape, 4100 + shape[1])
    check_ex(x, rht, sr, seed=shape[0] + shape[1])


@pytest.mark.parametrize("rht,sr", [(True, False), (False, True), (True, True)])
def test_nvfp4_options_full_size(rht, sr):
    x = synthetic.with_sparse_outliers(8192, 8192, 4000)
    check_ex(x, rht, sr, seed=77)


def test_nvfp4_options_edges():
    x = torch.randn(128, 256, generator=torch.Generator().manual_seed(8))
    x[0, :16] = 0.0
    x[1, :16] = 1e-9
    x[2, 0] = 300.0
    x[3, :16] = -0.0
    x[4, :16] = torch.linspace(-7, 7, 16)
    x[5, :16] = 2.0 ** -130
    xb = x.to(torch.bfloat16)
    for rht, sr in ((True, False), (False, True), (True, True)):
        check_ex(xb, rht, sr, seed=5)
    check_ex(torch.zeros(128, 128, dtype=torch.bfloat16), True, True)


def test_default_options_equal_plain_nvfp4():
    x = synthetic.with_sparse_outliers(256, 512, 4200)
    q0, s0, g0 = mx.nvfp4_quantize(x.cuda())
    q1, s1, g1 = mx.nvfp4_quantize_ex(x.cuda())
    assert torch.equal(q0, q1) and torch.equal(s0, s1) and torch.equal(g0, g1)


def test_transformed_operands_multiply_through_the_fp4_gemm():
    M, N, K = 256, 512, 1024
    a = synthetic.with_sparse_outliers(M, K, 4300)
    b = synthetic.with_sparse_outliers(N, K, 4301)
    qa, sa, ga, oa = check_ex(a, True, False)
    qb, sb, gb, ob = check_ex(b, True, False)
    y = mx.nvfp4_gemm(qa, sa, ga, qb, sb, gb, M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.nv_gemm(*oa, *ob)
    assert_close(y.cpu().numpy(), ref, ab, what="transformed operands")


# ------------------------------------------------------------------ 16x16 blocks
def check_2d(x):
    rows, cols = x.shape
    oq, os2, og = orc.nv_quantize_2d16(x)
    qr, sr, qc, sc, g = mx.nvfp4_quantize_2d(x.cuda())
    assert mx.mx_check() == mx.MX_OK
    assert np.float32(g.item()).view(np.uint32) == np.float32(og).view(np.uint32)
    assert np.array_equal(qr.cpu().numpy(), pack_fp4(oq))
    assert np.array_equal(chunked_to_plain(sr.cpu().numpy(), rows, cols // 16), np.repeat(os2, 16, axis=0))
    assert np.array_equal(qc.cpu().numpy(), pack_fp4(oq.T))
    assert np.array_equal(chunked_to_plain(sc.cpu().numpy(), cols, rows // 16), np.repeat(os2.T, 16, axis=0))
    return (qr, sr, qc, sc, g), (pack_fp4(oq), np.repeat(os2, 16, axis=0), pack_fp4(oq.T), np.repeat(os2.T, 16, axis=0), og)


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 256), (8192, 8192)])
def test_nvfp4_2d16(shape):
    check_2d(synthetic.with_sparse_outliers(*shape, 4400 + shape[1]))


def test_nvfp4_2d16_edges():
    x = torch.randn(128, 256, generator=torch.Generator().manual_seed(10))
    x[:16, :16] = 0.0
    x[16:32, 16:32] = 1e-9
    x[40, 200] = 300.0
    x[64:80, 0:16] = 2.0 ** -130
    check_2d(x.to(torch.bfloat16))
    check_2d(torch.zeros(128, 128, dtype=torch.bfloat16))


def test_nvfp4_2d16_weights_in_both_products():
    # the same 16x16-quantized weight serves Y = X W^T (row-wise copy) and dX = G W (the
    # column-wise copy is W^T's row-wise form)
    M, N, K = 256, 512, 256
    x = synthetic.with_sparse_outliers(M, K, 4500)
    w = synthetic.with_sparse_outliers(N, K, 4501)
    gr = synthetic.with_sparse_outliers(M, N, 4502)
    qx, sx, gx, oqx, osx, ogx = quantized.nv(x)
    qg, sg_, gg, oqg, osg, ogg = quantized.nv(gr)
    (qw, sw, qwT, swT, gw), (oqw, osw, oqwT, oswT, ogw) = check_2d(w)
    y = mx.nvfp4_gemm(qx, sx, gx, qw, sw, gw, M, N, K, out_dtype=mx.OUT_F32)
    dx = mx.nvfp4_gemm(qg, sg_, gg, qwT, swT, gw, M, K, N, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    for out, ref_args in ((y, (oqx, osx, ogx, oqw, osw, ogw)), (dx, (oqg, osg, ogg, oqwT, oswT, ogw))):
        ref, ab = orc.nv_gemm(*ref_args)
        assert_close(out.cpu().numpy(), ref, ab, what="2-D weights")
