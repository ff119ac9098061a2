"""GPU parity of the MXFP8 GEMM with its MX output quantization fused into the epilogue
(mx_gemm_mxout): codes and scales equal the oracle's row-wise MX quantization of the same
kernel's FP32 results (mx_gemm with FP32 output, checked against the double-precision oracle
product), bit for bit -- the decision is taken in the kernel's precision, FP32.  Also: Inf
results, E5M2 output, and the fused output used directly as the A operand of the next product.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests.layouts import chunked_to_plain, plain_to_chunked
from tests.test_gpu_gemm import assert_close

pytestmark = pytest.mark.gpu

MXFMT = {orc.E4M3: mx.E4M3, orc.E5M2: mx.E5M2}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    sign = lambda shape: rng.integers(0, 2, shape, dtype=np.uint8) << 7
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8) | sign((M, K))
    qb = rng.integers(0, 0x7E, (N, K), dtype=np.uint8) | sign((N, K))
    sa = rng.integers(110, 140, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
    return qa, sa, qb, sb


def check_fused(qa, sa, qb, sb, M, N, K, fmt, rows=None):
    args = (dev(qa), dev(plain_to_chunked(sa)), mx.E4M3, dev(qb), dev(plain_to_chunked(sb)), mx.E4M3)
    y32 = mx.mx_gemm(*args, M, N, K, out_dtype=mx.OUT_F32)
    q, s = mx.mx_gemm_mxout(*args, M, N, K, out_elem=MXFMT[fmt])
    assert mx.mx_check() == mx.MX_OK
    y = y32.cpu().numpy()
    r = np.arange(M) if rows is None else rows
    oq, osc = orc.mx_quantize_rowwise_f32(y[r], fmt)
    qn = q.cpu().numpy()[r]
    bad = np.argwhere(qn != oq)
    assert bad.size == 0, f"codes differ at {bad[:5].tolist()}"
    assert np.array_equal(chunked_to_plain(s.cpu().numpy(), M, N // 32)[r], osc)
    return y, q, s


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 768, 1024)])
def test_fused_quantization_equals_quantized_fp32_results(fmt, M, N, K):
    qa, sa, qb, sb = operands(M, N, K, M + N + K + fmt)
    y, _, _ = check_fused(qa, sa, qb, sb, M, N, K, fmt)
    ref, ab = orc.mx_gemm(qa, sa, orc.E4M3, qb, sb, orc.E4M3)
    assert_close(y, ref, ab, what="FP32 results before quantization")


def test_fused_quantization_inf_results():
    M, N, K = 256, 256, 128
    qa, sa, qb, sb = operands(M, N, K, 9)
    qa[5, :] = 0x7E
    sa[5, :] = 254                      # 448 * 2^127 in every element of row 5 -> Inf products
    qb[:, :] = 0x7E
    _, q, s = check_fused(qa, sa, qb, sb, M, N, K, orc.E4M3)
    assert (chunked_to_plain(s.cpu().numpy(), M, N // 32)[5] == 0xFF).all()


def test_fused_full_size_fprop():
    x, w, _ = synthetic.mxfp8_linear()
    qx, sx, _, _ = mx.mx_quantize(x.cuda(), layout=mx.ROWWISE)
    qw, sw, _, _ = mx.mx_quantize(w.cuda(), layout=mx.ROWWISE)
    M, N, K = 8192, 14336, 4096
    y32 = mx.mx_gemm(qx, sx, mx.E4M3, qw, sw, mx.E4M3, M, N, K, out_dtype=mx.OUT_F32)
    q, s = mx.mx_gemm_mxout(qx, sx, mx.E4M3, qw, sw, mx.E4M3, M, N, K)
    assert mx.mx_check() == mx.MX_OK
    rows = np.array([0, 1, 255, 256, 4097, 8191])
    oq, osc = orc.mx_quantize_rowwise_f32(y32.cpu().numpy()[rows], orc.E4M3)
    assert np.array_equal(q.cpu().numpy()[rows], oq)
    assert np.array_equal(chunked_to_plain(s.cpu().numpy(), M, N // 32)[rows], osc)


def test_fused_output_feeds_the_next_product():
    # Y = X W1^T quantized in the epilogue, then Z = Y W2^T reading Y's codes and scales as A
    M, N1, N2, K = 256, 512, 256, 256
    qa, sa, qb, sb = operands(M, N1, K, 21)
    _, q, s = check_fused(qa, sa, qb, sb, M, N1, K, orc.E4M3)
    rng = np.random.default_rng(22)
    q2 = rng.integers(0, 0x7E, (N2, N1), dtype=np.uint8)
    s2 = rng.integers(120, 134, (N2, N1 // 32), dtype=np.uint8)
    z = mx.mx_gemm(q, s, mx.E4M3, dev(q2), dev(plain_to_chunked(s2)), mx.E4M3, M, N2, N1, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(q.cpu().numpy(), chunked_to_plain(s.cpu().numpy(), M, N1 // 32), orc.E4M3, q2, s2, orc.E4M3)
    assert_close(z.cpu().numpy(), ref, ab, what="chained product")
