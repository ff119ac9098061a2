"""GPU parity of the MXFP8 GEMM with its MX output quantization fused into the epilogue
(mx_gemm_mxout).  The decision is taken in the kernel's precision, FP32, so the operands are
built for exact FP32 sums: every A and B value is a signed power of two (E4M3 codes with a zero
mantissa) and the scales are constant along K for each row and column, so within one output all
products are multiples of one power of two and span at most 2^6 of it; with K <= 4096 every
partial sum, in any order, is an integer below 2^18 in those units and exact in FP32.  The
oracle's double-precision product is then exactly the FP32 value the kernel quantizes, and the
expected codes and scales are the oracle's MX quantization of the oracle's product -- nothing on
the reference side comes from the GPU.  Cases: E4M3 and E5M2 outputs, several tile counts, the
full 8192 x 14336 x 4096 fprop shape on sampled rows, Inf results, and the fused output used
directly as the A operand of the next product.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
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
    """Exact-sum operands: E4M3 codes of 0 or +-2^e (e = -1 .. 2), E8M0 scales constant along K
    (2^-4 .. 2^4 per row of A, 2^-2 .. 2^2 per row of B)."""
    rng = np.random.default_rng(seed)

    def codes(shape):
        e = rng.integers(6, 10, shape, dtype=np.uint8)           # biased exponent 6..9: 2^-1 .. 2^2
        q = (e << 3) | (rng.integers(0, 2, shape, dtype=np.uint8) << 7)
        q[rng.random(shape) < 0.1] = 0
        return q
    qa, qb = codes((M, K)), codes((N, K))
    sa = np.repeat((127 + (np.arange(M) * 7) % 9 - 4).astype(np.uint8)[:, None], K // 32, axis=1)
    sb = np.repeat((127 + np.arange(N) % 5 - 2).astype(np.uint8)[:, None], K // 32, axis=1)
    return qa, sa, qb, sb


def check_fused(qa, sa, qb, sb, M, N, K, fmt, rows=None):
    """Fused codes and scales against the oracle's MX quantization of the oracle's product (exact
    in FP32 for the operands above, which the kernel's FP32 results must equal)."""
    args = (dev(qa), dev(plain_to_chunked(sa)), mx.E4M3, dev(qb), dev(plain_to_chunked(sb)), mx.E4M3)
    y32 = mx.mx_gemm(*args, M, N, K, out_dtype=mx.OUT_F32)
    q, s = mx.mx_gemm_mxout(*args, M, N, K, out_elem=MXFMT[fmt])
    assert mx.mx_check() == mx.MX_OK
    r = np.arange(M) if rows is None else np.asarray(rows)
    ref, _ = orc.mx_gemm(qa, sa, orc.E4M3, qb, sb, orc.E4M3, rows=None if rows is None else r)
    with np.errstate(over="ignore"):
        ref32 = ref.astype(np.float32)
    finite = np.isfinite(ref32)
    assert np.array_equal(ref32[finite].astype(np.float64), ref[finite]), "operands do not give exact FP32 sums"
    y = y32.cpu().numpy()[r]
    assert np.array_equal(y[finite], ref32[finite]), "FP32 results differ from the exact product"
    oq, osc = orc.mx_quantize_rowwise_f32(ref32, fmt)
    qn = q.cpu().numpy()[r]
    bad = np.argwhere(qn != oq)
    assert bad.size == 0, f"codes differ at {bad[:5].tolist()}"
    assert np.array_equal(chunked_to_plain(s.cpu().numpy(), M, N // 32)[r], osc)
    return q, s, oq, osc


def check_fused_ex(qa, sa, qb, sb, M, N, K, fmt, layout, cols=None):
    """mx_gemm_mxout_ex: the row-wise copy as check_fused; the column-wise copy (32x1 blocks,
    stored transposed) against the oracle's MX quantization of the transposed oracle product, on
    all output columns or the sampled ones (each column needs all M rows of the product)."""
    args = (dev(qa), dev(plain_to_chunked(sa)), mx.E4M3, dev(qb), dev(plain_to_chunked(sb)), mx.E4M3)
    q, s, qT, sT = mx.mx_gemm_mxout_ex(*args, M, N, K, out_elem=MXFMT[fmt], layout=layout)
    assert mx.mx_check() == mx.MX_OK
    c = np.arange(N) if cols is None else np.asarray(cols)
    ref, _ = orc.mx_gemm(qa, sa, orc.E4M3, qb[c], sb[c], orc.E4M3)      # [M][len(c)]
    with np.errstate(over="ignore"):
        ref32 = ref.astype(np.float32)
    finite = np.isfinite(ref32)
    assert np.array_equal(ref32[finite].astype(np.float64), ref[finite]), "operands do not give exact FP32 sums"
    if layout & mx.ROWWISE and cols is None:
        oq, osc = orc.mx_quantize_rowwise_f32(ref32, fmt)
        assert np.array_equal(q.cpu().numpy(), oq), "row codes"
        assert np.array_equal(chunked_to_plain(s.cpu().numpy(), M, N // 32), osc), "row scales"
    if layout & mx.COLWISE:
        oqT, osT = orc.mx_quantize_rowwise_f32(np.ascontiguousarray(ref32.T), fmt)   # [len(c)][M]
        qTn = qT.cpu().numpy()[c]
        bad = np.argwhere(qTn != oqT)
        assert bad.size == 0, f"column codes differ at {bad[:5].tolist()}"
        assert np.array_equal(chunked_to_plain(sT.cpu().numpy(), N, M // 32)[c], osT), "column scales"
    return q, s, qT, sT


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
@pytest.mark.parametrize("layout", [mx.COLWISE, mx.BOTH])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 768, 1024), (768, 512, 128)])
def test_fused_column_wise_copy(fmt, layout, M, N, K):
    qa, sa, qb, sb = operands(M, N, K, 7 * M + N + K + fmt)
    check_fused_ex(qa, sa, qb, sb, M, N, K, fmt, layout)


def test_fused_column_wise_copy_inf_results():
    M, N, K = 256, 256, 128
    qa, sa, qb, sb = operands(M, N, K, 19)
    qa[5, :] = 0x7E
    sa[5, :] = 254                      # every result of row 5 is Inf -> every 32x1 block holding row 5
    qb[:, :] = 0x7E
    _, _, _, sT = check_fused_ex(qa, sa, qb, sb, M, N, K, orc.E4M3, mx.BOTH)
    assert (chunked_to_plain(sT.cpu().numpy(), N, M // 32)[:, 0] == 0xFF).all()


def test_fused_column_wise_full_size_fprop():
    # the fprop shape of the linear-layer workload, exact-sum operands, sampled output columns
    M, N, K = 8192, 14336, 4096
    qa, sa, qb, sb = operands(M, N, K, 41)
    check_fused_ex(qa, sa, qb, sb, M, N, K, orc.E4M3, mx.BOTH, cols=[0, 1, 127, 128, 7000, 14335])


def test_fused_column_wise_copy_feeds_a_reduction_over_m():
    # Y = X W^T with its column-wise copy quantized in the epilogue; Y^T's codes then serve as the
    # A operand of a product reducing over M (the wgrad pattern)
    M, N, K, P = 256, 512, 256, 256
    qa, sa, qb, sb = operands(M, N, K, 23)
    _, _, qT, sT = check_fused_ex(qa, sa, qb, sb, M, N, K, orc.E4M3, mx.COLWISE)
    rng = np.random.default_rng(24)
    q2 = rng.integers(0, 0x7E, (P, M), dtype=np.uint8)
    s2 = rng.integers(120, 134, (P, M // 32), dtype=np.uint8)
    z = mx.mx_gemm(qT, sT, mx.E4M3, dev(q2), dev(plain_to_chunked(s2)), mx.E4M3, N, P, M, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, _ = orc.mx_gemm(qa, sa, orc.E4M3, qb, sb, orc.E4M3)
    oqT, osT = orc.mx_quantize_rowwise_f32(np.ascontiguousarray(ref.astype(np.float32).T), orc.E4M3)
    zr, ab = orc.mx_gemm(oqT, osT, orc.E4M3, q2, s2, orc.E4M3)
    assert_close(z.cpu().numpy(), zr, ab, what="product of the column-wise copy")


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (512, 768, 1024)])
def test_fused_quantization_equals_quantized_fp32_results(fmt, M, N, K):
    qa, sa, qb, sb = operands(M, N, K, M + N + K + fmt)
    check_fused(qa, sa, qb, sb, M, N, K, fmt)


def test_fused_quantization_inf_results():
    M, N, K = 256, 256, 128
    qa, sa, qb, sb = operands(M, N, K, 9)
    qa[5, :] = 0x7E
    sa[5, :] = 254                      # 448 * 2^127 in every element of row 5 -> Inf products
    qb[:, :] = 0x7E
    q, s, _, _ = check_fused(qa, sa, qb, sb, M, N, K, orc.E4M3)
    assert (chunked_to_plain(s.cpu().numpy(), M, N // 32)[5] == 0xFF).all()


def test_fused_full_size_fprop():
    # the fprop shape of the linear-layer workload, exact-sum operands, sampled rows
    M, N, K = 8192, 14336, 4096
    qa, sa, qb, sb = operands(M, N, K, 31)
    check_fused(qa, sa, qb, sb, M, N, K, orc.E4M3, rows=[0, 1, 255, 256, 4097, 8191])


def test_fused_output_feeds_the_next_product():
    # Y = X W1^T quantized in the epilogue, then Z = Y W2^T reading Y's codes and scales as A
    M, N1, N2, K = 256, 512, 256, 256
    qa, sa, qb, sb = operands(M, N1, K, 21)
    q, s, oq, osc = check_fused(qa, sa, qb, sb, M, N1, K, orc.E4M3)
    rng = np.random.default_rng(22)
    q2 = rng.integers(0, 0x7E, (N2, N1), dtype=np.uint8)
    s2 = rng.integers(120, 134, (N2, N1 // 32), dtype=np.uint8)
    z = mx.mx_gemm(q, s, mx.E4M3, dev(q2), dev(plain_to_chunked(s2)), mx.E4M3, M, N2, N1, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(oq, osc, orc.E4M3, q2, s2, orc.E4M3)   # the oracle's codes (equal, checked above)
    assert_close(z.cpu().numpy(), ref, ab, what="chained product")
