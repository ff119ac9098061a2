"""GPU parity of MXFP4 (E2M1 elements, one E8M0 scale per 32; "NVFP4: high accuracy with 4 bits"
(theluyuan.com), sec 5.5) against the CPU oracle.

Quantizer: codes and scales bit for bit, over every finite bf16 value against every reachable
scale exponent, row-wise and column-wise, plus edge blocks and several tile counts.  GEMM: the
oracle's double-precision product within |y - y_ref| <= 1e-5 * sum_k |a_k b_k| (+ one bf16 ulp
for bf16 output), on random codes and scales covering every byte position a stage's scale
chunks hold, on both kernels (CTA pairs for M, N multiples of 256, single CTA otherwise), and on
the 8192^3 workload through the quantizer on sampled rows.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests import quantized
from tests.layouts import chunked_to_plain, pack_fp4, plain_to_chunked, unpack_fp4
from tests.test_gpu_quantize import exhaustive_matrix
from tests.test_gpu_gemm import assert_close, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def check_mxfp4(x, layouts=(mx.BOTH, mx.ROWWISE, mx.COLWISE)):
    rows, cols = x.shape
    xd = x.cuda()
    oq, osc = orc.mx_quantize_rowwise(x, orc.E2M1)
    oqT, osT = orc.mx_quantize_colwise(x, orc.E2M1)
    for layout in layouts:
        qr, sr, qc, sc = mx.mx_quantize(xd, elem=mx.E2M1, layout=layout)
        if layout & mx.ROWWISE:
            assert qr.shape == (rows, cols // 2)
            q = unpack_fp4(qr.cpu().numpy())
            bad = np.argwhere(q != oq)
            assert bad.size == 0, f"row codes differ at {bad[:5].tolist()}: gpu {q[tuple(bad[0])]} oracle {oq[tuple(bad[0])]}"
            assert np.array_equal(chunked_to_plain(sr.cpu().numpy(), rows, cols // 32), osc), "row scales differ"
        if layout & mx.COLWISE:
            assert qc.shape == (cols, rows // 2)
            q = unpack_fp4(qc.cpu().numpy())
            bad = np.argwhere(q != oqT)
            assert bad.size == 0, f"col codes differ at {bad[:5].tolist()}"
            assert np.array_equal(chunked_to_plain(sc.cpu().numpy(), cols, rows // 32), osT), "col scales differ"
    assert mx.mx_check() == mx.MX_OK


def test_mxfp4_exhaustive_bf16_sweep_rowwise():
    check_mxfp4(exhaustive_matrix(orc.E2M1), layouts=(mx.ROWWISE,))


def test_mxfp4_exhaustive_bf16_sweep_colwise():
    check_mxfp4(exhaustive_matrix(orc.E2M1, cols=2048).t().contiguous(), layouts=(mx.COLWISE, mx.BOTH))


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 256), (1152, 640)])
def test_mxfp4_small_and_ragged_tile_counts(shape):
    g = torch.Generator().manual_seed(shape[0] * 5 + shape[1])
    x = (torch.randn(*shape, generator=g) * torch.logspace(-20, 20, shape[1])).to(torch.bfloat16)
    check_mxfp4(x)


def test_mxfp4_edge_blocks():
    x = torch.randn(128, 256, generator=torch.Generator().manual_seed(31))
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, :32] = torch.tensor([3 * 2.0 ** -133, -(2.0 ** -133)] + [2.0 ** -130] * 30)
    x[3, 5] = float("nan")
    x[4, 40] = float("inf")
    x[5, 70] = float("-inf")
    x[6, :32] = 7.5                        # k = 0, saturates to 6
    x[7, :32] = torch.tensor([6.0, 5.0, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25] * 4)   # ties -> even codes
    x[8, :32] = torch.linspace(-6, 6, 32)
    x[:32, 100] = float("nan")
    check_mxfp4(x.to(torch.bfloat16))


def test_mxfp4_full_size_workload():
    a, _ = synthetic.mxfp4_pair(M=8192, N=128, K=8192)
    check_mxfp4(a, layouts=(mx.BOTH,))


# ------------------------------------------------------------------ GEMM
def run_mxfp4(qa, sa, qb, sb, M, N, K, out_dtype):
    """qa/qb unpacked codes, sa/sb plain scales (numpy) -> GPU result (numpy)."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = mx.mx_gemm(dev(pack_fp4(qa)), dev(plain_to_chunked(sa)), mx.E2M1, dev(pack_fp4(qb)),
                   dev(plain_to_chunked(sb)), mx.E2M1, M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    return y.float().cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 256, 256), (128, 384, 512), (256, 512, 512),
                                   (384, 256, 768), (512, 768, 1024)])
@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_mxfp4_gemm_random_codes_and_scales(M, N, K, out_dtype):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    qa = rng.integers(0, 16, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 16, (N, K), dtype=np.uint8)
    sa = rng.integers(118, 137, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 137, (N, K // 32), dtype=np.uint8)
    y = run_mxfp4(qa, sa, qb, sb, M, N, K, out_dtype)
    ref, ab = orc.mx_gemm(qa, sa, orc.E2M1, qb, sb, orc.E2M1)
    assert_close(y, ref, ab, bf16=out_dtype == mx.OUT_BF16, what=f"mxfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N", [(128, 128), (256, 256)])   # single CTA, CTA pair
def test_mxfp4_gemm_one_hot_scale_per_block_position(M, N):
    # a stage holds 8 blocks of 32 per row (two 512-byte chunks, four bytes each): scale one block
    # at a time in A and in B and check that exactly the matching partial sum moves
    K = 256
    rng = np.random.default_rng(40 + M)
    qa = rng.integers(0, 16, (M, K), dtype=np.uint8)
    qb = rng.integers(0, 16, (N, K), dtype=np.uint8)
    base_a = np.full((M, K // 32), 127, np.uint8)
    base_b = np.full((N, K // 32), 127, np.uint8)
    for blk in range(K // 32):
        sa, sb = base_a.copy(), base_b.copy()
        sa[M - 3, blk] = 130                  # x8 on one block of one A row
        sb[5, (blk + 3) % 8] = 125            # /4 on another block of one B row
        y = run_mxfp4(qa, sa, qb, sb, M, N, K, mx.OUT_F32)
        ref, ab = orc.mx_gemm(qa, sa, orc.E2M1, qb, sb, orc.E2M1)
        assert_close(y, ref, ab, what=f"one-hot block {blk}")


def test_mxfp4_quantize_then_gemm_full_size():
    a, b = synthetic.mxfp4_pair()
    M = N = K = 8192
    qa, sa, oqa, osa = quantized.mx_rowwise(a, orc.E2M1)
    qb, sb, oqb, osb = quantized.mx_rowwise(b, orc.E2M1)
    y = mx.mx_gemm(qa, sa, mx.E2M1, qb, sb, mx.E2M1, M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    rows = tile_rows(M)
    ref, ab = orc.mx_gemm(oqa, osa, orc.E2M1, oqb, osb, orc.E2M1, rows=rows)
    assert_close(y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, ab, what="mxfp4 8192^3")
