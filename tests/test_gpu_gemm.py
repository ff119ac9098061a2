"""GPU parity of the block-scaled GEMMs against the double-precision CPU oracle.

Bar (per output element, on the decoded operands): |y - y_ref| <= 1e-5 * sum_k |a_k b_k| for
FP32 output; bf16 output adds one bf16 ulp of |y_ref| for the final rounding.  Cases: the
512^3 MXFP8 workload in full, tiny-K brute force with codes over the whole finite range,
one-hot scale probes (confirm the scale layout the tensor core reads by behaviour), mixed
E5M2 x E4M3, the 8192x4096x14336 fprop / dgrad / wgrad trio, NVFP4 (the scale-outside-the-sum
identity, 8192^3) and the DeepSeek GEMM with promotion (4096x7168x2048; error independent of K) at
full size on one row of every 128-row tile (all columns), and a 4096x2560 output (more tiles than
CTA pairs) in full for all three products.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests import quantized
from tests.layouts import chunked_to_plain, plain_to_chunked

pytestmark = pytest.mark.gpu

REL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def bf16_ulp(y):
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def assert_close(got, ref, absum, bf16=False, what=""):
    got = np.asarray(got, dtype=np.float64)
    tol = REL * absum + (bf16_ulp(ref) if bf16 else 0.0) + 1e-35
    err = np.abs(got - ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of tolerance, first {bad[:3].tolist()}: "
                           f"got {got[tuple(bad[0])]} ref {ref[tuple(bad[0])]} tol {tol[tuple(bad[0])]}")
    return float((err / np.maximum(absum, 1e-300)).max())


def to_dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def tile_rows(M, salt=0):
    """One output row from every 128-row M tile (all N columns are checked): row
    t * 128 + (37 t + 5 + salt) % 128 of tile t.  Consecutive tiles take rows of different TMEM lane
    quarters, and each 256-row CTA-pair tile has one row in each of its two CTAs, so every tile the
    persistent scheduler hands out -- first or later tile of a CTA -- is compared somewhere."""
    return np.array([t * 128 + (37 * t + 5 + salt) % 128 for t in range(M // 128)], dtype=np.int64)


# ------------------------------------------------------------------ MXFP8
def run_mx(qa, sa, ea, qb, sb, eb, M, N, K, out_dtype):
    """qa/qb plain codes, sa/sb plain scales (numpy) -> GPU result (numpy)."""
    y = mx.mx_gemm(to_dev_u8(qa), to_dev_u8(plain_to_chunked(sa)), ea, to_dev_u8(qb), to_dev_u8(plain_to_chunked(sb)),
                   eb, M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    return y.float().cpu().numpy()


def random_codes(rng, shape, fmt):
    q = rng.integers(0, 256, shape, dtype=np.uint8)
    if fmt == orc.E4M3:
        q[(q & 0x7F) == 0x7F] = 0x7E          # no NaN
    else:
        q[(q & 0x7C) == 0x7C] = 0x7B          # no Inf / NaN
    return q


@pytest.mark.parametrize("M", [128, 256])      # 128: single-CTA kernel; 256: CTA-pair kernel
@pytest.mark.parametrize("K", [128, 256])
@pytest.mark.parametrize("fa,fb", [(orc.E4M3, orc.E4M3), (orc.E5M2, orc.E4M3), (orc.E4M3, orc.E5M2), (orc.E5M2, orc.E5M2)])
def test_mx_gemm_tiny_bruteforce(M, K, fa, fb):
    rng = np.random.default_rng(K + 10 * fa + 100 * fb + M)
    N = 256
    qa, qb = random_codes(rng, (M, K), fa), random_codes(rng, (N, K), fb)
    sa = rng.integers(110, 145, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(110, 145, (N, K // 32), dtype=np.uint8)
    ref, ab = orc.mx_gemm(qa, sa, fa, qb, sb, fb)
    y = run_mx(qa, sa, fa, qb, sb, fb, M, N, K, mx.OUT_F32)
    assert_close(y, ref, ab, what="tiny")


def test_mx_gemm_same_addresses_other_shapes():
    # The library remembers encoded TMA tensor maps keyed by every encoding argument.  The same
    # device buffers are used here with other row counts, other K (so other row strides) and
    # other contents in turn; every call must match the oracle, as it would if each call encoded
    # its maps afresh.
    rng = np.random.default_rng(4242)
    qa_buf = torch.empty(512 * 512, dtype=torch.uint8, device="cuda")
    qb_buf = torch.empty(512 * 512, dtype=torch.uint8, device="cuda")
    sa_buf = torch.empty(mx.mx_scale_bytes(512, 512), dtype=torch.uint8, device="cuda")
    sb_buf = torch.empty(mx.mx_scale_bytes(512, 512), dtype=torch.uint8, device="cuda")
    y_buf = torch.empty(512 * 512, dtype=torch.float32, device="cuda")
    for (M, N, K) in [(256, 256, 256), (512, 256, 256), (256, 512, 512), (256, 256, 256), (512, 512, 128),
                      (128, 256, 512)]:
        qa, qb = random_codes(rng, (M, K), orc.E4M3), random_codes(rng, (N, K), orc.E4M3)
        sa = rng.integers(115, 140, (M, K // 32), dtype=np.uint8)
        sb = rng.integers(115, 140, (N, K // 32), dtype=np.uint8)
        csa, csb = plain_to_chunked(sa), plain_to_chunked(sb)
        qa_buf[: M * K].copy_(torch.from_numpy(qa.reshape(-1)))
        qb_buf[: N * K].copy_(torch.from_numpy(qb.reshape(-1)))
        sa_buf[: csa.size].copy_(torch.from_numpy(csa.reshape(-1)))
        sb_buf[: csb.size].copy_(torch.from_numpy(csb.reshape(-1)))
        y = mx.mx_gemm(qa_buf, sa_buf, mx.E4M3, qb_buf, sb_buf, mx.E4M3, M, N, K, out_dtype=mx.OUT_F32,
                       out=y_buf[: M * N].view(M, N))
        assert mx.mx_check() == mx.MX_OK
        ref, ab = orc.mx_gemm(qa, sa, orc.E4M3, qb, sb, orc.E4M3)
        assert_close(y.cpu().numpy(), ref, ab, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("N", [128, 256])       # 256 with M = 256: CTA-pair kernel
def test_mx_gemm_one_hot_scale_probe(N):
    # all scales 2^0 except one (row r, k-block b) = 2^1: exactly the outputs of row r (or column
    # r for B) change, by that block's partial sum -- confirms the scale layout by behaviour
    rng = np.random.default_rng(N)
    M, K = 256, 256
    qa = rng.integers(0x30, 0x50, (M, K), dtype=np.uint8)
    qb = rng.integers(0x30, 0x50, (N, K), dtype=np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    y0 = run_mx(qa, sa, 0, qb, sb, 0, M, N, K, mx.OUT_F32)
    for (r, b) in [(0, 0), (37, 3), (131, 7), (255, 5)]:
        sa2 = sa.copy()
        sa2[r, b] = 128
        y1 = run_mx(qa, sa2, 0, qb, sb, 0, M, N, K, mx.OUT_F32)
        d = y1 - y0
        changed = np.unique(np.argwhere(d != 0)[:, 0])
        assert changed.tolist() == [r], (r, b, changed[:10])
        ref, _ = orc.mx_gemm(qa, sa2, 0, qb, sb, 0, rows=[r])
        ref0, _ = orc.mx_gemm(qa, sa, 0, qb, sb, 0, rows=[r])
        assert np.allclose(d[r], (ref - ref0)[0], rtol=1e-6, atol=1e-6)
    for (c, b) in [(0, 0), (77, 2), (N - 1, 7), (N // 2, 1), (N // 2 - 1, 6)]:
        sb2 = sb.copy()
        sb2[c, b] = 128
        y1 = run_mx(qa, sa, 0, qb, sb2, 0, M, N, K, mx.OUT_F32)
        changed = np.unique(np.argwhere(y1 - y0 != 0)[:, 1])
        assert changed.tolist() == [c], (c, b, changed[:10])


@pytest.mark.parametrize("M", [128, 256])
def test_mx_gemm_one_hot_operand_probe(M):
    # a single nonzero code in A and B: the product lands in exactly one output
    N, K = 256, 256
    qa = np.zeros((M, K), np.uint8)
    qb = np.zeros((N, K), np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    for (m, n, k) in [(0, 0, 0), (5, 200, 77), (M - 1, 255, 255), (64, 129, 130), (M // 2 + 3, 127, 31),
                      (M - 40, 128, 128)]:
        qa[:] = 0
        qb[:] = 0
        qa[m, k] = 0x38   # 1.0
        qb[n, k] = 0x40   # 2.0
        y = run_mx(qa, sa, 0, qb, sb, 0, M, N, K, mx.OUT_F32)
        nz = np.argwhere(y != 0)
        assert nz.tolist() == [[m, n]] and y[m, n] == 2.0, (m, n, k, nz[:5])


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_mx_gemm_512_workload(out_dtype):
    a, b = synthetic.mxfp8_gemm_512()
    qa, sa, oqa, osa = quantized.mx_rowwise(a, orc.E4M3)
    qb, sb, oqb, osb = quantized.mx_rowwise(b, orc.E4M3)
    y = mx.mx_gemm(qa, sa, mx.E4M3, qb, sb, mx.E4M3, 512, 512, 512, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(oqa, osa, orc.E4M3, oqb, osb, orc.E4M3)
    assert_close(y.float().cpu().numpy(), ref, ab, bf16=out_dtype == mx.OUT_BF16, what="512^3")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 512), (384, 640, 1024), (1152, 256, 2048),
                                   (256, 256, 128), (768, 1024, 640), (2560, 512, 384)])
def test_mx_gemm_shapes(M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    a = (torch.randn(M, K, generator=g) * 3).to(torch.bfloat16)
    b = torch.randn(N, K, generator=g).to(torch.bfloat16)
    qa, sa, oqa, osa = quantized.mx_rowwise(a, orc.E5M2)
    qb, sb, oqb, osb = quantized.mx_rowwise(b, orc.E4M3)
    y = mx.mx_gemm(qa, sa, mx.E5M2, qb, sb, mx.E4M3, M, N, K, out_dtype=mx.OUT_F32)
    ref, ab = orc.mx_gemm(oqa, osa, orc.E5M2, oqb, osb, orc.E4M3)
    assert_close(y.cpu().numpy(), ref, ab, what=f"{M}x{N}x{K}")


def test_mx_gemm_strided_output():
    M, N, K = 256, 256, 256
    g = torch.Generator().manual_seed(3)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    b = torch.randn(N, K, generator=g).to(torch.bfloat16)
    qa, sa, oqa, osa = quantized.mx_rowwise(a, orc.E4M3)
    qb, sb, oqb, osb = quantized.mx_rowwise(b, orc.E4M3)
    big = torch.full((M, N + 64), 7.0, dtype=torch.float32, device="cuda")
    st = mx.load().mx_gemm(qa.data_ptr(), sa.data_ptr(), 0, qb.data_ptr(), sb.data_ptr(), 0, M, N, K,
                           big.data_ptr(), mx.OUT_F32, N + 64, torch.cuda.current_stream().cuda_stream)
    assert st == mx.MX_OK and mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(oqa, osa, 0, oqb, osb, 0)
    assert_close(big[:, :N].cpu().numpy(), ref, ab)
    assert (big[:, N:] == 7.0).all()


@pytest.fixture(scope="module")
def linear_layer():
    # each entry: (device q_row, s_row, q_col, s_col), (oracle codes / plain scales, same order)
    x, w, g = synthetic.mxfp8_linear()
    return quantized.mx_both(x, orc.E4M3), quantized.mx_both(w, orc.E4M3), quantized.mx_both(g, orc.E5M2)


@pytest.mark.parametrize("which", ["fprop", "dgrad", "wgrad"])
def test_mx_linear_layer_full_size(linear_layer, which):
    (Xd, Xo), (Wd, Wo), (Gd, Go) = linear_layer
    M_, K_, N_ = 8192, 4096, 14336
    if which == "fprop":      # Y[M,N] = X W^T
        a, b, ea, eb, M, N, K = (0, 1), (0, 1), 0, 0, M_, N_, K_
        (A, Ao), (B, Bo) = (Xd, Xo), (Wd, Wo)
    elif which == "dgrad":    # dX[M,K] = G W : A = G row-wise, B = W column-wise
        a, b, ea, eb, M, N, K = (0, 1), (2, 3), 1, 0, M_, K_, N_
        (A, Ao), (B, Bo) = (Gd, Go), (Wd, Wo)
    else:                     # dW[N,K] = G^T X : A = G column-wise, B = X column-wise
        a, b, ea, eb, M, N, K = (2, 3), (2, 3), 1, 0, N_, K_, M_
        (A, Ao), (B, Bo) = (Gd, Go), (Xd, Xo)
    y = mx.mx_gemm(A[a[0]], A[a[1]], ea, B[b[0]], B[b[1]], eb, M, N, K, out_dtype=mx.OUT_BF16)
    assert mx.mx_check() == mx.MX_OK
    rows = tile_rows(M)
    ref, ab = orc.mx_gemm(Ao[a[0]], Ao[a[1]], ea, Bo[b[0]], Bo[b[1]], eb, rows=rows)
    got = y[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert_close(got, ref, ab, bf16=True, what=which)


# ------------------------------------------------------------------ more tiles than CTA pairs, in full
# 4096 x 2560: 160 pair tiles of 256 x 256 for the persistent grid of CTA pairs (76 on 152 SMs),
# so most CTAs take a second or third tile and the accumulator / stage phases wrap across tiles;
# every output element is compared with the oracle.
MID = (4096, 2560)


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_mx_gemm_more_tiles_than_pairs_in_full(out_dtype):
    M, N = MID
    K = 256
    a = synthetic.normal(M, K, 1.0, 8100)
    b = synthetic.normal(N, K, 0.02, 8101)
    qa, sa, oqa, osa = quantized.mx_rowwise(a, orc.E4M3)
    qb, sb, oqb, osb = quantized.mx_rowwise(b, orc.E4M3)
    y = mx.mx_gemm(qa, sa, mx.E4M3, qb, sb, mx.E4M3, M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(oqa, osa, orc.E4M3, oqb, osb, orc.E4M3)
    assert_close(y.float().cpu().numpy(), ref, ab, bf16=out_dtype == mx.OUT_BF16, what="mx 4096x2560x256")


def test_nvfp4_gemm_more_tiles_than_pairs_in_full():
    M, N = MID
    K = 256
    a = synthetic.with_sparse_outliers(M, K, 8200)
    b = synthetic.with_sparse_outliers(N, K, 8201)
    qa, sa, ga, oqa, osa, oga = quantized.nv(a)
    qb, sb, gb, oqb, osb, ogb = quantized.nv(b)
    y = mx.nvfp4_gemm(qa, sa, ga, qb, sb, gb, M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.nv_gemm(oqa, osa, oga, oqb, osb, ogb)
    assert_close(y.cpu().numpy(), ref, ab, what="nvfp4 4096x2560x256")


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_deepseek_gemm_more_tiles_than_pairs_in_full(out_dtype):
    M, N = MID
    K = 256
    a = synthetic.normal(M, K, 1.0, 8300)
    b = synthetic.normal(N, K, 0.02, 8301)
    y, qa, sa, qb, sb = ds_run(a, b, out_dtype=out_dtype)
    ref, ab = orc.ds_gemm(qa, sa, qb, sb)
    assert_close(y.float().cpu().numpy(), ref, ab, bf16=out_dtype == mx.OUT_BF16, what="deepseek 4096x2560x256")


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_scale_outside_sum_identity():
    # q = [1, 1.5, 0.5, 2], p = [2, 1, 1.5, 0.5], s = 3 -> 15.75 (one 16-block, zero padded)
    M, N, K = 128, 128, 256
    enc = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4}
    ca = np.zeros((M, K), np.uint8)
    cb = np.zeros((N, K), np.uint8)
    ca[7, 16:20] = [enc[v] for v in (1, 1.5, 0.5, 2)]
    cb[9, 16:20] = [enc[v] for v in (2, 1, 1.5, 0.5)]
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    sa = np.full((M, K // 16), 0x38, np.uint8)   # 1.0
    sb = np.full((N, K // 16), 0x38, np.uint8)
    sa[7, 1] = 0x44                              # 3.0 for the block holding q
    ga = torch.ones(1, device="cuda")
    gb = torch.ones(1, device="cuda")
    y = mx.nvfp4_gemm(to_dev_u8(pack(ca)), to_dev_u8(plain_to_chunked(sa)), ga, to_dev_u8(pack(cb)),
                      to_dev_u8(plain_to_chunked(sb)), gb, M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    yn = y.cpu().numpy()
    assert yn[7, 9] == 15.75
    yn[7, 9] = 0
    assert not yn.any()
    gb.fill_(0.5)
    y2 = mx.nvfp4_gemm(to_dev_u8(pack(ca)), to_dev_u8(plain_to_chunked(sa)), ga, to_dev_u8(pack(cb)),
                       to_dev_u8(plain_to_chunked(sb)), gb, M, N, K, out_dtype=mx.OUT_F32)
    assert y2[7, 9].item() == 7.875


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (512, 256, 2048), (256, 256, 256),
                                   (768, 512, 1024)])
def test_nvfp4_gemm_random(M, N, K):
    a = synthetic.with_sparse_outliers(M, K, 4000 + M)
    b = synthetic.with_sparse_outliers(N, K, 4001 + N)
    qa, sa, ga, oqa, osa, oga = quantized.nv(a)
    qb, sb, gb, oqb, osb, ogb = quantized.nv(b)
    y = mx.nvfp4_gemm(qa, sa, ga, qb, sb, gb, M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.nv_gemm(oqa, osa, oga, oqb, osb, ogb)
    assert_close(y.cpu().numpy(), ref, ab, what="nvfp4")


def test_nvfp4_gemm_full_size():
    a, b = synthetic.nvfp4_pair()
    qa, sa, ga, oqa, osa, oga = quantized.nv(a)
    qb, sb, gb, oqb, osb, ogb = quantized.nv(b)
    M = N = K = 8192
    y = mx.nvfp4_gemm(qa, sa, ga, qb, sb, gb, M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    rows = tile_rows(M)
    ref, ab = orc.nv_gemm(oqa, osa, oga, oqb, osb, ogb, rows=rows)
    assert_close(y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, ab, what="nvfp4 8192^3")


# ------------------------------------------------------------------ DeepSeek
def ds_run(a, b, out_dtype=mx.OUT_F32):
    """GPU quantize (checked against the oracle) + GPU GEMM; returns the GPU result and the
    oracle's codes and scales for the reference product."""
    M, K = a.shape
    N = b.shape[0]
    qa, sa, oqa, osa = quantized.ds(a, 1)
    qb, sb, oqb, osb = quantized.ds(b, 128)
    y = mx.fp8_blockwise_gemm(qa, sa, qb, sb, M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    return y, oqa, osa, oqb, osb


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 512), (384, 256, 1024)])
def test_deepseek_gemm_small(M, N, K):
    a = synthetic.normal(M, K, 1.0, 5000 + K)
    b = synthetic.normal(N, K, 0.02, 5001 + K)
    y, qa, sa, qb, sb = ds_run(a, b)
    ref, ab = orc.ds_gemm(qa, sa, qb, sb)
    assert_close(y.cpu().numpy(), ref, ab, what="deepseek")


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (512, 768, 1024), (768, 512, 256)])
@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_deepseek_gemm_more_shapes(M, N, K, out_dtype):
    # several tiles in both directions, a single k-block (K = 128) and an odd k-block count
    a = synthetic.normal(M, K, 1.0, 5100 + K)
    b = synthetic.normal(N, K, 0.02, 5101 + K)
    y, qa, sa, qb, sb = ds_run(a, b, out_dtype=out_dtype)
    ref, ab = orc.ds_gemm(qa, sa, qb, sb)
    assert_close(y.float().cpu().numpy(), ref, ab, bf16=out_dtype == mx.OUT_BF16, what="deepseek shapes")


def test_deepseek_gemm_scale_per_block():
    # magnitudes that differ per row, per 128-column block of B and per k-block, so a scale taken
    # from the wrong row, N-block or k-block (or applied to the wrong TMEM buffer) shows
    M, N, K = 512, 512, 768
    a = synthetic.normal(M, K, 1.0, 5200)
    b = synthetic.normal(N, K, 1.0, 5201)
    ra = 2.0 ** (torch.arange(M) % 9 - 4).float()
    ka = 2.0 ** (torch.arange(K) // 128 * 3 - 6).float()
    nb_ = 2.0 ** (torch.arange(N) // 128 * 2 - 3).float()
    kb = 2.0 ** (5 - torch.arange(K) // 128 * 2).float()
    a = (a.float() * ra[:, None] * ka[None, :]).to(torch.bfloat16)
    b = (b.float() * nb_[:, None] * kb[None, :]).to(torch.bfloat16)
    y, qa, sa, qb, sb = ds_run(a, b)
    ref, ab = orc.ds_gemm(qa, sa, qb, sb)
    assert_close(y.cpu().numpy(), ref, ab, what="deepseek scales")


def test_deepseek_gemm_more_tiles_than_sms():
    # 1024 tiles of 128 x 128: every CTA runs several tiles, the buffers' phases wrap many times
    M, N, K = 4096, 4096, 384
    a = synthetic.normal(M, K, 1.0, 5300)
    b = synthetic.normal(N, K, 0.05, 5301)
    y, qa, sa, qb, sb = ds_run(a, b)
    rows = np.array([0, 255, 256, 1031, 2048, 3333, 4095])
    ref, ab = orc.ds_gemm(qa, sa, qb, sb, rows=rows)
    assert_close(y[torch.from_numpy(rows).cuda()].cpu().numpy(), ref, ab, what="deepseek tiles")


def test_deepseek_gemm_full_size():
    a, b = synthetic.deepseek_pair()
    M, K = a.shape
    N = b.shape[0]
    y, qa, sa, qb, sb = ds_run(a, b, out_dtype=mx.OUT_BF16)
    rows = tile_rows(M)
    ref, ab = orc.ds_gemm(qa, sa, qb, sb, rows=rows)
    assert_close(y[torch.from_numpy(rows).cuda()].float().cpu().numpy(), ref, ab, bf16=True, what="deepseek full")


def test_deepseek_error_does_not_grow_with_k():
    # random K = 1024 .. 7168 products: the worst relative error against the double-precision
    # oracle stays within the bound at every K (promotion every 128 keeps accumulation in FP32)
    worst = []
    for K in (1024, 4096, 7168):
        a = synthetic.normal(128, K, 1.0, 7000 + K)
        b = synthetic.normal(128, K, 1.0, 7001 + K)
        y, qa, sa, qb, sb = ds_run(a, b)
        ref, ab = orc.ds_gemm(qa, sa, qb, sb)
        worst.append(assert_close(y.cpu().numpy(), ref, ab, what=f"K={K}"))
    assert max(worst) <= REL
