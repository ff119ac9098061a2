"""GPU parity at the size limits: tensors of 2^31 elements and more (so that any 32-bit element
index or byte offset in a kernel would wrap), products with 2^31 outputs, and the quantizers'
widest input (65535 column tiles of 128).  Inputs are seeded synthetic bf16 blocks from the CPU
generators, replicated on the device and scaled per band by exact powers of two, so every band
differs; the oracle checks bands at both ends of each tensor (and, where a result depends on the
whole tensor, the planted global maximum is inside every checked band).
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

ROWS, COLS = 32768, 65536          # 2^31 elements, 4 GiB of bf16
BASE_ROWS = 1024


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def big_input(seed, plant=None):
    """[ROWS][COLS] bf16 on the device: a seeded 1024-row block repeated 32 times, band b scaled by
    2^(b % 5 - 2) (exact).  plant: value written at (5, 7) and (ROWS - 60, COLS - 500)."""
    base = synthetic.normal(BASE_ROWS, COLS, 1.0, seed).cuda()
    x = base.repeat(ROWS // BASE_ROWS, 1)
    del base
    for b in range(ROWS // BASE_ROWS):
        x[b * BASE_ROWS:(b + 1) * BASE_ROWS].mul_(2.0 ** (b % 5 - 2))
    if plant is not None:
        x[5, 7] = plant
        x[ROWS - 60, COLS - 500] = plant
    return x


def free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


BANDS = ((0, 128), (ROWS - 128, ROWS))          # row bands at both ends
CBANDS = ((0, 128), (COLS - 128, COLS))         # column bands at both ends


def test_mx_quantize_2g_elements_both_layouts():
    x = big_input(8100)
    q, s, qT, sT = mx.mx_quantize(x, elem=mx.E4M3, layout=mx.BOTH)
    assert mx.mx_check() == mx.MX_OK
    chunk_row = COLS * 4                          # scale bytes of one 128-row block (row-wise copy)
    for r0, r1 in BANDS:
        oq, osc = orc.mx_quantize_rowwise(x[r0:r1].cpu(), orc.E4M3)
        assert np.array_equal(q[r0:r1].cpu().numpy(), oq), (r0, "row codes")
        sl = s[(r0 // 128) * chunk_row:(r0 // 128 + 1) * chunk_row].cpu().numpy()
        assert np.array_equal(chunked_to_plain(sl, 128, COLS // 32), osc), (r0, "row scales")
    chunk_col = ROWS * 4
    for c0, c1 in CBANDS:
        oqT, osT = orc.mx_quantize_colwise(x[:, c0:c1].contiguous().cpu(), orc.E4M3)
        assert np.array_equal(qT[c0:c1].cpu().numpy(), oqT), (c0, "col codes")
        sl = sT[(c0 // 128) * chunk_col:(c0 // 128 + 1) * chunk_col].cpu().numpy()
        assert np.array_equal(chunked_to_plain(sl, 128, ROWS // 32), osT), (c0, "col scales")
    del x, q, s, qT, sT
    free()


def test_nvfp4_quantize_2g_elements():
    x = big_input(8200, plant=1000.0)             # the global maximum sits in both checked bands
    q, s, g = mx.nvfp4_quantize(x)
    assert mx.mx_check() == mx.MX_OK
    chunk_row = (COLS // 64) * 512
    for r0, r1 in ((0, 128), (ROWS - 128, ROWS)):
        oq, osc, og = orc.nv_quantize(x[r0:r1].cpu())
        assert np.float32(g.item()).view(np.uint32) == np.float32(og).view(np.uint32)
        assert np.array_equal(q[r0:r1].cpu().numpy(), oq), (r0, "codes")
        sl = s[(r0 // 128) * chunk_row:(r0 // 128 + 1) * chunk_row].cpu().numpy()
        assert np.array_equal(chunked_to_plain(sl, 128, COLS // 16), osc), (r0, "scales")
    del x, q, s
    free()


@pytest.mark.parametrize("block_rows", [1, 128])
def test_deepseek_quantize_2g_elements(block_rows):
    x = big_input(8300 + block_rows)
    q, s, _, _ = mx.mx_quantize(x, block=128, block_rows=block_rows, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE)
    assert mx.mx_check() == mx.MX_OK
    for r0, r1 in BANDS:
        xs = x[r0:r1].cpu()
        if block_rows == 1:
            oq, osc = orc.ds_quantize_1x128(xs)
            got_s = s[:, r0:r1].cpu().numpy().T
        else:
            oq, osc = orc.ds_quantize_128x128(xs)
            got_s = s[r0 // 128:r0 // 128 + 1].cpu().numpy()
        assert np.array_equal(q[r0:r1].cpu().numpy(), oq), (r0, "codes")
        assert np.array_equal(np.ascontiguousarray(got_s).view(np.uint32), osc.astype(np.float32).view(np.uint32))
    del x, q, s
    free()


def test_mx_quantize_widest_input():
    # 65535 tiles of 128 columns, the most a quantizer launch takes
    cols = 65535 * 128
    base = synthetic.normal(128, 65536, 1.0, 8400).cuda()
    x = base.repeat(1, 128)[:, :cols].contiguous()
    del base
    for t in range(0, cols // 65536 + 1):      # exact power-of-two scaling per 65536-column band
        x[:, t * 65536:(t + 1) * 65536].mul_(2.0 ** (t % 7 - 3))
    q, s, qT, sT = mx.mx_quantize(x, elem=mx.E5M2, layout=mx.BOTH)
    assert mx.mx_check() == mx.MX_OK
    for c0 in (0, cols - 4096):
        xs = x[:, c0:c0 + 4096].contiguous().cpu()
        oq, osc = orc.mx_quantize_rowwise(xs, orc.E5M2)
        assert np.array_equal(q[:, c0:c0 + 4096].cpu().numpy(), oq), (c0, "row codes")
        sl = s[(c0 // 128) * 512:(c0 // 128 + 32) * 512].cpu().numpy()
        assert np.array_equal(chunked_to_plain(sl, 128, 4096 // 32), osc), (c0, "row scales")
        oqT, osT = orc.mx_quantize_colwise(xs, orc.E5M2)
        assert np.array_equal(qT[c0:c0 + 4096].cpu().numpy(), oqT), (c0, "col codes")
        sl = sT[(c0 // 128) * 512:(c0 // 128 + 32) * 512].cpu().numpy()
        assert np.array_equal(chunked_to_plain(sl, 4096, 128 // 32), osT), (c0, "col scales")
    del x, q, s, qT, sT
    free()


GM, GN = 65536, 32768                          # 2^31 outputs, 4 GiB of bf16
GROWS = np.array([0, 1, 32767, 32768, 65535])


def test_mx_gemm_2g_outputs():
    K = 256
    rng = np.random.default_rng(8500)
    qa = rng.integers(0, 0x7E, (GM, K), dtype=np.uint8) | (rng.integers(0, 2, (GM, K), dtype=np.uint8) << 7)
    qb = rng.integers(0, 0x7E, (GN, K), dtype=np.uint8) | (rng.integers(0, 2, (GN, K), dtype=np.uint8) << 7)
    sa = rng.integers(118, 136, (GM, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 136, (GN, K // 32), dtype=np.uint8)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = mx.mx_gemm(dev(qa), dev(plain_to_chunked(sa)), mx.E4M3, dev(qb), dev(plain_to_chunked(sb)), mx.E4M3,
                   GM, GN, K, out_dtype=mx.OUT_BF16)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(qa, sa, orc.E4M3, qb, sb, orc.E4M3, rows=GROWS)
    assert_close(y[torch.from_numpy(GROWS).cuda()].float().cpu().numpy(), ref, ab, bf16=True, what="2^31 outputs")
    del y
    free()


def test_deepseek_gemm_2g_outputs():
    K = 256
    rng = np.random.default_rng(8600)
    qa = rng.integers(0, 0x7E, (GM, K), dtype=np.uint8) | (rng.integers(0, 2, (GM, K), dtype=np.uint8) << 7)
    qb = rng.integers(0, 0x7E, (GN, K), dtype=np.uint8) | (rng.integers(0, 2, (GN, K), dtype=np.uint8) << 7)
    sa = (rng.random((GM, K // 128)) * 0.01 + 0.001).astype(np.float32)       # [M][K/128]
    sb = (rng.random((GN // 128, K // 128)) * 0.01 + 0.001).astype(np.float32)
    y = mx.fp8_blockwise_gemm(torch.from_numpy(qa).cuda(), torch.from_numpy(np.ascontiguousarray(sa.T)).cuda(),
                              torch.from_numpy(qb).cuda(), torch.from_numpy(sb).cuda(), GM, GN, K,
                              out_dtype=mx.OUT_BF16)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.ds_gemm(qa, sa, qb, sb, rows=GROWS)
    assert_close(y[torch.from_numpy(GROWS).cuda()].float().cpu().numpy(), ref, ab, bf16=True, what="2^31 outputs")
    del y
    free()


def test_nvfp4_gemm_2g_outputs():
    K = 256
    rng = np.random.default_rng(8700)
    qa = rng.integers(0, 256, (GM, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (GN, K // 2), dtype=np.uint8)
    sa = rng.integers(0x20, 0x48, (GM, K // 16), dtype=np.uint8)
    sb = rng.integers(0x20, 0x48, (GN, K // 16), dtype=np.uint8)
    ga = torch.tensor([0.75], device="cuda")
    gb = torch.tensor([1.25], device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = mx.nvfp4_gemm(dev(qa), dev(plain_to_chunked(sa)), ga, dev(qb), dev(plain_to_chunked(sb)), gb, GM, GN, K,
                      out_dtype=mx.OUT_BF16)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.nv_gemm(qa, sa, 0.75, qb, sb, 1.25, rows=GROWS)
    assert_close(y[torch.from_numpy(GROWS).cuda()].float().cpu().numpy(), ref, ab, bf16=True, what="2^31 outputs")
    del y
    free()
