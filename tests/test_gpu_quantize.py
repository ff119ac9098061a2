"""GPU parity of the quantizers against the CPU oracle: codes and scales must match bit for bit.

Covers an exhaustive sweep of every finite bf16 value against every reachable MX scale exponent
(both element formats, row-wise and column-wise), the full 16384x4096 outlier-channel workload,
edge blocks (zeros, signed zeros, bf16 subnormals, NaN/Inf, maxima landing in (MAX, 2^(emax+1))),
the DeepSeek 1x128 / 128x128 quantizers at 4096x7168 / 2048x7168, and NVFP4 at 8192x8192.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests.layouts import chunked_to_plain, plain_to_chunked

pytestmark = pytest.mark.gpu

EMAX = {orc.E4M3: 8, orc.E5M2: 15, orc.E2M1: 2}
MXFMT = {orc.E4M3: mx.E4M3, orc.E5M2: mx.E5M2}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def bits_to_bf16(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def check_mx(x, fmt, layouts=(mx.BOTH, mx.ROWWISE, mx.COLWISE)):
    rows, cols = x.shape
    xd = x.cuda()
    oq, osc = orc.mx_quantize_rowwise(x, fmt)
    oqT, osT = orc.mx_quantize_colwise(x, fmt)
    for layout in layouts:
        qr, sr, qc, sc = mx.mx_quantize(xd, elem=MXFMT[fmt], layout=layout)
        if layout & mx.ROWWISE:
            q = qr.cpu().numpy()
            s = chunked_to_plain(sr.cpu().numpy(), rows, cols // 32)
            bad = np.argwhere(q != oq)
            assert bad.size == 0, f"row codes differ at {bad[:5].tolist()}: gpu {q[tuple(bad[0])]:#x} oracle {oq[tuple(bad[0])]:#x}"
            assert np.array_equal(s, osc), "row scales differ"
        if layout & mx.COLWISE:
            q = qc.cpu().numpy()
            s = chunked_to_plain(sc.cpu().numpy(), cols, rows // 32)
            bad = np.argwhere(q != oqT)
            assert bad.size == 0, f"col codes differ at {bad[:5].tolist()}"
            assert np.array_equal(s, osT), "col scales differ"
    assert mx.mx_check() == mx.MX_OK


def exhaustive_matrix(fmt, cols=4096):
    """Rows of 32-blocks: each block = one anchor fixing the scale exponent k plus 31 test values
    with |x| <= anchor.  Every finite bf16 value is tested against every k it can meet."""
    emax = EMAX[fmt]
    allb = np.arange(65536, dtype=np.uint32)
    finite = allb[((allb >> 7) & 0xFF) != 0xFF]
    blocks = []
    for e in range(1, 255):                  # anchor exponent field; k = e - 127 - emax (clamped)
        anchor = (e << 7) | 0x7F              # largest bf16 of that binade
        vals = finite[(finite & 0x7FFF) <= anchor].astype(np.uint16)
        n = -(-len(vals) // 31)
        pad = n * 31 - len(vals)
        vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(n, 31)
        anc = np.full((n, 1), anchor, np.uint16)
        anc[1::2] |= 0x8000                   # both anchor signs
        blocks.append(np.concatenate([anc, vals], axis=1))
    blk = np.concatenate(blocks).reshape(-1)
    per_row = cols
    nrows = -(-len(blk) // per_row)
    nrows = -(-nrows // 128) * 128
    out = np.zeros(nrows * per_row, np.uint16)
    out[: len(blk)] = blk
    return bits_to_bf16(out.reshape(nrows, per_row))


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_mx_exhaustive_bf16_sweep_rowwise(fmt):
    x = exhaustive_matrix(fmt)
    check_mx(x, fmt, layouts=(mx.ROWWISE,))


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_mx_exhaustive_bf16_sweep_colwise(fmt):
    x = exhaustive_matrix(fmt, cols=2048).t().contiguous()   # the designed blocks run down columns
    check_mx(x, fmt, layouts=(mx.COLWISE, mx.BOTH))


@pytest.mark.parametrize("fmt", [orc.E4M3, orc.E5M2])
def test_mx_outlier_workload_full_size(fmt):
    x = synthetic.mxfp8_quantize()          # 16384 x 4096, 4 outlier channels 2^10 .. 2^14
    check_mx(x, fmt, layouts=(mx.BOTH,))


@pytest.mark.parametrize("layout", [mx.BOTH, mx.ROWWISE, mx.COLWISE])
def test_mx_dual_format_one_read_full_size(layout):
    # both element formats from one read: every output equals the single-format oracle result
    x = synthetic.mxfp8_quantize()          # 16384 x 4096
    x[7, 9] = float("nan")
    x[300, :32] = 0.0
    rows, cols = x.shape
    e4, e5 = mx.mx_quantize_dual(x.cuda(), layout=layout)
    assert mx.mx_check() == mx.MX_OK
    for fmt, out in ((orc.E4M3, e4), (orc.E5M2, e5)):
        if layout & mx.ROWWISE:
            oq, osc = orc.mx_quantize_rowwise(x, fmt)
            assert np.array_equal(out[0].cpu().numpy(), oq)
            assert np.array_equal(chunked_to_plain(out[1].cpu().numpy(), rows, cols // 32), osc)
        if layout & mx.COLWISE:
            oqT, osT = orc.mx_quantize_colwise(x, fmt)
            assert np.array_equal(out[2].cpu().numpy(), oqT)
            assert np.array_equal(chunked_to_plain(out[3].cpu().numpy(), cols, rows // 32), osT)


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 256), (1152, 640)])
def test_mx_small_and_ragged_tile_counts(shape):
    g = torch.Generator().manual_seed(shape[0] * 7 + shape[1])
    x = (torch.randn(*shape, generator=g) * torch.logspace(-20, 20, shape[1])).to(torch.bfloat16)
    for fmt in (orc.E4M3, orc.E5M2):
        check_mx(x, fmt)


def test_mx_edge_blocks():
    rows, cols = 128, 256
    x = torch.randn(rows, cols, generator=torch.Generator().manual_seed(1))
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, :32] = torch.tensor([3 * 2.0 ** -133, -(2.0 ** -133)] + [2.0 ** -130] * 30)   # bf16 subnormals
    x[3, 5] = float("nan")
    x[4, 40] = float("inf")
    x[5, 70] = float("-inf")
    x[6, :32] = 480.0                         # k = 0 -> 480 saturates to 448
    x[7, :32] = 1.0
    x[7, 0] = 2.0 ** 127                      # largest binade
    x[8, :32] = torch.linspace(-500, 500, 32)
    x[:32, 100] = float("nan")                # NaN down a column block
    xb = x.to(torch.bfloat16)
    for fmt in (orc.E4M3, orc.E5M2):
        check_mx(xb, fmt)


def test_mx_zero_matrix():
    x = torch.zeros(256, 256, dtype=torch.bfloat16)
    check_mx(x, orc.E4M3)


# ------------------------------------------------------------------ DeepSeek
@pytest.mark.parametrize("shape", [(128, 128), (256, 640), (4096, 7168)])
def test_deepseek_1x128(shape):
    x = synthetic.normal(*shape, 1.0, 5000)
    x[3, 17] = 12.5
    oq, osc = orc.ds_quantize_1x128(x)
    q, s, _, _ = mx.mx_quantize(x.cuda(), block=128, block_rows=1, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().T.view(np.uint32), osc.view(np.uint32))


@pytest.mark.parametrize("shape", [(128, 128), (384, 256), (2048, 7168)])
def test_deepseek_128x128(shape):
    x = synthetic.normal(*shape, 0.02, 5001)
    x[130 % shape[0], 7] = 3.0
    oq, osc = orc.ds_quantize_128x128(x)
    q, s, _, _ = mx.mx_quantize(x.cuda(), block=128, block_rows=128, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), osc.view(np.uint32))


def test_deepseek_edge_tiles():
    x = torch.randn(128, 256, generator=torch.Generator().manual_seed(2))
    x[0, :128] = 0.0
    x[1, :128] = 1e-3
    x[1, 0] = 1000.0                          # subnormal codes next to a large outlier
    x[2, :128] = 2.0 ** -130                  # bf16 subnormal tile
    xb = x.to(torch.bfloat16)
    oq, osc = orc.ds_quantize_1x128(xb)
    q, s, _, _ = mx.mx_quantize(xb.cuda(), block=128, block_rows=1, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().T.view(np.uint32), osc.view(np.uint32))


# ------------------------------------------------------------------ NVFP4
def check_nv(x):
    rows, cols = x.shape
    oq, osc, og = orc.nv_quantize(x)
    q, s, g = mx.nvfp4_quantize(x.cuda())
    assert np.float32(g.item()).view(np.uint32) == np.float32(og).view(np.uint32)
    qn = q.cpu().numpy()
    bad = np.argwhere(qn != oq)
    assert bad.size == 0, f"packed codes differ at {bad[:5].tolist()}"
    assert np.array_equal(chunked_to_plain(s.cpu().numpy(), rows, cols // 16), osc)
    assert mx.mx_check() == mx.MX_OK


@pytest.mark.parametrize("shape", [(128, 64), (128, 192), (256, 512), (8192, 8192)])
def test_nvfp4_quantize(shape):
    check_nv(synthetic.with_sparse_outliers(*shape, 4000))


def test_nvfp4_edges():
    x = torch.randn(128, 256, generator=torch.Generator().manual_seed(4))
    x[0, :16] = 0.0                          # zero block -> scale code 0, codes 0
    x[1, :16] = 1e-9                         # t rounds to 0 -> s_hat = 0 -> codes 0
    x[2, 0] = 300.0                          # the global amax
    x[3, :16] = -0.0
    x[4, :16] = torch.linspace(-7, 7, 16)
    check_nv(x.to(torch.bfloat16))
    check_nv(torch.zeros(128, 128, dtype=torch.bfloat16))


def test_nvfp4_exhaustive_element_grid():
    # every finite bf16 magnitude in [2^-8, 2^8] against a block scale set by an anchor of 6*s
    allb = np.arange(65536, dtype=np.uint32)
    mag = allb[((allb >> 7) & 0xFF) != 0xFF]
    vals = mag.astype(np.uint16)
    fv = bits_to_bf16(vals).float().abs()
    vals = vals[(fv >= 2.0 ** -8) & (fv <= 2.0 ** 8)]
    n = -(-len(vals) // 15)
    vals = np.concatenate([vals, np.zeros(n * 15 - len(vals), np.uint16)]).reshape(n, 15)
    anchor = np.full((n, 1), 0x4380, np.uint16)   # bf16 256.0
    blk = np.concatenate([anchor, vals], axis=1).reshape(-1)
    cols = 2048
    rows = -(-len(blk) // cols)
    rows = -(-rows // 128) * 128
    out = np.zeros(rows * cols, np.uint16)
    out[: len(blk)] = blk
    check_nv(bits_to_bf16(out.reshape(rows, cols)))


# ------------------------------------------------------------------ scale layout permutations
@pytest.mark.parametrize("rows,nblocks", [(128, 4), (384, 12), (256, 512), (16384, 128)])
def test_scale_layout_permutations_random_bytes(rows, nblocks):
    # the library's byte permutation against the test-side one, and swizzle o unswizzle = identity
    g = torch.Generator().manual_seed(rows * 7 + nblocks)
    plain = torch.randint(0, 256, (rows, nblocks), dtype=torch.uint8, generator=g)
    chunked = mx.mx_swizzle_scales(plain.cuda())
    assert np.array_equal(chunked.cpu().numpy(), plain_to_chunked(plain.numpy()))
    back = mx.mx_unswizzle_scales(chunked, rows, nblocks)
    assert torch.equal(back.cpu(), plain)
    assert mx.mx_check() == mx.MX_OK


def test_unswizzled_scales_match_the_oracle():
    # MX scales (K/32 blocks) and NVFP4 scales (K/16 blocks) of the quantizers, unswizzled on the
    # device, equal the oracle's plain per-block scales
    x = synthetic.with_sparse_outliers(256, 512, 4100)
    _, osc = orc.mx_quantize_rowwise(x, orc.E4M3)
    _, osT = orc.mx_quantize_colwise(x, orc.E4M3)
    _, sr, _, sc = mx.mx_quantize(x.cuda(), elem=mx.E4M3, layout=mx.BOTH)
    assert np.array_equal(mx.mx_unswizzle_scales(sr, 256, 512 // 32).cpu().numpy(), osc)
    assert np.array_equal(mx.mx_unswizzle_scales(sc, 512, 256 // 32).cpu().numpy(), osT)
    _, onv, _ = orc.nv_quantize(x)
    _, snv, _ = mx.nvfp4_quantize(x.cuda())
    assert np.array_equal(mx.mx_unswizzle_scales(snv, 256, 512 // 16).cpu().numpy(), onv)
    assert mx.mx_check() == mx.MX_OK
