"""Out-of-bounds write checks for every entry point (a stand-in for a memory checker, which this
GPU pool does not offer).

Every output buffer (codes, scales, global scales, workspaces, products) is placed between two
4 KB guard bands filled with a byte pattern; strided products also get padding columns between
their rows.  After each call the guards and the padding must still hold the pattern and mx_check
must report no device error.  Shapes are the small and ragged ones where tail handling lives: one
tile, a half-full last column tile (NVFP4 cols % 128 == 64), products whose M or N is not a
multiple of 256 (single-CTA kernels) next to ones that are (CTA pairs), grouped products with an
empty group.  Values are not compared here; the parity tests do that.
"""
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic

pytestmark = pytest.mark.gpu

FILL = 0xA5
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


class Guarded:
    """n bytes of device memory between two guard bands of FILL bytes."""

    def __init__(self, n):
        self.n = int(n)
        self.raw = torch.full((2 * GUARD + self.n,), FILL, dtype=torch.uint8, device="cuda")

    def t(self, dtype=torch.uint8, shape=None):
        v = self.raw[GUARD:GUARD + self.n]
        if dtype != torch.uint8:
            v = v.view(dtype)
        return v.view(*shape) if shape is not None else v

    def intact(self):
        return bool((self.raw[:GUARD] == FILL).all()) and bool((self.raw[GUARD + self.n:] == FILL).all())


def check(bufs, what):
    torch.cuda.synchronize()
    assert mx.mx_check() == mx.MX_OK, what
    bad = [i for i, b in enumerate(bufs) if not b.intact()]
    assert not bad, f"{what}: a guard band of output(s) {bad} was written"


def x_bf16(rows, cols, seed):
    return synthetic.with_sparse_outliers(rows, cols, seed).cuda()


# ------------------------------------------------------------------ quantizers
@pytest.mark.parametrize("elem", [mx.E4M3, mx.E5M2, mx.E2M1])
@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384), (384, 640)])
def test_mx_quantize_outputs_stay_in_bounds(elem, rows, cols):
    x = x_bf16(rows, cols, 100 + rows + cols)
    pb = 2 if elem == mx.E2M1 else 1
    b = [Guarded(rows * cols // pb), Guarded(mx.mx_scale_bytes(rows, cols)), Guarded(cols * rows // pb),
         Guarded(mx.mx_scale_bytes(cols, rows))]
    mx.mx_quantize(x, elem=elem, layout=mx.BOTH, q_row=b[0].t(shape=(rows, cols // pb)), s_row=b[1].t(),
                   q_col=b[2].t(shape=(cols, rows // pb)), s_col=b[3].t())
    check(b, f"mx_quantize elem {elem} {rows}x{cols}")


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384)])
def test_mx_quantize_2d_blocks_and_dual_stay_in_bounds(rows, cols):
    x = x_bf16(rows, cols, 200 + cols)
    b = [Guarded(rows * cols), Guarded(mx.mx_scale_bytes(rows, cols)), Guarded(rows * cols),
         Guarded(mx.mx_scale_bytes(cols, rows))]
    mx.mx_quantize(x, block_rows=32, layout=mx.BOTH, q_row=b[0].t(shape=(rows, cols)), s_row=b[1].t(),
                   q_col=b[2].t(shape=(cols, rows)), s_col=b[3].t())
    check(b, "2-D 32x32 blocks")
    d = [Guarded(rows * cols), Guarded(mx.mx_scale_bytes(rows, cols)), Guarded(rows * cols),
         Guarded(mx.mx_scale_bytes(cols, rows))]
    e = [Guarded(rows * cols), Guarded(mx.mx_scale_bytes(rows, cols)), Guarded(rows * cols),
         Guarded(mx.mx_scale_bytes(cols, rows))]
    shapes = [(rows, cols), None, (cols, rows), None]
    mx.mx_quantize_dual(x, layout=mx.BOTH, e4m3=tuple(g.t(shape=s) for g, s in zip(d, shapes)),
                        e5m2=tuple(g.t(shape=s) for g, s in zip(e, shapes)))
    check(d + e, "mx_quantize_dual")


@pytest.mark.parametrize("sfmt", [mx.SCALE_FP32, mx.SCALE_FP32_POW2])
@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384), (384, 256)])
def test_deepseek_quantize_stays_in_bounds(sfmt, rows, cols):
    x = x_bf16(rows, cols, 300 + rows)
    a = [Guarded(rows * cols), Guarded(4 * (cols // 128) * rows)]
    mx.mx_quantize(x, block=128, block_rows=1, sfmt=sfmt, layout=mx.ROWWISE, q_row=a[0].t(shape=(rows, cols)),
                   s_row=a[1].t(torch.float32, (cols // 128, rows)))
    check(a, f"1x128 {rows}x{cols}")
    w = [Guarded(rows * cols), Guarded(4 * (rows // 128) * (cols // 128))]
    mx.mx_quantize(x, block=128, block_rows=128, sfmt=sfmt, layout=mx.ROWWISE, q_row=w[0].t(shape=(rows, cols)),
                   s_row=w[1].t(torch.float32, (rows // 128, cols // 128)))
    check(w, f"128x128 {rows}x{cols}")
    if sfmt == mx.SCALE_FP32_POW2:
        for br, s in ((1, a[1]), (128, w[1])):
            o = Guarded(rows * cols // 32)
            mx.mx_scales_from_fp32_blocks(s.t(torch.float32), rows, cols, br, out=o.t())
            check([o], f"mx_scales_from_fp32_blocks block_rows {br}")


def nv_bufs(rows, cols, groups=1):
    return [Guarded(rows * cols // 2), Guarded(mx.mx_scale_bytes(rows, cols, 16, 1, mx.SCALE_UE4M3)),
            Guarded(4 * groups), Guarded(max(16, (4 * groups + 15) // 16 * 16))]


@pytest.mark.parametrize("rows,cols", [(128, 64), (256, 192), (384, 1024)])
def test_nvfp4_quantize_variants_stay_in_bounds(rows, cols):
    x = x_bf16(rows, cols, 400 + cols)
    b = nv_bufs(rows, cols)
    mx.nvfp4_quantize(x, q_packed=b[0].t(shape=(rows, cols // 2)), s_ue4m3=b[1].t(), gscale=b[2].t(torch.float32),
                      workspace=b[3].t())
    check(b, f"nvfp4_quantize {rows}x{cols}")
    rbits = torch.randint(0, 256, (rows, cols), dtype=torch.uint8, generator=torch.Generator().manual_seed(5)).cuda()
    for rht, rb in ((True, None), (False, rbits), (True, rbits)):
        b = nv_bufs(rows, cols)
        mx.nvfp4_quantize_ex(x, rht=rht, signs=0x5A3C, rbits=rb, q_packed=b[0].t(shape=(rows, cols // 2)),
                             s_ue4m3=b[1].t(), gscale=b[2].t(torch.float32), workspace=b[3].t())
        check(b, f"nvfp4_quantize_ex rht={rht} sr={rb is not None} {rows}x{cols}")
    lib = mx.load()
    b = nv_bufs(rows, cols)[:3]
    st = lib.nvfp4_quantize_noalloc(x.data_ptr(), rows, cols, b[0].t().data_ptr(), b[1].t().data_ptr(),
                                    b[2].t().data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == mx.MX_OK
    check(b, f"nvfp4_quantize_noalloc {rows}x{cols}")


def test_nvfp4_quantize_2d_and_grouped_stay_in_bounds():
    rows, cols = 256, 384
    x = x_bf16(rows, cols, 500)
    b = [Guarded(rows * cols // 2), Guarded(mx.mx_scale_bytes(rows, cols, 16, 1, mx.SCALE_UE4M3)),
         Guarded(rows * cols // 2), Guarded(mx.mx_scale_bytes(cols, rows, 16, 1, mx.SCALE_UE4M3)), Guarded(4),
         Guarded(16)]
    mx.nvfp4_quantize_2d(x, out=(b[0].t(shape=(rows, cols // 2)), b[1].t(), b[2].t(shape=(cols, rows // 2)),
                                 b[3].t()), gscale=b[4].t(torch.float32), workspace=b[5].t())
    check(b, "nvfp4_quantize_2d")
    rows, cols = 512, 192
    x = x_bf16(rows, cols, 501)
    off = torch.tensor([0, 128, 128, 384, 512], dtype=torch.int64, device="cuda")
    b = nv_bufs(rows, cols, groups=4)
    mx.nvfp4_quantize_grouped(x, off, q_packed=b[0].t(shape=(rows, cols // 2)), s_ue4m3=b[1].t(),
                              gscale=b[2].t(torch.float32), workspace=b[3].t())
    check(b, "nvfp4_quantize_grouped")


def test_scale_layout_helpers_stay_in_bounds():
    rows, nblocks = 256, 12
    plain = torch.randint(0, 256, (rows, nblocks), dtype=torch.uint8, generator=torch.Generator().manual_seed(6))
    g = Guarded(rows * nblocks)
    mx.mx_swizzle_scales(plain.cuda(), out=g.t())
    check([g], "mx_swizzle_scales")
    p = Guarded(rows * nblocks)
    mx.mx_unswizzle_scales(g.t(), rows, nblocks, out=p.t(shape=(rows, nblocks)))
    check([p], "mx_unswizzle_scales")
    assert torch.equal(p.t(shape=(rows, nblocks)).cpu(), plain)


# ------------------------------------------------------------------ products
PAD = 24  # padding columns after each output row (ldc = N + PAD, a multiple of 8)


def strided_out(M, N, out_dtype):
    es = 4 if out_dtype == mx.OUT_F32 else 2
    g = Guarded(M * (N + PAD) * es)
    full = g.t(torch.float32 if out_dtype == mx.OUT_F32 else torch.bfloat16, (M, N + PAD))
    return g, full, full[:, :N]


def pad_intact(full, N):
    bits = full[:, N:].contiguous().view(torch.uint8)
    return bool((bits == FILL).all())


def mx_operands(M, N, K, elem=mx.E4M3, seed=0):
    a = x_bf16(M, K, 600 + seed)
    b = x_bf16(N, K, 601 + seed)
    qa, sa, _, _ = mx.mx_quantize(a, elem=elem, layout=mx.ROWWISE)
    qb, sb, _, _ = mx.mx_quantize(b, elem=elem, layout=mx.ROWWISE)
    return qa, sa, qb, sb


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 256, 128), (384, 640, 256), (512, 512, 512)])
def test_mx_gemm_writes_only_its_rows(M, N, K, out_dtype):
    qa, sa, qb, sb = mx_operands(M, N, K, seed=M + N)
    g, full, y = strided_out(M, N, out_dtype)
    mx.mx_gemm(qa, sa, mx.E4M3, qb, sb, mx.E4M3, M, N, K, out_dtype=out_dtype, out=y)
    check([g], f"mx_gemm {M}x{N}x{K}")
    assert pad_intact(full, N), "padding columns written"


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 256, 512)])
def test_mxfp4_and_nvfp4_gemm_write_only_their_rows(M, N, K):
    qa, sa, qb, sb = mx_operands(M, N, K, elem=mx.E2M1, seed=7)
    g, full, y = strided_out(M, N, mx.OUT_F32)
    mx.mx_gemm(qa, sa, mx.E2M1, qb, sb, mx.E2M1, M, N, K, out_dtype=mx.OUT_F32, out=y)
    check([g], f"MXFP4 {M}x{N}x{K}")
    assert pad_intact(full, N)
    qa, sa, ga = mx.nvfp4_quantize(x_bf16(M, K, 700))
    qb, sb, gb = mx.nvfp4_quantize(x_bf16(N, K, 701))
    for od in (mx.OUT_F32, mx.OUT_BF16):
        g, full, y = strided_out(M, N, od)
        mx.nvfp4_gemm(qa, sa, ga, qb, sb, gb, M, N, K, out_dtype=od, out=y)
        check([g], f"nvfp4_gemm {M}x{N}x{K}")
        assert pad_intact(full, N)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 256, 256), (384, 512, 384)])
def test_deepseek_gemm_writes_only_its_rows(M, N, K):
    qa, sa, _, _ = mx.mx_quantize(x_bf16(M, K, 800), block=128, block_rows=1, sfmt=mx.SCALE_FP32,
                                  layout=mx.ROWWISE)
    qb, sb, _, _ = mx.mx_quantize(x_bf16(N, K, 801), block=128, block_rows=128, sfmt=mx.SCALE_FP32,
                                  layout=mx.ROWWISE)
    for od in (mx.OUT_F32, mx.OUT_BF16):
        g, full, y = strided_out(M, N, od)
        mx.fp8_blockwise_gemm(qa, sa, qb, sb, M, N, K, out_dtype=od, out=y)
        check([g], f"fp8_blockwise_gemm {M}x{N}x{K}")
        assert pad_intact(full, N)


def test_grouped_gemms_write_only_their_rows():
    G, N, K = 3, 256, 256
    off = torch.tensor([0, 128, 128, 384], dtype=torch.int64, device="cuda")
    M = 384
    a = x_bf16(M, K, 900)
    w = x_bf16(G * N, K, 901)
    qa, sa, _, _ = mx.mx_quantize(a, layout=mx.ROWWISE)
    qw, sw, _, _ = mx.mx_quantize(w, layout=mx.ROWWISE)
    g, full, y = strided_out(M, N, mx.OUT_BF16)
    mx.mx_gemm_grouped(qa, sa, mx.E4M3, qw, sw, mx.E4M3, off, M, N, K, out_dtype=mx.OUT_BF16, out=y)
    check([g], "mx_gemm_grouped")
    assert pad_intact(full, N)
    qa4, sa4, ga4 = mx.nvfp4_quantize(a)
    qw4, sw4, gw4 = mx.nvfp4_quantize_grouped(w, torch.tensor([0, N, 2 * N, 3 * N], dtype=torch.int64,
                                                              device="cuda"))
    g, full, y = strided_out(M, N, mx.OUT_F32)
    mx.nvfp4_gemm_grouped(qa4, sa4, ga4, qw4, sw4, gw4, off, M, N, K, out_dtype=mx.OUT_F32, out=y)
    check([g], "nvfp4_gemm_grouped")
    assert pad_intact(full, N)
    qad, sad, _, _ = mx.mx_quantize(a, block=128, block_rows=1, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE)
    qwd, swd, _, _ = mx.mx_quantize(w, block=128, block_rows=128, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE)
    g, full, y = strided_out(M, N, mx.OUT_BF16)
    mx.fp8_blockwise_gemm_grouped(qad, sad, qwd, swd, off, M, N, K, out_dtype=mx.OUT_BF16, out=y)
    check([g], "fp8_blockwise_gemm_grouped")
    assert pad_intact(full, N)


@pytest.mark.parametrize("layout", [mx.ROWWISE, mx.COLWISE, mx.BOTH])
def test_gemm_with_mx_output_writes_only_its_buffers(layout):
    M, N, K = 256, 512, 128
    qa, sa, qb, sb = mx_operands(M, N, K, seed=11)
    b = [Guarded(M * N), Guarded(M * N // 32), Guarded(N * M), Guarded(M * N // 32)]
    row, col = bool(layout & mx.ROWWISE), bool(layout & mx.COLWISE)
    mx.mx_gemm_mxout_ex(qa, sa, mx.E4M3, qb, sb, mx.E4M3, M, N, K, layout=layout,
                        q_row=b[0].t(shape=(M, N)) if row else None, s_row=b[1].t() if row else None,
                        q_col=b[2].t(shape=(N, M)) if col else None, s_col=b[3].t() if col else None)
    check(b, f"mx_gemm_mxout_ex layout {layout}")
    if not row:
        assert bool((b[0].t() == FILL).all()) and bool((b[1].t() == FILL).all()), "row-wise copy written"
    if not col:
        assert bool((b[2].t() == FILL).all()) and bool((b[3].t() == FILL).all()), "column-wise copy written"
