"""GPU parity of the grouped MXFP8 GEMM (mixture-of-experts expert products in one launch; "MXFP8
on SM120: software support" (xuesongtap.github.io), sec 1.2) against the CPU oracle, group by
group: rows off[g] .. off[g+1] of A times the g-th [N][K] block of B, within |y - y_ref| <=
1e-5 * sum_k |a_k b_k| (+ one bf16 ulp for bf16 output).  Covers groups whose rows end in half
a 256-row tile, empty groups, one group equal to the plain GEMM, and offsets that break the
contract (no work, MX_ERR_INVALID_ARG from mx_check).  Also the NVFP4 experts: grouped NVFP4
quantization (each row group a tensor of its own: codes, scales and global scale bit-identical to
the oracle's quantization of that group's rows, "NVFP4: high accuracy with 4 bits"
(theluyuan.com), sec 5.4), and the grouped NVFP4 product with per-expert global scales; and the
DeepSeek FP8 expert products with FP32 promotion per 128 of K ("Why FP8 training is stable"
(magicnetworld.com), sec 6.3), each expert's 128x128 weight-block scales its own rows of sB.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
import oracle as orc
from tests.layouts import chunked_to_plain, pack_fp4, plain_to_chunked
from tests.test_gpu_gemm import assert_close, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def random_operands(M, G, N, K, seed):
    rng = np.random.default_rng(seed)
    sign = lambda shape: rng.integers(0, 2, shape, dtype=np.uint8) << 7
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8) | sign((M, K))
    qb = rng.integers(0, 0x7E, (G * N, K), dtype=np.uint8) | sign((G * N, K))
    sa = rng.integers(118, 136, (M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 136, (G * N, K // 32), dtype=np.uint8)
    return qa, sa, qb, sb


def run_grouped(sizes, N, K, out_dtype, seed, sample=None):
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    qa, sa, qb, sb = random_operands(M, G, N, K, seed)
    y = mx.mx_gemm_grouped(dev(qa), dev(plain_to_chunked(sa)), mx.E4M3, dev(qb), dev(plain_to_chunked(sb)), mx.E4M3,
                           dev(off), M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    yn = y.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        rows = (np.arange(hi - lo) if sample is None else tile_rows(hi - lo, salt=g) if sample == "tiles" else
                np.unique(np.linspace(0, hi - lo - 1, sample).astype(np.int64)))
        ref, ab = orc.mx_gemm(qa[lo:hi], sa[lo:hi], orc.E4M3, qb[g * N:(g + 1) * N], sb[g * N:(g + 1) * N], orc.E4M3,
                              rows=rows)
        assert_close(yn[lo + rows], ref, ab, bf16=out_dtype == mx.OUT_BF16, what=f"group {g}")


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_grouped_half_tiles_and_empty_groups(out_dtype):
    run_grouped([256, 128, 0, 384], 512, 512, out_dtype, seed=1)


def test_grouped_many_groups_moe_shape():
    rng = np.random.default_rng(2)
    sizes = (rng.integers(0, 9, 16) * 128).tolist()           # 16 experts, 0 .. 1024 rows each
    run_grouped(sizes, 1024, 2048, mx.OUT_BF16, seed=3, sample="tiles")


def test_grouped_moe_workload_shape_every_tile():
    # the bench's grouped MXFP8 workload: 8 experts 4096 -> 14336, 16384 routed rows split unevenly;
    # one row of every 128-row tile of every expert, all columns
    run_grouped([3328, 1536, 2432, 1024, 2816, 1920, 2176, 1152], 14336, 4096, mx.OUT_BF16, seed=5, sample="tiles")


def test_single_group_equals_plain_gemm():
    M, N, K = 512, 768, 1024
    qa, sa, qb, sb = random_operands(M, 1, N, K, 4)
    args = (dev(qa), dev(plain_to_chunked(sa)), mx.E4M3, dev(qb), dev(plain_to_chunked(sb)), mx.E4M3)
    y1 = mx.mx_gemm(*args, M, N, K, out_dtype=mx.OUT_F32)
    y2 = mx.mx_gemm_grouped(*args, dev(np.array([0, M], np.int64)), M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("off", [[0, 100, 256], [0, 384, 256], [128, 256, 512], [0, 256, 384]])
def test_grouped_rejects_broken_offsets_on_the_device(off):
    # not a multiple of 128, decreasing, not starting at 0, not ending at M (= 512): no tile runs
    M, N, K = 512, 256, 256
    qa, sa, qb, sb = random_operands(M, 2, N, K, 5)
    out = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    st = mx.load().mx_gemm_grouped(dev(qa).data_ptr(), dev(plain_to_chunked(sa)).data_ptr(), mx.E4M3,
                                   dev(qb).data_ptr(), dev(plain_to_chunked(sb)).data_ptr(), mx.E4M3,
                                   dev(np.array(off, np.int64)).data_ptr(), 2, M, N, K, out.data_ptr(), mx.OUT_F32, N,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == mx.MX_OK                          # the host cannot see device offsets
    assert mx.mx_check() == mx.MX_ERR_INVALID_ARG
    assert bool((out == 7.0).all())
    assert mx.mx_check() == mx.MX_OK               # the error word was cleared


# ------------------------------------------------------------------ FP4 experts
def fp4_grouped_operands(M, G, N, K, seed, nv):
    rng = np.random.default_rng(seed)
    ca = rng.integers(0, 16, (M, K), dtype=np.uint8)          # E2M1 codes (all 16 are finite)
    cb = rng.integers(0, 16, (G * N, K), dtype=np.uint8)
    if nv:   # UE4M3 block scales per 16, positive and finite
        sa = rng.integers(0x28, 0x48, (M, K // 16), dtype=np.uint8)
        sb = rng.integers(0x28, 0x48, (G * N, K // 16), dtype=np.uint8)
    else:    # E8M0 per 32
        sa = rng.integers(118, 136, (M, K // 32), dtype=np.uint8)
        sb = rng.integers(118, 136, (G * N, K // 32), dtype=np.uint8)
    return ca, sa, cb, sb


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_grouped_mxfp4(out_dtype):
    sizes, N, K = [256, 128, 0, 384], 512, 512
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    ca, sa, cb, sb = fp4_grouped_operands(M, G, N, K, 31, nv=False)
    y = mx.mx_gemm_grouped(dev(pack_fp4(ca)), dev(plain_to_chunked(sa)), mx.E2M1, dev(pack_fp4(cb)),
                           dev(plain_to_chunked(sb)), mx.E2M1, dev(off), M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    yn = y.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        ref, ab = orc.mx_gemm(ca[lo:hi], sa[lo:hi], orc.E2M1, cb[g * N:(g + 1) * N], sb[g * N:(g + 1) * N], orc.E2M1)
        assert_close(yn[lo:hi], ref, ab, bf16=out_dtype == mx.OUT_BF16, what=f"mxfp4 group {g}")


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_grouped_nvfp4_per_expert_global_scales(out_dtype):
    sizes, N, K = [128, 384, 0, 256, 128], 256, 512
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    ca, sa, cb, sb = fp4_grouped_operands(M, G, N, K, 32, nv=True)
    ga = np.float32(0.75)
    gb = np.array([0.5, 1.25, 3.0, 0.125, 2.0], np.float32)
    qa, qb = pack_fp4(ca), pack_fp4(cb)
    y = mx.nvfp4_gemm_grouped(dev(qa), dev(plain_to_chunked(sa)), torch.tensor([ga], device="cuda"), dev(qb),
                              dev(plain_to_chunked(sb)), torch.from_numpy(gb).cuda(), dev(off), M, N, K,
                              out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    yn = y.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        ref, ab = orc.nv_gemm(qa[lo:hi], sa[lo:hi], float(ga), qb[g * N:(g + 1) * N], sb[g * N:(g + 1) * N], float(gb[g]))
        assert_close(yn[lo:hi], ref, ab, bf16=out_dtype == mx.OUT_BF16, what=f"nvfp4 group {g}")


def test_grouped_nvfp4_single_group_equals_plain_gemm():
    M, N, K = 512, 768, 1024
    ca, sa, cb, sb = fp4_grouped_operands(M, 1, N, K, 33, nv=True)
    ga = torch.tensor([0.5], device="cuda")
    gb = torch.tensor([1.5], device="cuda")
    args = (dev(pack_fp4(ca)), dev(plain_to_chunked(sa)), ga, dev(pack_fp4(cb)), dev(plain_to_chunked(sb)), gb)
    y1 = mx.nvfp4_gemm(*args, M, N, K, out_dtype=mx.OUT_F32)
    y2 = mx.nvfp4_gemm_grouped(*args, dev(np.array([0, M], np.int64)), M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    assert torch.equal(y1, y2)


# ------------------------------------------------------------------ grouped NVFP4 quantization
from block_scaled_precision_mx_gb300 import synthetic  # noqa: E402


def nv_grouped_input(sizes, cols, seed):
    """bf16 rows of each group drawn at their own magnitude (and with sparse outliers), so every
    group has its own amax and global scale."""
    parts = [synthetic.with_sparse_outliers(n, cols, seed + g) * (4.0 ** (g % 5 - 2)) for g, n in enumerate(sizes) if n]
    return torch.cat(parts).to(torch.bfloat16)


def check_nv_grouped(x, sizes):
    """Quantize x by groups on the GPU and compare every group with the oracle's quantization of
    that group's rows as a tensor of its own (codes, scales, global scale bit for bit)."""
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    rows, cols = x.shape
    q, s, g = mx.nvfp4_quantize_grouped(x.cuda(), dev(off))
    assert mx.mx_check() == mx.MX_OK
    qn, gn = q.cpu().numpy(), g.cpu().numpy()
    sn = chunked_to_plain(s.cpu().numpy(), rows, cols // 16)
    for k in range(len(sizes)):
        lo, hi = int(off[k]), int(off[k + 1])
        if hi == lo:
            assert gn[k] == np.float32(1.0), f"empty group {k}: global scale {gn[k]}"
            continue
        oq, osc, og = orc.nv_quantize(x[lo:hi])
        assert np.array_equal(qn[lo:hi], oq), f"group {k}: codes"
        assert np.array_equal(sn[lo:hi], osc), f"group {k}: scales"
        assert gn[k].view(np.uint32) == np.float32(og).view(np.uint32), f"group {k}: global scale"
    return q, s, g, off


def test_nvfp4_quantize_grouped_per_group_scales():
    # uneven groups, an empty one, and a half-filled last 128-column tile (cols % 128 == 64)
    check_nv_grouped(nv_grouped_input([384, 0, 128, 640], 320, 9100), [384, 0, 128, 640])


def test_nvfp4_quantize_grouped_single_group():
    check_nv_grouped(nv_grouped_input([512], 256, 9200), [512])


def test_nvfp4_quantize_grouped_moe_weights_full_size():
    # the MoE weights of the grouped-GEMM workload: 8 experts of 14336 x 4096, one global scale each
    sizes = [14336] * 8
    x = torch.cat([synthetic.normal(14336, 4096, 0.02 * (1 + e), 9300 + e) for e in range(8)])
    check_nv_grouped(x, sizes)


def test_nvfp4_quantize_grouped_feeds_grouped_gemm():
    # experts' weights quantized by groups, tokens as one tensor, then the grouped product
    sizes, N, K = [256, 128, 0, 384], 256, 512
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    a = synthetic.with_sparse_outliers(M, K, 9400)
    w = nv_grouped_input([N] * G, K, 9500)
    qa, sa, ga = mx.nvfp4_quantize(a.cuda())
    qb, sb, gb, _ = check_nv_grouped(w, [N] * G)
    y = mx.nvfp4_gemm_grouped(qa, sa, ga, qb, sb, gb, dev(off), M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    oqa, osa, oga = orc.nv_quantize(a)
    yn = y.cpu().numpy()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        oqb, osb, ogb = orc.nv_quantize(w[g * N:(g + 1) * N])
        ref, ab = orc.nv_gemm(oqa[lo:hi], osa[lo:hi], oga, oqb, osb, ogb)
        assert_close(yn[lo:hi], ref, ab, bf16=False, what=f"expert {g}")


@pytest.mark.parametrize("off", [[0, 100, 256], [0, 128], [0, 256, 128, 256]])
def test_nvfp4_quantize_grouped_rejects_broken_offsets_on_the_device(off):
    x = synthetic.normal(256, 128, 1.0, 9600).cuda()
    offsets = dev(np.array(off, np.int64))
    mx.nvfp4_quantize_grouped(x, offsets)
    assert mx.mx_check() == mx.MX_ERR_INVALID_ARG
    # the context stays usable: a valid call right after is exact
    check_nv_grouped(synthetic.normal(256, 128, 1.0, 9601), [128, 128])


def test_nvfp4_grouped_gemm_per_expert_token_scales():
    # the routed tokens quantized by expert (one global scale per expert's tokens) and the experts'
    # weights by expert: group g's results scaled by ga[g] * gb[g]
    sizes, N, K = [384, 0, 128, 256], 256, 512
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    a = nv_grouped_input(sizes, K, 9700)
    w = nv_grouped_input([N] * G, K, 9800)
    qa, sa, ga, _ = check_nv_grouped(a, sizes)
    qb, sb, gb, _ = check_nv_grouped(w, [N] * G)
    y = mx.nvfp4_gemm_grouped_ex(qa, sa, ga, True, qb, sb, gb, dev(off), M, N, K, out_dtype=mx.OUT_BF16)
    assert mx.mx_check() == mx.MX_OK
    yn = y.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        oqa, osa, oga = orc.nv_quantize(a[lo:hi])
        oqb, osb, ogb = orc.nv_quantize(w[g * N:(g + 1) * N])
        ref, ab = orc.nv_gemm(oqa, osa, oga, oqb, osb, ogb)
        assert_close(yn[lo:hi], ref, ab, bf16=True, what=f"expert {g}")


# ------------------------------------------------------------------ grouped DeepSeek FP8
def ds_grouped_operands(M, G, N, K, seed):
    rng = np.random.default_rng(seed)
    sign = lambda shape: rng.integers(0, 2, shape, dtype=np.uint8) << 7
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8) | sign((M, K))
    qb = rng.integers(0, 0x7E, (G * N, K), dtype=np.uint8) | sign((G * N, K))
    sa = (rng.random((M, K // 128)) * 0.01 + 0.001).astype(np.float32)             # [M][K/128]
    sb = (rng.random((G * N // 128, K // 128)) * 0.01 + 0.001).astype(np.float32)   # [G N/128][K/128]
    return qa, sa, qb, sb


def run_ds_grouped(sizes, N, K, out_dtype, seed, sample=None):
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    qa, sa, qb, sb = ds_grouped_operands(M, G, N, K, seed)
    y = mx.fp8_blockwise_gemm_grouped(dev(qa), dev(sa.T), dev(qb), dev(sb), dev(off), M, N, K, out_dtype=out_dtype)
    assert mx.mx_check() == mx.MX_OK
    yn = y.float().cpu().numpy()
    for g in range(G):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi == lo:
            continue
        rows = (np.arange(hi - lo) if sample is None else tile_rows(hi - lo, salt=g) if sample == "tiles" else
                np.unique(np.linspace(0, hi - lo - 1, sample).astype(np.int64)))
        ref, ab = orc.ds_gemm(qa[lo:hi], sa[lo:hi], qb[g * N:(g + 1) * N], sb[g * N // 128:(g + 1) * N // 128], rows=rows)
        assert_close(yn[lo + rows], ref, ab, bf16=out_dtype == mx.OUT_BF16, what=f"deepseek group {g}")
    return qa, sa, qb, sb, off, y


@pytest.mark.parametrize("out_dtype", [mx.OUT_F32, mx.OUT_BF16])
def test_ds_grouped_half_tiles_and_empty_groups(out_dtype):
    run_ds_grouped([128, 384, 0, 256, 128], 256, 512, out_dtype, 9900)


def test_ds_grouped_moe_shape_every_tile():
    # the grouped-GEMM workload: 8 experts 4096 -> 14336, 16384 routed rows split unevenly; one row of
    # every 128-row tile of every expert, all columns
    run_ds_grouped([3328, 1536, 2432, 1024, 2816, 1920, 2176, 1152], 14336, 4096, mx.OUT_BF16, 9910, sample="tiles")


def test_ds_grouped_single_group_equals_plain_gemm():
    M, N, K = 512, 768, 1024
    qa, sa, qb, sb = ds_grouped_operands(M, 1, N, K, 9920)
    args = (dev(qa), dev(sa.T), dev(qb), dev(sb))
    y1 = mx.fp8_blockwise_gemm(*args, M, N, K, out_dtype=mx.OUT_F32)
    y2 = mx.fp8_blockwise_gemm_grouped(*args, dev(np.array([0, M], np.int64)), M, N, K, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    assert torch.equal(y1, y2)


def test_ds_grouped_rejects_broken_offsets_on_the_device():
    M, N, K = 256, 256, 256
    qa, sa, qb, sb = ds_grouped_operands(M, 2, N, K, 9930)
    mx.fp8_blockwise_gemm_grouped(dev(qa), dev(sa.T), dev(qb), dev(sb), dev(np.array([0, 100, 256], np.int64)),
                                  M, N, K)
    assert mx.mx_check() == mx.MX_ERR_INVALID_ARG
    run_ds_grouped([128, 128], N, K, mx.OUT_BF16, 9931)


def test_nvfp4_quantize_grouped_many_groups():
    # the most groups a call takes (1024), most of them empty, at the narrowest width (64 columns)
    rng = np.random.default_rng(9950)
    sizes = np.zeros(1024, np.int64)
    sizes[rng.choice(1024, 40, replace=False)] = rng.integers(1, 4, 40) * 128
    x = torch.cat([synthetic.normal(int(n), 64, 2.0 ** (k % 9 - 4), 9960 + k) for k, n in enumerate(sizes) if n])
    check_nv_grouped(x.to(torch.bfloat16), [int(n) for n in sizes])


def test_ds_grouped_many_small_groups():
    # 64 experts of 128 or 256 rows (some empty): tiles of one group never mix with another's
    rng = np.random.default_rng(9970)
    sizes = (rng.integers(0, 3, 64) * 128).tolist()
    run_ds_grouped(sizes, 256, 256, mx.OUT_F32, 9971)
