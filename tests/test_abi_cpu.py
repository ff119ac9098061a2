"""CPU checks of the C ABI: the library builds, loads without a GPU, exports every symbol that
include/mx.h declares, and rejects invalid arguments on the host before any launch.  Also
checks the test-side layout permutations."""
import ctypes
import os
import re

import numpy as np
import pytest

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import build as mxbuild
from tests.layouts import chunked_to_plain, plain_to_chunked, unpack_fp4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mxbuild.build()
    return mx.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "mx_quantize" in names and "fp8_blockwise_gemm" in names and "nvfp4_gemm" in names
    cdll = ctypes.CDLL(mx.library_path())
    for n in names:
        assert hasattr(cdll, n), n
    assert set(names) <= set(mx.EXPORTS)


def test_status_strings_and_version(lib):
    assert lib.mx_abi_version() == 1
    assert mx.status_string(mx.MX_OK) == "MX_OK"
    assert mx.status_string(mx.MX_ERR_TIMEOUT) == "MX_ERR_TIMEOUT"
    assert mx.status_string(99) == "MX_ERR_UNKNOWN"


def test_scale_bytes(lib):
    assert mx.mx_scale_bytes(16384, 4096, 32, 1, mx.SCALE_E8M0) == 16384 * 128
    assert mx.mx_scale_bytes(8192, 8192, 16, 1, mx.SCALE_UE4M3) == 8192 * 512
    assert mx.mx_scale_bytes(4096, 7168, 128, 1, mx.SCALE_FP32) == 4 * 4096 * 56
    assert mx.mx_scale_bytes(2048, 7168, 128, 128, mx.SCALE_FP32) == 4 * 16 * 56
    assert mx.mx_scale_bytes(128, 128, 64, 1, mx.SCALE_E8M0) == 0


FAKE = 1 << 20  # non-null, 16-byte aligned, never dereferenced: validation fails first


def test_quantize_rejects_bad_arguments(lib):
    q = lib.mx_quantize
    ok_args = dict(x=FAKE, rows=256, cols=256, block=32, block_rows=1, elem=0, sfmt=0, layout=3,
                   qr=FAKE, sr=FAKE, qc=FAKE, sc=FAKE)

    def call(**kw):
        a = dict(ok_args, **kw)
        return q(a["x"], a["rows"], a["cols"], a["block"], a["block_rows"], a["elem"], a["sfmt"], a["layout"],
                 a["qr"], a["sr"], a["qc"], a["sc"], None)

    assert call(x=None) == mx.MX_ERR_INVALID_ARG
    assert call(rows=100) == mx.MX_ERR_INVALID_ARG
    assert call(cols=0) == mx.MX_ERR_INVALID_ARG
    assert call(x=FAKE + 8) == mx.MX_ERR_INVALID_ARG
    assert call(elem=7) == mx.MX_ERR_INVALID_ARG
    assert call(layout=0) == mx.MX_ERR_INVALID_ARG
    assert call(qc=None) == mx.MX_ERR_INVALID_ARG          # column-wise requested, no buffer
    assert call(block=64) == mx.MX_ERR_UNSUPPORTED
    assert call(block=128, sfmt=2, layout=2) == mx.MX_ERR_UNSUPPORTED   # DeepSeek column-wise
    assert call(elem=2, block=16) == mx.MX_ERR_UNSUPPORTED  # E2M1 blocks of 16 with E8M0: not MX
    assert call(rows=128, cols=65536 * 128) == mx.MX_ERR_INVALID_ARG   # more than 65535 column tiles
    assert call(block_rows=32, elem=2) == mx.MX_ERR_UNSUPPORTED      # 2-D blocks are MXFP8 only
    assert call(sfmt=3) == mx.MX_ERR_UNSUPPORTED                     # power-of-two FP32 needs block 128
    assert call(block=128, sfmt=3, layout=3) == mx.MX_ERR_UNSUPPORTED
    assert call(sfmt=4) == mx.MX_ERR_INVALID_ARG


def test_nvfp4_option_entries_reject_bad_arguments(lib):
    e = lib.nvfp4_quantize_ex
    assert e(FAKE, 128, 128, 2, 0, None, FAKE, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG   # use_rht
    assert e(FAKE, 128, 128, 1, 0x10000, None, FAKE, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert e(FAKE, 128, 128, 0, 0, FAKE + 4, FAKE, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG  # rbits
    assert e(FAKE, 128, 96, 0, 0, None, FAKE, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG
    d = lib.nvfp4_quantize_2d
    assert d(FAKE, 128, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG      # cols % 128
    assert d(FAKE, 128, 128, FAKE, FAKE, None, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert d(FAKE, 128, 128, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == mx.MX_ERR_INVALID_ARG


def test_grouped_gemm_rejects_bad_arguments(lib):
    g = lib.mx_gemm_grouped
    ok = [FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 2, 512, 512, 256, FAKE, 1, 512, None]

    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return g(*a)
    assert call(a6=None) == mx.MX_ERR_INVALID_ARG          # no offsets
    assert call(a7=0) == mx.MX_ERR_INVALID_ARG             # no groups
    assert call(a7=1025) == mx.MX_ERR_INVALID_ARG
    assert call(a9=384) == mx.MX_ERR_INVALID_ARG           # N % 256
    assert call(a6=FAKE + 4) == mx.MX_ERR_INVALID_ARG      # offsets alignment
    assert call(a2=2) == mx.MX_ERR_UNSUPPORTED             # MXFP4 operands
    assert call(a2=9) == mx.MX_ERR_INVALID_ARG


def test_fused_output_gemm_rejects_bad_arguments(lib):
    f = lib.mx_gemm_mxout
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 256, 256, 0, FAKE, FAKE, 256, None) == mx.MX_ERR_INVALID_ARG  # M % 256
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 0, 256, 256, 256, 0, FAKE, FAKE, 128, None) == mx.MX_ERR_INVALID_ARG  # ldq < N
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 0, 256, 256, 256, 0, None, FAKE, 256, None) == mx.MX_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 0, 256, 256, 256, 2, FAKE, FAKE, 256, None) == mx.MX_ERR_UNSUPPORTED  # E2M1 out
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 0, 256, 256, 256, 5, FAKE, FAKE, 256, None) == mx.MX_ERR_INVALID_ARG


def test_scale_conversion_rejects_bad_arguments(lib):
    c = lib.mx_scales_from_fp32_blocks
    assert c(None, 128, 128, 1, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert c(FAKE, 100, 128, 1, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert c(FAKE, 128, 128, 32, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert c(FAKE, 128, 128, 1, FAKE + 8, None) == mx.MX_ERR_INVALID_ARG
    assert c(FAKE + 2, 128, 128, 128, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert mx.mx_scale_bytes(256, 512, 32, 32, mx.SCALE_E8M0) == 256 * 16
    assert mx.mx_scale_bytes(256, 512, 128, 128, mx.SCALE_FP32_POW2) == 4 * 2 * 4


def test_scale_layout_permutations_reject_bad_arguments(lib):
    for f in (lib.mx_unswizzle_scales, lib.mx_swizzle_scales):
        assert f(None, 128, 4, FAKE, None) == mx.MX_ERR_INVALID_ARG
        assert f(FAKE, 128, 4, None, None) == mx.MX_ERR_INVALID_ARG
        assert f(FAKE, 96, 4, FAKE, None) == mx.MX_ERR_INVALID_ARG       # rows not a multiple of 128
        assert f(FAKE, 128, 6, FAKE, None) == mx.MX_ERR_INVALID_ARG      # blocks not a multiple of 4
        assert f(FAKE, 128, 0, FAKE, None) == mx.MX_ERR_INVALID_ARG
    # the chunked side must be 16-byte aligned, the plain side 4-byte aligned
    assert lib.mx_unswizzle_scales(FAKE + 4, 128, 4, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_unswizzle_scales(FAKE, 128, 4, FAKE + 2, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_swizzle_scales(FAKE + 2, 128, 4, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_swizzle_scales(FAKE, 128, 4, FAKE + 4, None) == mx.MX_ERR_INVALID_ARG


def test_wait_selftest_rejects_bad_budgets(lib):
    for budget in (0, -5, 1000001):
        assert lib.mx_selftest_wait_timeout(budget, None) == mx.MX_ERR_INVALID_ARG


def test_fused_output_ex_rejects_bad_arguments(lib):
    f = lib.mx_gemm_mxout_ex
    base = [FAKE, FAKE, mx.E4M3, FAKE, FAKE, mx.E4M3, 256, 256, 256, mx.E4M3]
    ok_row = [FAKE, FAKE, 256]
    ok_col = [FAKE, FAKE, 256]
    assert f(*base, 0, *ok_row, *ok_col, None) == mx.MX_ERR_INVALID_ARG             # no layout
    assert f(*base, mx.COLWISE, *ok_row, None, FAKE, 256, None) == mx.MX_ERR_INVALID_ARG
    assert f(*base, mx.ROWWISE, None, FAKE, 256, *ok_col, None) == mx.MX_ERR_INVALID_ARG
    assert f(*base, mx.COLWISE, None, None, 0, FAKE, FAKE, 128, None) == mx.MX_ERR_INVALID_ARG   # ldq_col < M
    assert f(*base, mx.COLWISE, None, None, 0, FAKE + 8, FAKE, 256, None) == mx.MX_ERR_INVALID_ARG
    b2 = list(base)
    b2[6] = 128                                                                         # M not a multiple of 256
    assert f(*b2, mx.BOTH, *ok_row, *ok_col, None) == mx.MX_ERR_INVALID_ARG
    b3 = list(base)
    b3[9] = mx.E2M1
    assert f(*b3, mx.BOTH, *ok_row, *ok_col, None) == mx.MX_ERR_UNSUPPORTED


def test_nvfp4_quantize_grouped_rejects_bad_arguments(lib):
    f = lib.nvfp4_quantize_grouped
    ok = [FAKE, 256, 128, FAKE, 2, FAKE, FAKE, FAKE, FAKE, None]
    for i, v, why in ((3, None, "no offsets"), (4, 0, "no groups"), (4, 1025, "too many groups"),
                      (3, FAKE + 4, "offsets not 8-byte aligned"), (1, 192, "rows % 128"), (2, 96, "cols % 64"),
                      (0, None, "no input"), (7, None, "no global scales"), (8, None, "no workspace"),
                      (8, FAKE + 8, "workspace alignment")):
        bad = list(ok); bad[i] = v
        assert f(*bad) == mx.MX_ERR_INVALID_ARG, why


def test_nvfp4_grouped_ex_rejects_bad_arguments(lib):
    f = lib.nvfp4_gemm_grouped_ex
    ok = [FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, 2, 256, 256, 256, FAKE, mx.OUT_F32, 256, None]
    for i, v, why in ((3, 2, "ga_per_group not 0 or 1"), (3, -1, "ga_per_group not 0 or 1"), (2, None, "no ga"),
                      (8, 0, "no groups"), (7, FAKE + 4, "offsets alignment"), (11, 128, "K % 256")):
        bad = list(ok); bad[i] = v
        assert f(*bad) == mx.MX_ERR_INVALID_ARG, why


def test_ds_grouped_rejects_bad_arguments(lib):
    f = lib.fp8_blockwise_gemm_grouped
    ok = [FAKE, FAKE, FAKE, FAKE, FAKE, 2, 256, 256, 256, FAKE, mx.OUT_BF16, 256, None]
    for i, v, why in ((4, None, "no offsets"), (5, 0, "no groups"), (5, 1025, "too many groups"),
                      (7, 128, "N % 256"), (8, 64, "K % 128"), (6, 192, "M % 128"), (4, FAKE + 4, "offsets alignment"),
                      (1, FAKE + 2, "scale alignment"), (0, None, "no A")):
        bad = list(ok); bad[i] = v
        assert f(*bad) == mx.MX_ERR_INVALID_ARG, why


def test_nvfp4_grouped_rejects_bad_arguments(lib):
    f = lib.nvfp4_gemm_grouped
    ok = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 256, 256, 256, FAKE, mx.OUT_F32, 256, None]
    bad = list(ok); bad[2] = None                     # no global scale of A
    assert f(*bad) == mx.MX_ERR_INVALID_ARG
    bad = list(ok); bad[7] = 0                        # no groups
    assert f(*bad) == mx.MX_ERR_INVALID_ARG
    bad = list(ok); bad[10] = 128                     # K not a multiple of 256
    assert f(*bad) == mx.MX_ERR_INVALID_ARG
    bad = list(ok); bad[9] = 128                      # N not a multiple of 256
    assert f(*bad) == mx.MX_ERR_INVALID_ARG
    bad = list(ok); bad[6] = FAKE + 4                 # offsets not 8-byte aligned
    assert f(*bad) == mx.MX_ERR_INVALID_ARG
    g = lib.mx_gemm_grouped
    assert g(FAKE, FAKE, mx.E2M1, FAKE, FAKE, mx.E4M3, FAKE, 1, 256, 256, 256, FAKE, mx.OUT_F32, 256,
             None) == mx.MX_ERR_UNSUPPORTED              # FP4 x FP8 experts
    assert g(FAKE, FAKE, mx.E2M1, FAKE, FAKE, mx.E2M1, FAKE, 1, 256, 256, 128, FAKE, mx.OUT_F32, 256,
             None) == mx.MX_ERR_INVALID_ARG              # MXFP4 needs K % 256


def test_dual_quantize_rejects_bad_arguments(lib):
    d = lib.mx_quantize_dual
    ptrs = [FAKE] * 8
    # only argument combinations the host rejects: valid ones would launch on fake pointers
    assert d(None, 256, 256, 3, *ptrs, None) == mx.MX_ERR_INVALID_ARG
    assert d(FAKE, 200, 256, 3, *ptrs, None) == mx.MX_ERR_INVALID_ARG
    assert d(FAKE, 256, 256, 0, *ptrs, None) == mx.MX_ERR_INVALID_ARG
    bad = list(ptrs)
    bad[6] = None                            # column-wise E5M2 codes missing
    assert d(FAKE, 256, 256, 3, *bad, None) == mx.MX_ERR_INVALID_ARG
    assert d(FAKE, 256, 256, 2, *bad, None) == mx.MX_ERR_INVALID_ARG
    bad[1] = FAKE + 4                        # misaligned row-wise E4M3 scales
    assert d(FAKE, 256, 256, 1, *bad, None) == mx.MX_ERR_INVALID_ARG


def test_gemms_reject_bad_arguments(lib):
    g = lib.mx_gemm
    assert g(None, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, FAKE, 1, 128, None) == mx.MX_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 0, FAKE, FAKE, 0, 100, 128, 128, FAKE, 1, 128, None) == mx.MX_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 96, FAKE, 1, 128, None) == mx.MX_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, FAKE, 1, 64, None) == mx.MX_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 0, FAKE, FAKE, 0, 128, 128, 128, FAKE, 5, 128, None) == mx.MX_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 2, FAKE, FAKE, 0, 128, 128, 128, FAKE, 1, 128, None) == mx.MX_ERR_UNSUPPORTED  # FP4 x FP8
    assert g(FAKE, FAKE, 2, FAKE, FAKE, 2, 128, 128, 128, FAKE, 1, 128, None) == mx.MX_ERR_INVALID_ARG  # MXFP4 K % 256
    assert g(FAKE, FAKE, 7, FAKE, FAKE, 2, 128, 128, 256, FAKE, 1, 128, None) == mx.MX_ERR_INVALID_ARG  # bad enum
    n = lib.nvfp4_gemm
    assert n(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 128, FAKE, 0, 128, None) == mx.MX_ERR_INVALID_ARG
    assert n(FAKE, FAKE, None, FAKE, FAKE, FAKE, 128, 128, 256, FAKE, 0, 128, None) == mx.MX_ERR_INVALID_ARG
    d = lib.fp8_blockwise_gemm
    assert d(FAKE, FAKE, FAKE, FAKE, 128, 100, 128, FAKE, 1, 128, None) == mx.MX_ERR_INVALID_ARG
    nq = lib.nvfp4_quantize
    assert nq(FAKE, 128, 96, FAKE, FAKE, FAKE, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert nq(FAKE, 128, 128, FAKE, FAKE, FAKE, None, None) == mx.MX_ERR_INVALID_ARG
    assert lib.nvfp4_workspace_bytes(8192, 8192) >= 16


def test_layout_permutations_roundtrip():
    rng = np.random.default_rng(0)
    plain = rng.integers(0, 256, (256, 12), dtype=np.uint8)
    flat = plain_to_chunked(plain)
    assert flat.shape == (256 * 12,)
    assert np.array_equal(chunked_to_plain(flat, 256, 12), plain)
    # spot-check the documented byte offset: row 128*rb + i, block 4*kc + j
    rb, i, kc, j = 1, 77, 2, 3
    off = (rb * 3 + kc) * 512 + (i % 32) * 16 + (i // 32) * 4 + j
    assert flat[off] == plain[128 * rb + i, 4 * kc + j]
    qp = np.array([[0x21, 0x43]], np.uint8)
    assert unpack_fp4(qp).tolist() == [[1, 2, 3, 4]]
