"""GB300 (sm_103a) block-scaled quantization and GEMMs: MXFP8, MXFP4, NVFP4, DeepSeek FP8.

Thin Python binding over the C ABI of ``libmxgb.so`` (declared in include/mx.h).
Every function here only marshals arguments: tensors are torch CUDA tensors
(device memory), the stream is torch's current stream unless one is given,
and every step of the computation runs in the library's CUDA kernels.  There
is no CPU fallback: if the library cannot be loaded, every call raises.

Entry points (same names as the C ABI):
  mx_quantize, mx_quantize_dual, mx_gemm, nvfp4_quantize, nvfp4_gemm, fp8_blockwise_gemm,
  mx_gemm_grouped, mx_gemm_mxout, mx_scales_from_fp32_blocks, nvfp4_quantize_ex, nvfp4_quantize_2d,
  nvfp4_quantize_grouped, nvfp4_gemm_grouped, nvfp4_gemm_grouped_ex, fp8_blockwise_gemm_grouped, mx_scale_bytes,
  nvfp4_workspace_bytes, mx_check.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB as _LIB_PATH

# enums (include/mx.h)
MX_OK, MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED, MX_ERR_CUDA, MX_ERR_TIMEOUT = range(5)
E4M3, E5M2, E2M1 = 0, 1, 2
SCALE_E8M0, SCALE_UE4M3, SCALE_FP32, SCALE_FP32_POW2 = 0, 1, 2, 3
ROWWISE, COLWISE, BOTH = 1, 2, 3
OUT_F32, OUT_BF16 = 0, 1

EXPORTS = (
    "mx_abi_version", "mx_status_string", "mx_quantize", "mx_gemm", "nvfp4_workspace_bytes",
    "nvfp4_quantize", "nvfp4_gemm", "fp8_blockwise_gemm", "mx_scale_bytes", "mx_check", "mx_num_sms",
    "nvfp4_quantize_noalloc", "mx_quantize_dual", "mx_scales_from_fp32_blocks", "nvfp4_quantize_ex",
    "nvfp4_quantize_2d", "mx_gemm_grouped", "mx_gemm_mxout", "mx_unswizzle_scales", "mx_swizzle_scales",
    "mx_selftest_wait_timeout", "mx_gemm_mxout_ex", "nvfp4_gemm_grouped", "nvfp4_quantize_grouped",
    "nvfp4_gemm_grouped_ex", "fp8_blockwise_gemm_grouped",
)


class MxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libmxgb.so (built by build.py / __graft_entry__.build()).  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmxgb.so not built ({_LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        fp = ctypes.POINTER(ctypes.c_float)
        sig = {
            "mx_abi_version": (i32, []),
            "mx_status_string": (ctypes.c_char_p, [i32]),
            "mx_quantize": (i32, [vp, i64, i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]),
            "mx_gemm": (i32, [vp, vp, i32, vp, vp, i32, i64, i64, i64, vp, i32, i64, vp]),
            "nvfp4_workspace_bytes": (ctypes.c_size_t, [i64, i64]),
            "nvfp4_quantize": (i32, [vp, i64, i64, vp, vp, vp, vp, vp]),
            "nvfp4_gemm": (i32, [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, i32, i64, vp]),
            "fp8_blockwise_gemm": (i32, [vp, vp, vp, vp, i64, i64, i64, vp, i32, i64, vp]),
            "mx_scale_bytes": (ctypes.c_size_t, [i64, i64, i32, i32, i32]),
            "mx_check": (i32, [vp]),
            "mx_num_sms": (i32, []),
            "nvfp4_quantize_noalloc": (i32, [vp, i64, i64, vp, vp, vp, vp]),
            "mx_quantize_dual": (i32, [vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "mx_scales_from_fp32_blocks": (i32, [vp, i64, i64, i32, vp, vp]),
            "nvfp4_quantize_ex": (i32, [vp, i64, i64, i32, ctypes.c_uint32, vp, vp, vp, vp, vp, vp]),
            "nvfp4_quantize_2d": (i32, [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp]),
            "mx_gemm_grouped": (i32, [vp, vp, i32, vp, vp, i32, vp, i64, i64, i64, i64, vp, i32, i64, vp]),
            "mx_gemm_mxout": (i32, [vp, vp, i32, vp, vp, i32, i64, i64, i64, i32, vp, vp, i64, vp]),
            "mx_unswizzle_scales": (i32, [vp, i64, i64, vp, vp]),
            "mx_swizzle_scales": (i32, [vp, i64, i64, vp, vp]),
            "mx_selftest_wait_timeout": (i32, [i64, vp]),
            "nvfp4_gemm_grouped": (i32, [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, i32, i64, vp]),
            "nvfp4_quantize_grouped": (i32, [vp, i64, i64, vp, i64, vp, vp, vp, vp, vp]),
            "nvfp4_gemm_grouped_ex": (i32, [vp, vp, vp, i32, vp, vp, vp, vp, i64, i64, i64, i64, vp, i32, i64, vp]),
            "fp8_blockwise_gemm_grouped": (i32, [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, i32, i64, vp]),
            "mx_gemm_mxout_ex": (i32, [vp, vp, i32, vp, vp, i32, i64, i64, i64, i32, i32, vp, vp, i64, vp, vp, i64,
                                       vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().mx_status_string(status).decode()


def _check(status: int, where: str):
    if status != MX_OK:
        raise MxError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:   # the current stream's handle without building a Stream object
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _u8(n, device):
    return torch.empty(int(n), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ sizes
def mx_scale_bytes(rows: int, cols: int, block: int = 32, block_rows: int = 1, sfmt: int = SCALE_E8M0) -> int:
    return int(load().mx_scale_bytes(rows, cols, block, block_rows, sfmt))


def nvfp4_workspace_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_workspace_bytes(rows, cols))


# ------------------------------------------------------------------ quantizers
def mx_quantize(x: torch.Tensor, block: int = 32, block_rows: int = 1, elem: int = E4M3,
                sfmt: int = SCALE_E8M0, layout: int = BOTH, q_row=None, s_row=None, q_col=None,
                s_col=None, stream=None):
    """Block-quantize bf16 x[rows][cols] (see include/mx.h, mx_quantize).

    Returns (q_row, s_row, q_col, s_col); outputs not given are allocated (torch), copies not
    requested are None.  MX scales are returned as flat uint8 tensors in the GEMM layout;
    DeepSeek FP32 scales as float tensors ([cols/128][rows] for 1x128, [rows/128][cols/128]
    for 128x128)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    row, col = bool(layout & ROWWISE), bool(layout & COLWISE)
    if sfmt in (SCALE_FP32, SCALE_FP32_POW2):
        if row and q_row is None:
            q_row = torch.empty(rows, cols, dtype=torch.uint8, device=dev)
        if row and s_row is None:
            shape = (cols // 128, rows) if block_rows == 1 else (rows // 128, cols // 128)
            s_row = torch.empty(shape, dtype=torch.float32, device=dev)
    else:
        per_byte = 2 if elem == E2M1 else 1          # MXFP4 codes are packed two per byte
        if row and q_row is None:
            q_row = torch.empty(rows, cols // per_byte, dtype=torch.uint8, device=dev)
        if row and s_row is None:
            s_row = _u8(mx_scale_bytes(rows, cols, block, block_rows, sfmt), dev)
        if col and q_col is None:
            q_col = torch.empty(cols, rows // per_byte, dtype=torch.uint8, device=dev)
        if col and s_col is None:
            s_col = _u8(mx_scale_bytes(cols, rows, block, block_rows, sfmt), dev)
    st = load().mx_quantize(_ptr(x), rows, cols, block, block_rows, elem, sfmt, layout,
                            _ptr(q_row) if row else None, _ptr(s_row) if row else None,
                            _ptr(q_col) if col else None, _ptr(s_col) if col else None, _stream(stream))
    _check(st, "mx_quantize")
    return (q_row if row else None, s_row if row else None, q_col if col else None, s_col if col else None)


def mx_scales_from_fp32_blocks(s: torch.Tensor, rows: int, cols: int, block_rows: int, out=None, stream=None):
    """Per-32 E8M0 scales (MX GEMM layout, flat uint8) for a [rows][cols] code matrix from its
    power-of-two FP32 block scales (include/mx.h, mx_scales_from_fp32_blocks)."""
    if s.dtype != torch.float32:
        raise ValueError("s must be float32")
    if out is None:
        out = _u8(rows * cols // 32, s.device)
    st = load().mx_scales_from_fp32_blocks(_ptr(s), rows, cols, block_rows, _ptr(out), _stream(stream))
    _check(st, "mx_scales_from_fp32_blocks")
    return out


def mx_selftest_wait_timeout(budget_us: int = 10000, stream=None):
    """Make one device-side bounded wait run out (include/mx.h, mx_selftest_wait_timeout); the
    next mx_check() reports MX_ERR_TIMEOUT."""
    _check(load().mx_selftest_wait_timeout(budget_us, _stream(stream)), "mx_selftest_wait_timeout")


def mx_unswizzle_scales(s: torch.Tensor, rows: int, nblocks: int, out=None, stream=None):
    """GEMM-layout scale bytes -> plain uint8 [rows][nblocks] (include/mx.h, mx_unswizzle_scales);
    nblocks = K/32 for MX scales, K/16 for NVFP4 scales."""
    if s.dtype != torch.uint8:
        raise ValueError("s must be uint8")
    if out is None:
        out = torch.empty(rows, nblocks, dtype=torch.uint8, device=s.device)
    _check(load().mx_unswizzle_scales(_ptr(s), rows, nblocks, _ptr(out), _stream(stream)), "mx_unswizzle_scales")
    return out


def mx_swizzle_scales(plain: torch.Tensor, out=None, stream=None):
    """plain uint8 [rows][nblocks] -> GEMM-layout scale bytes, flat (include/mx.h, mx_swizzle_scales)."""
    if plain.dtype != torch.uint8 or plain.dim() != 2:
        raise ValueError("plain must be a 2-D uint8 tensor")
    rows, nblocks = plain.shape
    if out is None:
        out = _u8(rows * nblocks, plain.device)
    _check(load().mx_swizzle_scales(_ptr(plain), rows, nblocks, _ptr(out), _stream(stream)), "mx_swizzle_scales")
    return out


def mx_quantize_dual(x: torch.Tensor, layout: int = BOTH, e4m3=None, e5m2=None, stream=None):
    """E4M3 and E5M2 MX quantization of bf16 x from one read (include/mx.h, mx_quantize_dual).
    e4m3 / e5m2: optional (q_row, s_row, q_col, s_col) output tuples; returns both tuples."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    row, col = bool(layout & ROWWISE), bool(layout & COLWISE)

    def alloc():
        return (torch.empty(rows, cols, dtype=torch.uint8, device=dev) if row else None,
                _u8(mx_scale_bytes(rows, cols), dev) if row else None,
                torch.empty(cols, rows, dtype=torch.uint8, device=dev) if col else None,
                _u8(mx_scale_bytes(cols, rows), dev) if col else None)
    e4m3 = e4m3 if e4m3 is not None else alloc()
    e5m2 = e5m2 if e5m2 is not None else alloc()
    st = load().mx_quantize_dual(_ptr(x), rows, cols, layout, *[_ptr(t) for t in e4m3], *[_ptr(t) for t in e5m2],
                                 _stream(stream))
    _check(st, "mx_quantize_dual")
    return e4m3, e5m2


def nvfp4_quantize(x: torch.Tensor, q_packed=None, s_ue4m3=None, gscale=None, workspace=None, stream=None):
    """NVFP4 two-level quantization of bf16 x[rows][cols] (include/mx.h, nvfp4_quantize).
    Returns (q_packed [rows][cols/2] u8, s_ue4m3 flat u8 in the NVFP4 GEMM layout,
    gscale float[1])."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    if q_packed is None:
        q_packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    if s_ue4m3 is None:
        s_ue4m3 = _u8(mx_scale_bytes(rows, cols, 16, 1, SCALE_UE4M3), dev)
    if gscale is None:
        gscale = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _u8(max(16, nvfp4_workspace_bytes(rows, cols)), dev)
    st = load().nvfp4_quantize(_ptr(x), rows, cols, _ptr(q_packed), _ptr(s_ue4m3), _ptr(gscale),
                               _ptr(workspace), _stream(stream))
    _check(st, "nvfp4_quantize")
    return q_packed, s_ue4m3, gscale


def nvfp4_quantize_grouped(x: torch.Tensor, group_offsets: torch.Tensor, q_packed=None, s_ue4m3=None, gscale=None,
                           workspace=None, stream=None):
    """NVFP4 quantization of row groups of bf16 x[rows][cols], each group with its own global scale
    (include/mx.h, nvfp4_quantize_grouped).  group_offsets: int64 CUDA tensor [G + 1].  Returns
    (q_packed [rows][cols/2] u8, s_ue4m3 flat u8 in the NVFP4 GEMM layout, gscale float[G])."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    if group_offsets.dtype != torch.int64:
        raise ValueError("group_offsets must be int64")
    rows, cols = x.shape
    dev = x.device
    groups = group_offsets.numel() - 1
    if q_packed is None:
        q_packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    if s_ue4m3 is None:
        s_ue4m3 = _u8(mx_scale_bytes(rows, cols, 16, 1, SCALE_UE4M3), dev)
    if gscale is None:
        gscale = torch.empty(max(groups, 1), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _u8(max(16, (4 * groups + 15) // 16 * 16), dev)
    st = load().nvfp4_quantize_grouped(_ptr(x), rows, cols, _ptr(group_offsets), groups, _ptr(q_packed),
                                       _ptr(s_ue4m3), _ptr(gscale), _ptr(workspace), _stream(stream))
    _check(st, "nvfp4_quantize_grouped")
    return q_packed, s_ue4m3, gscale


def nvfp4_quantize_ex(x: torch.Tensor, rht: bool = False, signs: int = 0, rbits=None, q_packed=None,
                      s_ue4m3=None, gscale=None, workspace=None, stream=None):
    """NVFP4 with the 16-point random Hadamard transform (rht, 16-bit sign mask) and/or stochastic
    rounding (rbits: uint8 [rows][cols] random bytes) (include/mx.h, nvfp4_quantize_ex).
    Returns (q_packed, s_ue4m3, gscale) as nvfp4_quantize."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    if q_packed is None:
        q_packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    if s_ue4m3 is None:
        s_ue4m3 = _u8(mx_scale_bytes(rows, cols, 16, 1, SCALE_UE4M3), dev)
    if gscale is None:
        gscale = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _u8(max(16, nvfp4_workspace_bytes(rows, cols)), dev)
    st = load().nvfp4_quantize_ex(_ptr(x), rows, cols, int(bool(rht)), int(signs),
                                  None if rbits is None else _ptr(rbits), _ptr(q_packed), _ptr(s_ue4m3),
                                  _ptr(gscale), _ptr(workspace), _stream(stream))
    _check(st, "nvfp4_quantize_ex")
    return q_packed, s_ue4m3, gscale


def nvfp4_quantize_2d(x: torch.Tensor, out=None, gscale=None, workspace=None, stream=None):
    """NVFP4 with 16x16 blocks, both orientations (include/mx.h, nvfp4_quantize_2d).
    Returns (q_row, s_row, q_col, s_col, gscale)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    rows, cols = x.shape
    dev = x.device
    if out is None:
        out = (torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev),
               _u8(mx_scale_bytes(rows, cols, 16, 1, SCALE_UE4M3), dev),
               torch.empty(cols, rows // 2, dtype=torch.uint8, device=dev),
               _u8(mx_scale_bytes(cols, rows, 16, 1, SCALE_UE4M3), dev))
    if gscale is None:
        gscale = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = _u8(max(16, nvfp4_workspace_bytes(rows, cols)), dev)
    st = load().nvfp4_quantize_2d(_ptr(x), rows, cols, *[_ptr(t) for t in out], _ptr(gscale), _ptr(workspace),
                                  _stream(stream))
    _check(st, "nvfp4_quantize_2d")
    return (*out, gscale)


# ------------------------------------------------------------------ GEMMs
def _out(M, N, out_dtype, out, dev):
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32, device=dev)
    return out, out.stride(0)


def mx_gemm(qa, sa, ea, qb, sb, eb, M, N, K, out_dtype=OUT_BF16, out=None, stream=None):
    """C[m][n] = sum_b sA sB sum_i qA qB (MXFP8, or MXFP4 with packed E2M1 codes; include/mx.h
    mx_gemm)."""
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().mx_gemm(_ptr(qa), _ptr(sa), ea, _ptr(qb), _ptr(sb), eb, M, N, K, out.data_ptr(), out_dtype, ldc,
                        _stream(stream))
    _check(st, "mx_gemm")
    return out


def mx_gemm_mxout(qa, sa, ea, qb, sb, eb, M, N, K, out_elem=E4M3, q_out=None, s_out=None, stream=None):
    """MXFP8 GEMM with the MX quantization of its results fused into the epilogue (include/mx.h,
    mx_gemm_mxout).  Returns (q_out [M][N] u8 codes, s_out flat u8 scales in the MX GEMM layout)."""
    dev = qa.device
    if q_out is None:
        q_out = torch.empty(M, N, dtype=torch.uint8, device=dev)
    if s_out is None:
        s_out = _u8(M * N // 32, dev)
    st = load().mx_gemm_mxout(_ptr(qa), _ptr(sa), ea, _ptr(qb), _ptr(sb), eb, M, N, K, out_elem, _ptr(q_out),
                              _ptr(s_out), q_out.stride(0), _stream(stream))
    _check(st, "mx_gemm_mxout")
    return q_out, s_out


def nvfp4_gemm_grouped(qa, sa, ga, qb, sb, gb, group_offsets, M, N, K, out_dtype=OUT_F32, out=None, stream=None):
    """NVFP4 grouped GEMM (include/mx.h, nvfp4_gemm_grouped): rows off[g] .. off[g+1] of A times the
    g-th [N][K] block of B, scaled by ga * gb[g].  ga: float CUDA tensor [1]; gb: [G]."""
    if group_offsets.dtype != torch.int64:
        raise ValueError("group_offsets must be int64")
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().nvfp4_gemm_grouped(_ptr(qa), _ptr(sa), _ptr(ga), _ptr(qb), _ptr(sb), _ptr(gb), _ptr(group_offsets),
                                   group_offsets.numel() - 1, M, N, K, out.data_ptr(), out_dtype, ldc,
                                   _stream(stream))
    _check(st, "nvfp4_gemm_grouped")
    return out


def nvfp4_gemm_grouped_ex(qa, sa, ga, ga_per_group, qb, sb, gb, group_offsets, M, N, K, out_dtype=OUT_F32, out=None,
                          stream=None):
    """nvfp4_gemm_grouped with one global scale of A per group when ga_per_group (ga: float CUDA
    tensor [G], e.g. from nvfp4_quantize_grouped over the same offsets) (include/mx.h)."""
    if group_offsets.dtype != torch.int64:
        raise ValueError("group_offsets must be int64")
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().nvfp4_gemm_grouped_ex(_ptr(qa), _ptr(sa), _ptr(ga), int(bool(ga_per_group)), _ptr(qb), _ptr(sb),
                                      _ptr(gb), _ptr(group_offsets), group_offsets.numel() - 1, M, N, K,
                                      out.data_ptr(), out_dtype, ldc, _stream(stream))
    _check(st, "nvfp4_gemm_grouped_ex")
    return out


def mx_gemm_mxout_ex(qa, sa, ea, qb, sb, eb, M, N, K, out_elem=E4M3, layout=BOTH, q_row=None, s_row=None,
                     q_col=None, s_col=None, stream=None):
    """MXFP8 GEMM with row-wise and / or column-wise MX quantization of its results in the epilogue
    (include/mx.h, mx_gemm_mxout_ex).  Returns (q_row [M][N], s_row, q_col [N][M], s_col); copies
    not requested are None; scales are flat uint8 in the MX GEMM layout."""
    dev = qa.device
    row, col = bool(layout & ROWWISE), bool(layout & COLWISE)
    if row and q_row is None:
        q_row = torch.empty(M, N, dtype=torch.uint8, device=dev)
    if row and s_row is None:
        s_row = _u8(M * N // 32, dev)
    if col and q_col is None:
        q_col = torch.empty(N, M, dtype=torch.uint8, device=dev)
    if col and s_col is None:
        s_col = _u8(M * N // 32, dev)
    if not row:
        q_row = s_row = None
    if not col:
        q_col = s_col = None
    st = load().mx_gemm_mxout_ex(_ptr(qa), _ptr(sa), ea, _ptr(qb), _ptr(sb), eb, M, N, K, out_elem, layout,
                                 _ptr(q_row), _ptr(s_row), N, _ptr(q_col), _ptr(s_col), M, _stream(stream))
    _check(st, "mx_gemm_mxout_ex")
    return q_row, s_row, q_col, s_col


def mx_gemm_grouped(qa, sa, ea, qb, sb, eb, group_offsets, M, N, K, out_dtype=OUT_BF16, out=None, stream=None):
    """MXFP8 grouped GEMM (include/mx.h, mx_gemm_grouped): rows off[g] .. off[g+1] of A times the
    g-th [N][K] block of B.  group_offsets: int64 CUDA tensor [G + 1]."""
    if group_offsets.dtype != torch.int64:
        raise ValueError("group_offsets must be int64")
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().mx_gemm_grouped(_ptr(qa), _ptr(sa), ea, _ptr(qb), _ptr(sb), eb, _ptr(group_offsets),
                                group_offsets.numel() - 1, M, N, K, out.data_ptr(), out_dtype, ldc, _stream(stream))
    _check(st, "mx_gemm_grouped")
    return out


def nvfp4_gemm(qa, sa, ga, qb, sb, gb, M, N, K, out_dtype=OUT_F32, out=None, stream=None):
    """C = gA gB sum_b sA sB sum_i qA qB (NVFP4, include/mx.h nvfp4_gemm)."""
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().nvfp4_gemm(_ptr(qa), _ptr(sa), _ptr(ga), _ptr(qb), _ptr(sb), _ptr(gb), M, N, K, out.data_ptr(),
                           out_dtype, ldc, _stream(stream))
    _check(st, "nvfp4_gemm")
    return out


def fp8_blockwise_gemm_grouped(qa, sa, qb, sb, group_offsets, M, N, K, out_dtype=OUT_BF16, out=None, stream=None):
    """DeepSeek FP8 grouped GEMM (include/mx.h, fp8_blockwise_gemm_grouped): rows off[g] .. off[g+1] of
    A times the g-th [N][K] block of B, FP32 promotion every 128 of K.  sa float [K/128][M] (1x128
    tiles), sb float [G*N/128][K/128] (128x128 blocks of the stacked weights)."""
    if group_offsets.dtype != torch.int64:
        raise ValueError("group_offsets must be int64")
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().fp8_blockwise_gemm_grouped(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(group_offsets),
                                           group_offsets.numel() - 1, M, N, K, out.data_ptr(), out_dtype, ldc,
                                           _stream(stream))
    _check(st, "fp8_blockwise_gemm_grouped")
    return out


def fp8_blockwise_gemm(qa, sa, qb, sb, M, N, K, out_dtype=OUT_BF16, out=None, stream=None):
    """DeepSeek FP8 GEMM with FP32 promotion every 128 of K (include/mx.h)."""
    out, ldc = _out(M, N, out_dtype, out, qa.device)
    st = load().fp8_blockwise_gemm(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, out.data_ptr(), out_dtype, ldc,
                                   _stream(stream))
    _check(st, "fp8_blockwise_gemm")
    return out


def mx_check(stream=None) -> int:
    """Synchronize the stream and return the library's device status (MX_OK / MX_ERR_TIMEOUT / ...)."""
    return int(load().mx_check(_stream(stream)))


def num_sms() -> int:
    return int(load().mx_num_sms())
