"""CPU oracle for block-scaled quantization and block-scaled GEMMs.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``block_scaled_precision_mx_gb300``) never imports it, and this package never
imports the product path: the two share no code.

The arithmetic lives in ``mx_oracle.c`` (plain C, double precision except for
the steps the method fixes in FP32).  This module only compiles it with gcc and
marshals numpy arrays through ctypes.  Plain (un-swizzled) layouts are used
throughout: scales are ``[rows][cols / block]`` row-major arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_LIB = os.path.join(_HERE, "libmx_oracle.so")
_lock = threading.Lock()
_lib = None

E4M3, E5M2, E2M1, E8M0 = 0, 1, 2, 3
FMT = {"e4m3": E4M3, "e5m2": E5M2, "e2m1": E2M1, "e8m0": E8M0}


def build(force: bool = False) -> str:
    """Compile mx_oracle.c into libmx_oracle.so (gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, u32, f32, f64, i32 = (ctypes.c_int64, ctypes.c_uint32, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_int)
            p = ctypes.c_void_p
            sig = {
                "orc_decode": (f64, [i32, u32]),
                "orc_encode": (u32, [i32, f64]),
                "orc_encode_bruteforce": (u32, [i32, f64]),
                "orc_emax": (i32, [i32]),
                "orc_bf16": (f64, [ctypes.c_uint16]),
                "orc_mx_scale_exp": (i32, [f64, i32]),
                "orc_mx_quantize_rowwise": (None, [p, i64, i64, i32, p, p]),
                "orc_mx_quantize_colwise": (None, [p, i64, i64, i32, p, p]),
                "orc_ds_scale": (f32, [f32]),
                "orc_ds_encode": (ctypes.c_uint8, [f32, f32]),
                "orc_ds_quantize_1x128": (None, [p, i64, i64, p, p]),
                "orc_ds_quantize_128x128": (None, [p, i64, i64, p, p]),
                "orc_nv_global_scale": (f32, [f32]),
                "orc_nv_block_scale": (ctypes.c_uint8, [f32, f32, ctypes.POINTER(f32)]),
                "orc_nv_encode": (ctypes.c_uint8, [f32, f32]),
                "orc_nv_amax": (f32, [p, i64]),
                "orc_nv_quantize": (None, [p, i64, i64, p, p, ctypes.POINTER(f32)]),
                "orc_mx_gemm": (None, [p, p, i32, p, p, i32, i64, i64, i64, p, i64, p, p]),
                "orc_nv_gemm": (None, [p, p, f32, p, p, f32, i64, i64, i64, p, i64, p, p]),
                "orc_ds_gemm": (None, [p, p, p, p, i64, i64, i64, p, i64, p, p]),
                "orc_num_threads": (i32, []),
                "orc_pow2_scale_exp": (i32, [f64]),
                "orc_ds_quantize_1x128_pow2": (None, [p, i64, i64, p, p]),
                "orc_ds_quantize_128x128_pow2": (None, [p, i64, i64, p, p]),
                "orc_e8m0_of_scale": (ctypes.c_uint8, [f32]),
                "orc_mx_scales_from_blocks": (None, [p, i64, i64, i32, p]),
                "orc_mx_quantize_2d32": (None, [p, i64, i64, i32, p, p]),
                "orc_fwht16_f32": (None, [p, u32]),
                "orc_e2m1_stochastic": (ctypes.c_uint8, [f32, ctypes.c_uint8]),
                "orc_nv_quantize_ex": (None, [p, i64, i64, i32, u32, p, p, p, ctypes.POINTER(f32)]),
                "orc_nv_quantize_2d16": (None, [p, i64, i64, p, p, ctypes.POINTER(f32)]),
                "orc_mx_quantize_rowwise_f32": (None, [p, i64, i64, i32, p, p]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a uint16 bit array, or a torch bf16 tensor (CPU) -> uint16 array."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # plain CPU tensor plumbing only
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ---------------------------------------------------------------- formats
def decode(fmt: int, code: int) -> float:
    return _load().orc_decode(fmt, code)


def encode(fmt: int, v: float) -> int:
    return _load().orc_encode(fmt, v)


def encode_bruteforce(fmt: int, v: float) -> int:
    return _load().orc_encode_bruteforce(fmt, v)


def emax(fmt: int) -> int:
    return _load().orc_emax(fmt)


def bf16_value(bits: int) -> float:
    return _load().orc_bf16(bits)


def mx_scale_exp(amax: float, fmt: int) -> int:
    return _load().orc_mx_scale_exp(amax, fmt)


def num_threads() -> int:
    return _load().orc_num_threads()


# ---------------------------------------------------------------- MX
def mx_quantize_rowwise(x, fmt: int):
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    _load().orc_mx_quantize_rowwise(_ptr(xb), rows, cols, fmt, _ptr(q), _ptr(s))
    return q, s


def mx_quantize_rowwise_f32(x, fmt: int):
    """Row-wise MX quantization of FP32 values x[rows][cols]: (q, s [rows][cols/32])."""
    xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    rows, cols = xf.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    _load().orc_mx_quantize_rowwise_f32(_ptr(xf), rows, cols, fmt, _ptr(q), _ptr(s))
    return q, s


def mx_quantize_colwise(x, fmt: int):
    """Returns (qT [cols][rows], sT [cols][rows/32])."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((cols, rows), np.uint8)
    s = np.empty((cols, rows // 32), np.uint8)
    _load().orc_mx_quantize_colwise(_ptr(xb), rows, cols, fmt, _ptr(q), _ptr(s))
    return q, s


# ---------------------------------------------------------------- DeepSeek
def ds_scale(amax: float) -> float:
    return _load().orc_ds_scale(amax)


def ds_encode(x: float, s: float) -> int:
    return _load().orc_ds_encode(x, s)


def ds_quantize_1x128(x):
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    _load().orc_ds_quantize_1x128(_ptr(xb), rows, cols, _ptr(q), _ptr(s))
    return q, s


def ds_quantize_128x128(x):
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 128, cols // 128), np.float32)
    _load().orc_ds_quantize_128x128(_ptr(xb), rows, cols, _ptr(q), _ptr(s))
    return q, s


# ---------------------------------------------------------------- power-of-two blocks, 2-D MX
def pow2_scale_exp(amax: float) -> int:
    return _load().orc_pow2_scale_exp(amax)


def ds_quantize_1x128_pow2(x):
    """1x128 tiles, power-of-two FP32 scales: (q [rows][cols], s [rows][cols/128])."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    _load().orc_ds_quantize_1x128_pow2(_ptr(xb), rows, cols, _ptr(q), _ptr(s))
    return q, s


def ds_quantize_128x128_pow2(x):
    """128x128 blocks, power-of-two FP32 scales: (q [rows][cols], s [rows/128][cols/128])."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 128, cols // 128), np.float32)
    _load().orc_ds_quantize_128x128_pow2(_ptr(xb), rows, cols, _ptr(q), _ptr(s))
    return q, s


def e8m0_of_scale(sc: float) -> int:
    return _load().orc_e8m0_of_scale(sc)


def mx_scales_from_blocks(s, rows: int, cols: int, block_rows: int):
    """Per-32 E8M0 codes [rows][cols/32] from 1x128 (s [rows][cols/128]) or 128x128
    (s [rows/128][cols/128]) power-of-two FP32 block scales; 0xFF where a scale is not 2^k."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    out = np.empty((rows, cols // 32), np.uint8)
    _load().orc_mx_scales_from_blocks(_ptr(s), rows, cols, block_rows, _ptr(out))
    return out


def mx_quantize_2d32(x, fmt: int):
    """2-D 32x32 MX blocks: (q [rows][cols], s [rows/32][cols/32])."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 32, cols // 32), np.uint8)
    _load().orc_mx_quantize_2d32(_ptr(xb), rows, cols, fmt, _ptr(q), _ptr(s))
    return q, s


# ---------------------------------------------------------------- NVFP4
def nv_global_scale(amax: float) -> float:
    return _load().orc_nv_global_scale(amax)


def nv_block_scale(sg: float, bamax: float):
    sh = ctypes.c_float(0.0)
    code = _load().orc_nv_block_scale(sg, bamax, ctypes.byref(sh))
    return code, sh.value


def nv_encode(x: float, s_hat: float) -> int:
    return _load().orc_nv_encode(x, s_hat)


def nv_quantize(x):
    """Returns (q_packed [rows][cols/2], s [rows][cols/16] E4M3 codes, s_global)."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols // 2), np.uint8)
    s = np.empty((rows, cols // 16), np.uint8)
    sg = ctypes.c_float(0.0)
    _load().orc_nv_quantize(_ptr(xb), rows, cols, _ptr(q), _ptr(s), ctypes.byref(sg))
    return q, s, sg.value


# ---------------------------------------------------------------- NVFP4 training options
def fwht16(v, signs: int = 0):
    """FP32 16-point transform 0.25 * H16 * (d .* v) in the fixed butterfly order."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).copy())
    _load().orc_fwht16_f32(_ptr(a), signs)
    return a


def e2m1_stochastic(y: float, r: int) -> int:
    return _load().orc_e2m1_stochastic(y, r)


def nv_quantize_ex(x, rht: bool = False, signs: int = 0, rbits=None):
    """NVFP4 with the transform and/or stochastic rounding: (codes [rows][cols] unpacked,
    s [rows][cols/16], s_global)."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 16), np.uint8)
    sg = ctypes.c_float(0.0)
    rb = None if rbits is None else np.ascontiguousarray(rbits, dtype=np.uint8)
    _load().orc_nv_quantize_ex(_ptr(xb), rows, cols, int(bool(rht)), signs, None if rb is None else _ptr(rb),
                               _ptr(q), _ptr(s), ctypes.byref(sg))
    return q, s, sg.value


def nv_quantize_2d16(x):
    """NVFP4 with 16x16 blocks: (codes [rows][cols] unpacked, s [rows/16][cols/16], s_global)."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 16, cols // 16), np.uint8)
    sg = ctypes.c_float(0.0)
    _load().orc_nv_quantize_2d16(_ptr(xb), rows, cols, _ptr(q), _ptr(s), ctypes.byref(sg))
    return q, s, sg.value


# ---------------------------------------------------------------- GEMMs
def _rows(rows, M):
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def mx_gemm(qa, sa, fa, qb, sb, fb, rows=None):
    """y[i][n] = sum_k A[rows[i]][k] B[n][k] for MX operands; returns (y, absum)."""
    M, K = qa.shape
    N = qb.shape[0]
    r = _rows(rows, M)
    out = np.empty((len(r), N), np.float64)
    ab = np.empty((len(r), N), np.float64)
    _load().orc_mx_gemm(_ptr(np.ascontiguousarray(qa)), _ptr(np.ascontiguousarray(sa)), fa,
                        _ptr(np.ascontiguousarray(qb)), _ptr(np.ascontiguousarray(sb)), fb,
                        M, N, K, _ptr(r), len(r), _ptr(out), _ptr(ab))
    return out, ab


def nv_gemm(qa, sa, sga, qb, sb, sgb, rows=None):
    M, Kh = qa.shape
    N = qb.shape[0]
    r = _rows(rows, M)
    out = np.empty((len(r), N), np.float64)
    ab = np.empty((len(r), N), np.float64)
    _load().orc_nv_gemm(_ptr(np.ascontiguousarray(qa)), _ptr(np.ascontiguousarray(sa)), sga,
                        _ptr(np.ascontiguousarray(qb)), _ptr(np.ascontiguousarray(sb)), sgb,
                        M, N, 2 * Kh, _ptr(r), len(r), _ptr(out), _ptr(ab))
    return out, ab


def ds_gemm(qa, sa, qb, sb, rows=None):
    M, K = qa.shape
    N = qb.shape[0]
    r = _rows(rows, M)
    out = np.empty((len(r), N), np.float64)
    ab = np.empty((len(r), N), np.float64)
    _load().orc_ds_gemm(_ptr(np.ascontiguousarray(qa)), _ptr(np.ascontiguousarray(sa, dtype=np.float32)),
                        _ptr(np.ascontiguousarray(qb)), _ptr(np.ascontiguousarray(sb, dtype=np.float32)),
                        M, N, K, _ptr(r), len(r), _ptr(out), _ptr(ab))
    return out, ab
