"""Checked quantization for the GEMM parity tests.

Every helper quantizes the same seeded bf16 tensor twice -- with the library on the GPU and with
the CPU oracle -- asserts that codes and scales agree bit for bit, and returns both: the device
tensors feed the GPU products, the oracle's arrays feed the reference products.  So no reference
value is computed from anything the CUDA path produced, and every GEMM test also exercises the
quantize -> GEMM pipeline a user runs.  Layout conversions only (see tests/layouts.py); no
arithmetic of the method here.
"""
import numpy as np
import torch

import block_scaled_precision_mx_gb300 as mx
import oracle as orc
from tests.layouts import chunked_to_plain, unpack_fp4

MXFMT = {orc.E4M3: mx.E4M3, orc.E5M2: mx.E5M2, orc.E2M1: mx.E2M1}


def _same(got, ref, what):
    got, ref = np.asarray(got), np.asarray(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{what}: {len(bad)} differ, first at {bad[:3].tolist()}"


def mx_rowwise(x, fmt):
    """MX row-wise: (q, s) on the device, (oq, osc) from the oracle (codes unpacked, scales plain)."""
    rows, cols = x.shape
    q, s, _, _ = mx.mx_quantize(x.cuda(), elem=MXFMT[fmt], layout=mx.ROWWISE)
    oq, osc = orc.mx_quantize_rowwise(x, fmt)
    qn = q.cpu().numpy()
    _same(unpack_fp4(qn) if fmt == orc.E2M1 else qn, oq, "row codes")
    _same(chunked_to_plain(s.cpu().numpy(), rows, cols // 32), osc, "row scales")
    return q, s, oq, osc


def mx_both(x, fmt, block_rows=1):
    """MX row- and column-wise from one call (block_rows 32: 2-D 32x32 blocks)."""
    rows, cols = x.shape
    q, s, qT, sT = mx.mx_quantize(x.cuda(), elem=MXFMT[fmt], block_rows=block_rows, layout=mx.BOTH)
    if block_rows == 1:
        oq, osc = orc.mx_quantize_rowwise(x, fmt)
        oqT, osT = orc.mx_quantize_colwise(x, fmt)
    else:
        # one scale per 32x32 block ([rows/32][cols/32]), carried by every 1x32 block of both
        # copies; the column-wise codes are the transpose of the row-wise ones
        oq, s2 = orc.mx_quantize_2d32(x, fmt)
        osc = np.repeat(s2, 32, axis=0)
        oqT, osT = np.ascontiguousarray(oq.T), np.repeat(s2.T, 32, axis=0)
    _same(q.cpu().numpy(), oq, "row codes")
    _same(chunked_to_plain(s.cpu().numpy(), rows, cols // 32), osc, "row scales")
    _same(qT.cpu().numpy(), oqT, "col codes")
    _same(chunked_to_plain(sT.cpu().numpy(), cols, rows // 32), osT, "col scales")
    return (q, s, qT, sT), (oq, osc, oqT, osT)


def nv(x):
    """NVFP4: (q, s, g) on the device, (oq, osc, og) from the oracle (codes packed)."""
    rows, cols = x.shape
    q, s, g = mx.nvfp4_quantize(x.cuda())
    oq, osc, og = orc.nv_quantize(x)
    _same(q.cpu().numpy(), oq, "codes")
    _same(chunked_to_plain(s.cpu().numpy(), rows, cols // 16), osc, "scales")
    assert np.float32(g.item()).view(np.uint32) == np.float32(og).view(np.uint32), "global scale"
    return q, s, g, oq, osc, og


def ds(x, block_rows, pow2=False):
    """DeepSeek 1x128 (block_rows 1) or 128x128 (block_rows 128) blocks with FP32 scales
    (power-of-two scales when pow2).  Oracle scales come as [rows][K/128] for 1x128 tiles and
    [rows/128][K/128] for 128x128 blocks."""
    sfmt = mx.SCALE_FP32_POW2 if pow2 else mx.SCALE_FP32
    q, s, _, _ = mx.mx_quantize(x.cuda(), block=128, block_rows=block_rows, sfmt=sfmt, layout=mx.ROWWISE)
    if block_rows == 1:
        oq, osc = (orc.ds_quantize_1x128_pow2 if pow2 else orc.ds_quantize_1x128)(x)
        sg = s.cpu().numpy().T
    else:
        oq, osc = (orc.ds_quantize_128x128_pow2 if pow2 else orc.ds_quantize_128x128)(x)
        sg = s.cpu().numpy()
    _same(q.cpu().numpy(), oq, "codes")
    _same(np.ascontiguousarray(sg).view(np.uint32), np.ascontiguousarray(osc).astype(np.float32).view(np.uint32), "scales")
    return q, s, oq, osc
