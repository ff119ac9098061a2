"""Test-side layout conversions between the library's scale layouts and the oracle's plain ones.

These are index permutations only (no arithmetic of the method): the library stores MX / NVFP4
scales in 512-byte chunks of 128 rows x 4 blocks (byte (i % 32) * 16 + (i // 32) * 4 + j inside
the chunk, chunks ordered [row block][k chunk]) and DeepSeek 1x128 scales k-block-major.
"""
import numpy as np


def chunked_to_plain(flat, rows, nblocks):
    """flat chunk-layout scale bytes -> plain [rows][nblocks] (nblocks % 4 == 0)."""
    a = np.asarray(flat).reshape(rows // 128, nblocks // 4, 32, 4, 4)
    return np.ascontiguousarray(a.transpose(0, 3, 2, 1, 4).reshape(rows, nblocks))


def plain_to_chunked(plain):
    """plain [rows][nblocks] -> flat chunk-layout bytes."""
    rows, nblocks = plain.shape
    a = np.asarray(plain).reshape(rows // 128, 4, 32, nblocks // 4, 4)
    return np.ascontiguousarray(a.transpose(0, 3, 2, 1, 4).reshape(-1))


def unpack_fp4(qp):
    """packed [rows][cols/2] -> codes [rows][cols] (element 2i in the low nibble)."""
    qp = np.asarray(qp)
    return np.stack([qp & 0xF, qp >> 4], axis=-1).reshape(qp.shape[0], -1)


def pack_fp4(codes):
    """codes [rows][cols] (4-bit values) -> packed [rows][cols/2], element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return np.ascontiguousarray(c[:, 0::2] | (c[:, 1::2] << 4))
