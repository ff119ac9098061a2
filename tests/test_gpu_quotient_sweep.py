"""Divisor sweeps of the quantizers whose codes round an FP32 quotient.

The DeepSeek recipe ("Why FP8 training is stable" (magicnetworld.com), sec 4-5: s = amax / 448,
q = E4M3(fl32(x / s))) and the NVFP4 recipe ("NVFP4: high accuracy with 4 bits" (theluyuan.com),
sec 5.4: s_hat = dec(E4M3(fl32(fl32(bamax / 6) / s_g))) * s_g, q = E2M1(fl32(x / s_hat))) define
each code as the rounding of an FP32 quotient.  The kernels decide most codes without dividing
(a reciprocal bracket) and divide only near a rounding boundary; these tests show on many divisors
that the result equals the oracle's, which divides every element, bit for bit:
  * DeepSeek 1x128 tiles: s = fl32(amax / 448) for all 128 bf16 mantissas of amax in five binades
    (two with s an FP32 subnormal, where the kernels must divide), each against every bf16 value x
    with amax * 2^-20 <= |x| <= amax (both signs); the same sweep through 128x128 weight blocks;
  * NVFP4: 32 global scales s_g (32 mantissas of the global amax) with, for each, block maxima that
    give every E4M3 block-scale code, i.e. at least 8 x 32 = 256 divisors s_hat per binade, each
    against every bf16 x with bamax * 2^-6 <= |x| <= bamax (both signs); plus tensors whose s_g,
    or whose smaller s_hat, is an FP32 subnormal.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from tests import quantized

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


POS = np.arange(0x7F80, dtype=np.uint32)               # every finite non-negative bf16 bit pattern
POS_VAL = (POS << 16).view(np.float32).astype(np.float64)


def bf16_in(lo, hi):
    """bit patterns of every bf16 v with lo <= v <= hi (v >= 0), both signs."""
    b = POS[(POS_VAL >= lo) & (POS_VAL <= hi)].astype(np.uint16)
    return np.concatenate([b, b | 0x8000])


def to_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bf16_bits_of(v):
    """nearest bf16 bit pattern of positive float64 values (round half to even on the FP32 bits)."""
    f = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def fill_blocks(anchors, values_of, width):
    """Blocks of `width` elements: the anchor first (the block's largest magnitude), then the
    values values_of(anchor) in order, as many blocks per anchor as they need (zero padded)."""
    out = []
    for a in anchors:
        v = values_of(a)
        n = -(-len(v) // (width - 1))
        v = np.concatenate([v, np.zeros(n * (width - 1) - len(v), np.uint16)]).reshape(n, width - 1)
        anc = np.full((n, 1), a, np.uint16)
        out.append(np.concatenate([anc, v], axis=1))
    return np.concatenate(out)


def as_matrix(blocks, cols):
    flat = blocks.reshape(-1)
    rows = -(-len(flat) // cols)
    rows = -(-rows // 128) * 128
    m = np.zeros(rows * cols, np.uint16)
    m[: len(flat)] = flat
    return m.reshape(rows, cols)


# ------------------------------------------------------------------ DeepSeek (E4M3 of x / s)
# amax binades: [1, 2), [2^-3, 2^-2), [2^10, 2^11), and two whose s = amax / 448 is an FP32
# subnormal ([2^-120, 2^-119): bf16 normal; [2^-129, 2^-128): a bf16 subnormal amax)
DS_BINADES = (0, -3, 10, -120, -129)


def ds_anchors():
    out = []
    for e in DS_BINADES:
        lo = 2.0 ** e
        b = POS[(POS_VAL >= lo) & (POS_VAL < 2 * lo)].astype(np.uint16)
        out.append(b)
    return np.concatenate(out)


def ds_values(a):
    amax = float(POS_VAL[a])
    return bf16_in(amax * 2.0 ** -20, amax)


def test_deepseek_1x128_divisor_sweep():
    anchors = ds_anchors()
    assert len(anchors) >= 4 * 128
    blocks = fill_blocks(anchors, ds_values, 128)
    x = to_bf16(as_matrix(blocks, 1024))
    _, _, oq, osc = quantized.ds(x, 1)            # codes and scales bit-exact against the oracle
    s = osc.reshape(-1)
    assert (s[s > 0] < np.float32(2.0 ** -126)).sum() > 100, "subnormal scales not exercised"


def test_deepseek_128x128_divisor_sweep():
    # one 128x128 block per amax: the anchor and every test value inside it
    anchors = ds_anchors()[::4]                   # 160 amax values, 32 mantissas per binade
    blocks = []
    for a in anchors:
        v = ds_values(a)
        blk = np.zeros(128 * 128, np.uint16)
        blk[0] = a
        blk[1: 1 + len(v)] = v
        blocks.append(blk.reshape(128, 128))
    nb = len(blocks)
    per_row = 16
    while nb % per_row:
        blocks.append(np.zeros((128, 128), np.uint16))
        nb += 1
    grid = np.block([[blocks[r * per_row + c] for c in range(per_row)] for r in range(nb // per_row)])
    _, _, oq, osc = quantized.ds(to_bf16(grid), 128)
    s = osc.reshape(-1)
    assert (s[s > 0] < np.float32(2.0 ** -126)).sum() > 10, "subnormal scales not exercised"


# ------------------------------------------------------------------ NVFP4 (E2M1 of x / s_hat)
E4M3_VALUES = np.array([orc.decode(orc.E4M3, c) for c in range(1, 0x7F)])   # positive finite codes


def nv_tensor(gamax):
    """One tensor with global amax `gamax` (bf16 bits): for every E4M3 block-scale code, block
    maxima near dec(code) * 6 * s_g (the bf16 value nearest it and its two neighbours), each block
    followed by every bf16 x with bamax * 2^-6 <= |x| <= bamax."""
    g = float(POS_VAL[gamax])
    sg = float(np.float32(np.float32(g) / np.float32(2688.0)))
    targets = bf16_bits_of(E4M3_VALUES * 6.0 * sg)
    cand = np.unique(np.concatenate([targets - 1, targets, targets + 1]).astype(np.int64))
    cand = cand[(cand > 0) & (cand < gamax)].astype(np.uint16)
    anchors = np.concatenate([[gamax], cand]).astype(np.uint16)
    blocks = fill_blocks(anchors, lambda a: bf16_in(float(POS_VAL[a]) * 2.0 ** -6, float(POS_VAL[a])), 16)
    return to_bf16(as_matrix(blocks, 1024))


def nv_check(gamax, want_codes):
    x = nv_tensor(gamax)
    _, _, _, _, osc, og = quantized.nv(x)         # codes, scales and global scale bit-exact
    codes = np.unique(osc)
    assert len(set(codes.tolist()) & set(range(1, 0x7F))) >= want_codes, len(codes)
    return og


@pytest.mark.parametrize("m", range(0, 128, 4))
def test_nvfp4_divisor_sweep_global_scales(m):
    # global amax 2^3 * (1 + m / 128): 32 global scales; every block-scale code at each
    nv_check(np.uint16((130 << 7) | m), want_codes=120)


@pytest.mark.parametrize("gexp,m", [(-116, 5), (-118, 77), (-110, 33)])
def test_nvfp4_divisor_sweep_tiny_global_amax(gexp, m):
    # global amax 2^-116 (1 + m/128), 2^-118 (...): s_g = amax / 2688 is an FP32 subnormal (the
    # kernels divide every element); 2^-110: s_g is normal and the smaller s_hat = dec(code) * s_g
    # are subnormal
    og = nv_check(np.uint16(((127 + gexp) << 7) | m), want_codes=20)
    assert og > 0
    assert (og < 2.0 ** -126) == (gexp <= -116), og
