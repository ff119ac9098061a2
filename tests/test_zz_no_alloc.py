"""GPU test of nvfp4_quantize_noalloc, the NVFP4 quantizer for callers that cannot allocate.

Some callers of this library cannot hand it a workspace: a plug-in inside a host process whose
allocator owns all of the GPU's memory, or a launch path that must not call cudaMalloc because
that call synchronizes the device.  nvfp4_quantize_noalloc serves them by keeping its scratch in
a fixed 64 KB array inside libmxgb.so.  These tests call it through the C ABI and check its codes,
block scales and global scale bit for bit (the quantizer's outputs are integer codes, so the bar
is bit equality, as in the other quantizer tests) against the CPU oracle's NVFP4 recipe and
against the workspace-taking nvfp4_quantize:
  * two calls in a row, the first with more rows and a larger maximum than the second, so a
    second call that read stale partial maxima from the shared array would fail;
  * the smallest legal shape (128 x 64: 8 bands of 16 rows, one half-full column tile) and a
    width that ends in a half tile (256 x 192), on a stream of their own;
  * the documented limit of 262144 rows, where every slot of the array is used.

This file is named to be collected last, so that a run stopping at the first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests.layouts import chunked_to_plain

pytestmark = pytest.mark.gpu

MAX_ROWS = 262144


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return mx.load()


def call_noalloc(lib, x, stream):
    rows, cols = x.shape
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    s = torch.empty(mx.mx_scale_bytes(rows, cols, 16, 1, mx.SCALE_UE4M3), dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    st = lib.nvfp4_quantize_noalloc(x.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr(), g.data_ptr(),
                                    stream.cuda_stream)
    assert st == mx.MX_OK, mx.status_string(st)
    return q, s, g


def check(lib, x_host, stream):
    """No-alloc result == oracle == nvfp4_quantize on the same stream, bit for bit."""
    rows, cols = x_host.shape
    x = x_host.cuda()
    torch.cuda.current_stream().synchronize()
    with torch.cuda.stream(stream):
        q, s, g = call_noalloc(lib, x, stream)
        q_ref, s_ref, g_ref = mx.nvfp4_quantize(x, stream=stream)
    assert mx.mx_check(stream) == mx.MX_OK
    oq, osc, og = orc.nv_quantize(x_host)
    assert np.float32(g.item()).view(np.uint32) == np.float32(og).view(np.uint32), "global scale vs oracle"
    assert np.array_equal(q.cpu().numpy(), oq), "codes vs oracle"
    assert np.array_equal(chunked_to_plain(s.cpu().numpy(), rows, cols // 16), osc), "block scales vs oracle"
    assert torch.equal(g, g_ref) and torch.equal(q, q_ref) and torch.equal(s, s_ref), "vs nvfp4_quantize"


def test_noalloc_two_calls_in_a_row(lib):
    first = synthetic.with_sparse_outliers(2048, 1024, 901, factor=500.0)
    second = synthetic.with_sparse_outliers(256, 768, 902)
    assert first.float().abs().max() > second.float().abs().max()
    stream = torch.cuda.current_stream()
    for x in (first, second):
        check(lib, x, stream)


@pytest.mark.parametrize("rows,cols", [(128, 64), (256, 192)])
def test_noalloc_small_shapes_on_a_side_stream(lib, rows, cols):
    stream = torch.cuda.Stream()
    check(lib, synthetic.with_sparse_outliers(rows, cols, 903 + cols), stream)


def test_noalloc_at_the_row_limit(lib):
    # 262144 x 64 bf16 (32 MB): 16384 bands of 16 rows, every slot of the array; the largest
    # element sits in the last band, so a maximum that skipped any band would show
    x = synthetic.with_sparse_outliers(MAX_ROWS, 64, 904)
    x[MAX_ROWS - 3, 17] = 4096.0
    check(lib, x, torch.cuda.current_stream())


def test_noalloc_rejects_inputs_beyond_its_scratch(lib):
    fake = 1 << 20  # never dereferenced: the size check fails first
    st = lib.nvfp4_quantize_noalloc(fake, MAX_ROWS + 128, 64, fake, fake, fake, None)
    assert st == mx.MX_ERR_INVALID_ARG
    st = lib.nvfp4_quantize_noalloc(None, 128, 64, fake, fake, fake, None)
    assert st == mx.MX_ERR_INVALID_ARG
