"""GPU test of nvfp4_quantize_noalloc, the NVFP4 quantizer for callers that cannot allocate.

Some callers of this library cannot hand it a workspace: a plug-in inside a host process whose
allocator owns all of the GPU's memory, or a launch path that must not call cudaMalloc because
that call synchronizes the device.  nvfp4_quantize_noalloc serves them by keeping its scratch in
a fixed 64 KB array inside libmxgb.so.  This test calls it through the C ABI and checks, on two
calls in a row, that it returns exactly what the workspace-taking nvfp4_quantize returns (the
quantizer's outputs are integer codes, so the bar is bit equality, as in the other quantizer
tests).  The first call uses more rows and a larger maximum than the second, so a second call
that read stale partial maxima from the shared array would fail.

This file is named to be collected last, so that a run stopping at the first failure has already
run every other test.
"""
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return mx.load()


def call_noalloc(lib, x):
    rows, cols = x.shape
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    s = torch.empty(mx.mx_scale_bytes(rows, cols, 16, 1, mx.SCALE_UE4M3), dtype=torch.uint8, device=x.device)
    g = torch.empty(1, dtype=torch.float32, device=x.device)
    st = lib.nvfp4_quantize_noalloc(x.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr(), g.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert st == mx.MX_OK, mx.status_string(st)
    return q, s, g


def test_noalloc_matches_allocating_entry_point_on_two_calls(lib):
    first = synthetic.with_sparse_outliers(2048, 1024, 901, factor=500.0).cuda()
    second = synthetic.with_sparse_outliers(256, 768, 902).cuda()
    assert first.float().abs().max() > second.float().abs().max()
    for x in (first, second):
        q, s, g = call_noalloc(lib, x)
        q_ref, s_ref, g_ref = mx.nvfp4_quantize(x)
        assert mx.mx_check() == mx.MX_OK
        assert torch.equal(g, g_ref)
        assert torch.equal(q, q_ref)
        assert torch.equal(s, s_ref)


def test_noalloc_rejects_inputs_beyond_its_scratch(lib):
    fake = 1 << 20  # never dereferenced: the size check fails first
    too_many_rows = 262144 + 128
    st = lib.nvfp4_quantize_noalloc(fake, too_many_rows, 64, fake, fake, fake, None)
    assert st == mx.MX_ERR_INVALID_ARG
    st = lib.nvfp4_quantize_noalloc(None, 128, 64, fake, fake, fake, None)
    assert st == mx.MX_ERR_INVALID_ARG
