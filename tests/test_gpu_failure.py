"""The failure path of the device-side waits, on the GPU, without a fault: a bounded wait that
nothing satisfies runs out, the kernel returns, mx_check() reports MX_ERR_TIMEOUT once (and
clears the word), and the context keeps working."""
import time

import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests import quantized

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_bounded_wait_runs_out_and_reports_timeout():
    assert mx.mx_check() == mx.MX_OK
    t0 = time.time()
    mx.mx_selftest_wait_timeout(20000)            # 20 ms budget
    assert mx.mx_check() == mx.MX_ERR_TIMEOUT
    assert time.time() - t0 < 5.0
    assert mx.mx_check() == mx.MX_OK              # reported once, then cleared
    # the context still works: a quantize + GEMM right after match the oracle
    a = synthetic.normal(256, 256, 1.0, 9100)
    b = synthetic.normal(256, 256, 0.02, 9101)
    qa, sa, oqa, osa = quantized.mx_rowwise(a, orc.E4M3)
    qb, sb, oqb, osb = quantized.mx_rowwise(b, orc.E4M3)
    y = mx.mx_gemm(qa, sa, mx.E4M3, qb, sb, mx.E4M3, 256, 256, 256, out_dtype=mx.OUT_F32)
    assert mx.mx_check() == mx.MX_OK
    ref, ab = orc.mx_gemm(oqa, osa, orc.E4M3, oqb, osb, orc.E4M3)
    assert (np.abs(y.cpu().numpy() - ref) <= 1e-5 * ab + 1e-30).all()


def test_timeout_reports_do_not_accumulate_across_streams():
    s = torch.cuda.Stream()
    mx.mx_selftest_wait_timeout(1000, stream=s)
    assert mx.mx_check(s) == mx.MX_ERR_TIMEOUT
    assert mx.mx_check() == mx.MX_OK
