"""Host threads calling the library at once, each on its own CUDA stream: the first calls of a
process fill per-device caches (SM count, cluster occupancy, shared-memory attributes) that every
thread reads; each thread's quantize + GEMM must still match the CPU oracle exactly (codes and
scales bit for bit, products within 1e-5 * sum |a b|)."""
import threading

import numpy as np
import pytest
import torch

import block_scaled_precision_mx_gb300 as mx
from block_scaled_precision_mx_gb300 import synthetic
import oracle as orc
from tests.layouts import chunked_to_plain
from tests.test_gpu_gemm import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_threads_on_their_own_streams():
    M, N, K = 512, 768, 1024
    inputs = [(synthetic.normal(M, K, 1.0, 10100 + i), synthetic.normal(N, K, 0.05, 10200 + i)) for i in range(4)]
    results, errors = {}, []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            a, b = inputs[i]
            with torch.cuda.stream(s):
                qa, sa, _, _ = mx.mx_quantize(a.cuda(), layout=mx.ROWWISE)
                qb, sb, _, _ = mx.mx_quantize(b.cuda(), layout=mx.ROWWISE)
                y = mx.mx_gemm(qa, sa, mx.E4M3, qb, sb, mx.E4M3, M, N, K, out_dtype=mx.OUT_F32)
                status = mx.mx_check()
            s.synchronize()
            results[i] = (qa.cpu().numpy(), sa.cpu().numpy(), y.cpu().numpy(), status)
        except Exception as e:  # reported below, on the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(4):
        a, b = inputs[i]
        qa, sa, y, status = results[i]
        assert status == mx.MX_OK
        oqa, osa = orc.mx_quantize_rowwise(a, orc.E4M3)
        oqb, osb = orc.mx_quantize_rowwise(b, orc.E4M3)
        assert np.array_equal(qa, oqa) and np.array_equal(chunked_to_plain(sa, M, K // 32), osa), f"thread {i}"
        rows = np.arange(0, M, 37)
        ref, ab = orc.mx_gemm(oqa, osa, orc.E4M3, oqb, osb, orc.E4M3, rows=rows)
        assert_close(y[rows], ref, ab, bf16=False, what=f"thread {i}")
