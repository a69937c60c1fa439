"""Concurrent callers: host threads issuing calls on their own streams.

The library keeps one workspace, one host pipeline and one set of TMA
descriptors per (device, stream) and plans under a lock, so independent
streams must not disturb each other.  Each thread checks its own results
against the oracle.
"""

import threading

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload

from .test_gemm_gpu import _check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load()
    yield
    g.gemm_f32_release()


def test_threads_on_their_own_streams():
    import torch
    shapes = [(1025, 1023, 1000), (300, 260, 3000), (2304, 2304, 512), (512, 512, 512)]
    inputs = [make_workload(2, M=M, N=N, K=K) for M, N, K in shapes]
    refs = [oracle.ref_gemm(A, B) for A, B in inputs]
    results = [None] * len(shapes)
    errors = []

    def worker(i):
        try:
            M, N, K = shapes[i]
            A, B = inputs[i]
            s = torch.cuda.Stream()
            a = torch.from_numpy(A).cuda()
            b = torch.from_numpy(B).cuda()
            c = torch.empty((M, N), device="cuda")
            for rep in range(20):
                algo = (g.ALGO_AUTO, g.ALGO_3XTF32, g.ALGO_FFMA)[rep % 3]
                with torch.cuda.stream(s):
                    c.fill_(float("nan"))
                    g.check(g.gemm_f32_algo(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                            algo, s.cuda_stream), "gemm_f32_algo")
            s.synchronize()
            results[i] = c.cpu().numpy()
        except Exception as e:  # reported by the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    g.check(g.gemm_f32_device_status(1), "device status")
    for i, shape in enumerate(shapes):
        _check(results[i], refs[i], label=f"thread {i} {shape}")


def test_host_entry_from_two_threads():
    import torch
    shapes = [(2048, 1536, 700), (1025, 1023, 1000)]
    inputs = [make_workload(1, M=M, N=N, K=K) for M, N, K in shapes]
    outs = [torch.empty((M, N)).pin_memory() for M, N, _ in shapes]
    errors = []

    def worker(i):
        try:
            M, N, K = shapes[i]
            A, B = inputs[i]
            hA = torch.from_numpy(A).pin_memory()
            hB = torch.from_numpy(B).pin_memory()
            s = torch.cuda.Stream()
            for _ in range(3):
                g.check(g.gemm_f32_host(hA.data_ptr(), hB.data_ptr(), outs[i].data_ptr(), M, N, K,
                                        g.ALGO_AUTO, s.cuda_stream), "gemm_f32_host")
            s.synchronize()
        except Exception as e:
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (M, N, K) in enumerate(shapes):
        A, B = inputs[i]
        _check(outs[i].numpy().copy(), oracle.ref_gemm(A, B), label=f"host thread {i}")
