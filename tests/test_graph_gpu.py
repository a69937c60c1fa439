"""Calls captured into a CUDA graph and replayed.

A call's launches (staging, GEMM, split-K or tail reduction, the host
entry's copies on its side streams) can be captured from a stream and
replayed: the graph keeps the pointers and shapes of the capture and reads
whatever the buffers hold at replay.  What capture does not allow (setting up
the device, growing the per-stream workspace or the host entry's device
copies) the library refuses with GEMM_F32_ERR_CAPTURE before it enqueues
anything, so the first call of a shape on a stream goes before the capture.

Every replay is compared with the oracle on inputs written after the
capture, within 1e-3 + 1e-3 |C_ref|.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle

from . import _gpu
from .test_gemm_gpu import _check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load()
    yield
    torch.cuda.synchronize()
    g.gemm_f32_release()


# (M, N, K, algo, alpha, beta): the two-CTA kernel, K splits (added in a
# cluster, or through the workspace and the reduction kernel: 512^2 x 4096,
# 9 splits), the single-CTA kernel with a clipped output box and a beta
# term, and the CUDA-core kernel
CASES = [(2304, 2304, 512, g.ALGO_AUTO, 1.0, 0.0),
         (600, 700, 5000, g.ALGO_3XTF32, 1.0, 0.0),
         (512, 512, 4096, g.ALGO_3XTF32, 1.0, 0.0),
         (300, 200, 40, g.ALGO_3XTF32, 0.5, -0.75),
         (200, 160, 96, g.ALGO_FFMA, 1.0, 0.0)]


def _enqueue(case, bufs, stream):
    M, N, K, algo, alpha, beta = case
    a, b, c = bufs
    return g.gemm_f32_ex(0, 0, M, N, K, alpha, a.data_ptr(), K, b.data_ptr(), N, beta,
                         c.data_ptr(), N, algo, 0, stream.cuda_stream)


def test_captured_calls_replay_on_new_inputs():
    t = _gpu.torch()
    s = t.cuda.Stream()
    bufs = [tuple(t.zeros(n, device="cuda") for n in ((M, K), (K, N), (M, N)))
            for M, N, K, *_ in CASES]
    # first calls outside the capture: they size this stream's workspace
    for case, bb in zip(CASES, bufs):
        g.check(_enqueue(case, bb, s), "warm-up")
    s.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph, stream=s):
        for case, bb in zip(CASES, bufs):
            g.check(_enqueue(case, bb, s), "captured call")
    rng = np.random.default_rng(7)
    for rep in range(2):
        want = []
        for (M, N, K, _, alpha, beta), (a, b, c) in zip(CASES, bufs):
            A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
            B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
            C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
            a.copy_(t.from_numpy(A))
            b.copy_(t.from_numpy(B))
            c.copy_(t.from_numpy(C0))
            want.append(oracle.ref_gemm_ex(0, 0, M, N, K, alpha, A, K, B, N, beta, C0, N)
                        .reshape(M, N))
        t.cuda.synchronize()
        graph.replay()
        t.cuda.synchronize()
        g.check(g.gemm_f32_device_status(1), "device status")
        for case, (_, _, c), w in zip(CASES, bufs, want):
            _check(c.cpu().numpy(), w, label=f"replay {rep} of {case}")


def test_capture_refuses_to_grow_the_workspace():
    t = _gpu.torch()
    s = t.cuda.Stream()  # a new stream: its workspace is empty
    M = N = K = 3072
    # A 4 bytes off a 16-byte boundary: a padded copy of A, in the workspace
    a = t.rand((M * K + 1,), device="cuda")[1:].view(M, K)
    b = t.rand((K, N), device="cuda")
    c = t.zeros((M, N), device="cuda")
    t.cuda.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph, stream=s):
        st = g.gemm_f32_algo(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, g.ALGO_3XTF32,
                             s.cuda_stream)
        c.add_(1.0)  # the capture goes on after the refusal
    assert st == g.ERR_CAPTURE, g.gemm_f32_status_string(st)
    assert "captured" in g.gemm_f32_status_string(st)
    graph.replay()
    t.cuda.synchronize()
    assert float(c.min()) == 1.0 and float(c.max()) == 1.0, "the refused call enqueued work"
    # once called outside a capture, the same call can be captured
    g.check(g.gemm_f32_algo(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, g.ALGO_3XTF32,
                            s.cuda_stream), "call outside the capture")
    s.synchronize()
    graph2 = t.cuda.CUDAGraph()
    with t.cuda.graph(graph2, stream=s):
        g.check(g.gemm_f32_algo(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                g.ALGO_3XTF32, s.cuda_stream), "captured call")
    c.zero_()
    t.cuda.synchronize()
    graph2.replay()
    t.cuda.synchronize()
    rows = np.arange(0, M, 97)
    cols = (rows * 31) % N
    want = oracle.ref_gemm_entries(a.cpu().numpy(), b.cpu().numpy(), rows, cols)
    _check(c.cpu().numpy()[rows, cols], want, label="replay after the refusal")


def test_replay_after_the_workspace_grew():
    # a later, larger call on the same stream grows its workspace; the buffer
    # the captured graph holds must stay allocated (retired, not freed)
    t = _gpu.torch()
    s = t.cuda.Stream()
    M, N, K = 300, 260, 514  # A's rows not 16-byte strides: its padded copy is in the workspace
    a = t.rand((M, K), device="cuda") - 0.5
    b = t.rand((K, N), device="cuda") - 0.5
    c = t.zeros((M, N), device="cuda")
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_3XTF32, 0, A=a.data_ptr(), B=b.data_ptr(),
                            C=c.data_ptr())
    assert st == 0 and p["workspace_bytes"] > 0, p

    def call():
        return g.gemm_f32_algo(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                               g.ALGO_3XTF32, s.cuda_stream)

    g.check(call(), "warm-up")
    s.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph, stream=s):
        g.check(call(), "captured call")
    # a much larger call on the same stream: its workspace grows past the old one
    big = 4096
    x = t.rand((big, big), device="cuda")
    y = t.empty((big, big), device="cuda")
    g.check(g.gemm_f32_algo(x.data_ptr(), x.data_ptr(), y.data_ptr(), big, big, big,
                            g.ALGO_3XTF32, s.cuda_stream), "large call")
    s.synchronize()
    a.copy_(t.rand((M, K), device="cuda") - 0.5)
    c.zero_()
    t.cuda.synchronize()
    graph.replay()
    t.cuda.synchronize()
    g.check(g.gemm_f32_device_status(1), "device status")
    A = a.cpu().numpy()
    B = b.cpu().numpy()
    _check(c.cpu().numpy(), oracle.ref_gemm(A, B), label="replay after the workspace grew")


@pytest.mark.parametrize("shape", [(2304, 2304, 1024), (1024, 1024, 4096)],
                         ids=["row-panels", "k-panels"])
def test_host_entry_captured(shape):
    # the host-buffer entry: copies on its side streams, joined back into
    # the captured stream (row panels with column blocks, and K panels)
    t = _gpu.torch()
    M, N, K = shape
    s = t.cuda.Stream()
    hA = t.empty((M, K), pin_memory=True)
    hB = t.empty((K, N), pin_memory=True)
    hC = t.empty((M, N), pin_memory=True)
    hA.uniform_(-1, 1)
    hB.uniform_(-1, 1)

    def call():
        return g.gemm_f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K,
                               g.ALGO_AUTO, s.cuda_stream)

    g.check(call(), "warm-up")
    s.synchronize()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph, stream=s):
        g.check(call(), "captured host call")
    rng = np.random.default_rng(11)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    hA.copy_(t.from_numpy(A))
    hB.copy_(t.from_numpy(B))
    hC.fill_(float("nan"))
    graph.replay()
    t.cuda.synchronize()
    g.check(g.gemm_f32_device_status(1), "device status")
    rows = np.concatenate([np.arange(M), np.full(N, M - 1)])
    cols = np.concatenate([(np.arange(M) * 13) % N, np.arange(N)])
    want = oracle.ref_gemm_entries(A, B, rows, cols)
    _check(hC.numpy()[rows, cols], want, label=f"captured host entry {shape}")
