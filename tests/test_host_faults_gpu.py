"""Host-side fault injection: the workspace and descriptor error paths.

The status codes GEMM_F32_ERR_WORKSPACE (-3) and GEMM_F32_ERR_DESCRIPTOR
(-5) replace the exit of the error-check macro of "Lecture 5".  A real
cudaMalloc or cuTensorMapEncodeTiled failure cannot be provoked safely, so
gemm_f32_inject_host_fault makes the next one report failure on the host;
nothing faults on the GPU.  Each test checks that the call returns the code,
writes nothing into or around C (NaN guard bands), leaves no device fault,
and that the next call on the same stream succeeds and matches the oracle.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload, uniform_stream

from . import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load()
    yield
    g.gemm_f32_inject_host_fault(g.INJECT_NONE)
    g.gemm_f32_release()


def _buffers(A, B):
    t = _gpu.torch()
    M, K = A.shape
    N = B.shape[1]
    _, a = _gpu.upload(A)
    _, b = _gpu.upload(B)
    cbuf = t.empty(M * N + 2 * _gpu.GUARD, dtype=t.float32, device="cuda")
    cbuf.view(t.int32).fill_(int(_gpu.SENTINEL_BITS.view(np.int32)))
    return a, b, cbuf, cbuf[_gpu.GUARD:_gpu.GUARD + M * N]


def _untouched(cbuf):
    return bool(np.all(cbuf.cpu().numpy().view(np.uint32) == _gpu.SENTINEL_BITS))


def _call(a, b, c, M, N, K, algo, splits, stream):
    return g.gemm_f32_algo_splitk(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, algo,
                                  splits, stream.cuda_stream)


# FFMA with 8 splits keeps its partials in the workspace; the 3xTF32 call
# needs one for A's padded copy (K = 514: rows not a multiple of 16 bytes)
@pytest.mark.parametrize("algo,splits,K", [(g.ALGO_FFMA, 8, 512), (g.ALGO_3XTF32, 0, 514)],
                         ids=["ffma_split_workspace", "3xtf32_staging_workspace"])
def test_workspace_allocation_failure(algo, splits, K):
    t = _gpu.torch()
    A, B = make_workload(1, M=512, N=512, K=K)
    M, K = A.shape
    N = B.shape[1]
    a, b, cbuf, c = _buffers(A, B)
    s = t.cuda.Stream()  # a stream the library has no workspace for yet
    with t.cuda.stream(s):
        assert g.gemm_f32_inject_host_fault(g.INJECT_WORKSPACE) == g.SUCCESS
        assert _call(a, b, c, M, N, K, algo, splits, s) == g.ERR_WORKSPACE
        s.synchronize()
        assert _untouched(cbuf), "a failed call wrote into or around C"
        assert g.gemm_f32_device_status(0) == g.SUCCESS
        # the injection was one-shot: the same call now allocates and runs
        assert _call(a, b, c, M, N, K, algo, splits, s) == g.SUCCESS
        s.synchronize()
    res = oracle.compare(c.cpu().numpy().reshape(M, N), oracle.ref_gemm(A, B))
    assert res["pass"], res
    assert g.gemm_f32_device_status(1) == g.SUCCESS


@pytest.mark.parametrize("algo", [g.ALGO_FFMA, g.ALGO_3XTF32], ids=["ffma", "3xtf32"])
def test_descriptor_encoding_failure(algo):
    t = _gpu.torch()
    v, _ = uniform_stream(384 * 256 + 256 * 320, 4242)
    A = v[:384 * 256].reshape(384, 256)
    B = v[384 * 256:].reshape(256, 320)
    M, K = A.shape
    N = B.shape[1]
    a, b, cbuf, c = _buffers(A, B)
    s = t.cuda.current_stream()
    assert g.gemm_f32_inject_host_fault(g.INJECT_DESCRIPTOR) == g.SUCCESS
    assert _call(a, b, c, M, N, K, algo, 1, s) == g.ERR_DESCRIPTOR
    s.synchronize()
    assert _untouched(cbuf), "a failed call wrote into or around C"
    assert g.gemm_f32_device_status(0) == g.SUCCESS
    assert _call(a, b, c, M, N, K, algo, 1, s) == g.SUCCESS
    s.synchronize()
    res = oracle.compare(c.cpu().numpy().reshape(M, N), oracle.ref_gemm(A, B))
    assert res["pass"], res
    assert g.gemm_f32_device_status(1) == g.SUCCESS


def test_host_entry_buffer_allocation_failure():
    t = _gpu.torch()
    A, B = make_workload(1, M=300, N=260, K=200)
    M, K = A.shape
    N = B.shape[1]
    Ah = t.from_numpy(A).pin_memory()
    Bh = t.from_numpy(B).pin_memory()
    Ch = t.full((M, N), float("nan")).pin_memory()
    s = t.cuda.Stream()  # no host-entry buffers for this stream yet
    assert g.gemm_f32_inject_host_fault(g.INJECT_WORKSPACE) == g.SUCCESS
    st = g.gemm_f32_host(Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), M, N, K, g.ALGO_AUTO,
                         s.cuda_stream)
    assert st == g.ERR_WORKSPACE
    s.synchronize()
    assert bool(t.isnan(Ch).all()), "a failed call wrote C"
    g.check(g.gemm_f32_host(Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), M, N, K, g.ALGO_AUTO,
                            s.cuda_stream), "gemm_f32_host")
    s.synchronize()
    res = oracle.compare(Ch.numpy(), oracle.ref_gemm(A, B))
    assert res["pass"], res
