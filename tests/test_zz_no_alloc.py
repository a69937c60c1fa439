"""gemm_f32_noalloc: the allocation-free entry point, against the oracle.

Some callers cannot let a library allocate device memory while they run: a
program that reserves its whole memory budget up front and hands it out from
its own pool, or a loop that cannot absorb cudaFree's device-wide
synchronisation.  For them the library offers gemm_f32_noalloc, whose scratch
is a fixed array compiled into the library.  These tests call it twice in a
row through the C ABI on each case and check every result against the CPU
oracle elementwise, within the tolerance used everywhere else
(|C - C_ref| <= 1e-3 + 1e-3 |C_ref|, "Lecture 12: final project", section 4),
and bit for bit against the allocating entry point's CUDA-core kernel with
the same split count (each output is summed in ascending k within a split and
the splits are added in split order on both paths).  The cases stage A, B or
both into the fixed array (a row stride or base address TMA cannot describe)
as well as the split partials.  A watchdog self-test aimed at the array's
fault word checks that a timeout in this entry point's kernels is reported by
gemm_f32_device_status and cleared by it.

The file is named to be collected last; it works alone in a fresh process
(where its first call performs the per-device set-up) and after the others.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload, uniform_stream

from . import _gpu

pytestmark = pytest.mark.gpu


def _call(entry, A, B, splits, offsets=(0, 0, 0)):
    """One call of `entry` on device copies of A and B (each `offsets` floats
    into its buffer), with NaN guard bands around C; returns C."""
    t = _gpu.torch()
    M, K = A.shape
    N = B.shape[1]
    _, a = _gpu.upload(A, offsets[0])
    _, b = _gpu.upload(B, offsets[1])
    cbuf = t.empty(M * N + 2 * _gpu.GUARD + offsets[2], dtype=t.float32, device="cuda")
    cbuf.view(t.int32).fill_(int(_gpu.SENTINEL_BITS.view(np.int32)))
    lo = _gpu.GUARD + offsets[2]
    c = cbuf[lo:lo + M * N]
    s = t.cuda.current_stream()
    if entry == "noalloc":
        st = g.gemm_f32_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, splits,
                                s.cuda_stream)
    else:
        st = g.gemm_f32_algo_splitk(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                    g.ALGO_FFMA, splits, s.cuda_stream)
    g.check(st, entry)
    s.synchronize()
    g.check(g.gemm_f32_device_status(1), "device status")
    host = cbuf.cpu().numpy()
    assert np.all(host[:lo].view(np.uint32) == _gpu.SENTINEL_BITS), "write before C"
    assert np.all(host[lo + M * N:].view(np.uint32) == _gpu.SENTINEL_BITS), "write after C"
    return host[lo:lo + M * N].reshape(M, N).copy()


def _uniform(M, N, K, seed):
    v, _ = uniform_stream(M * K + K * N, seed)
    return v[:M * K].reshape(M, K), v[M * K:].reshape(K, N)


# (label, inputs, explicit split count, operand offsets in floats)
CASES = [
    # deep K: only the split partials live in the scratch
    ("deep_k_256x256x65536", lambda: make_workload(4), 8, (0, 0, 0)),
    # ragged: N % 4 != 0 stages B, two splits
    ("ragged_1025x1023x1000", lambda: make_workload(1), 2, (0, 0, 0)),
    # K % 4 != 0 and N % 4 != 0: both A and B staged, then the partials
    ("staged_a_and_b_97x130x1001", lambda: _uniform(97, 130, 1001, 97), 2, (0, 0, 0)),
    # A's base 4 bytes off a 16-byte boundary: A staged although K % 4 == 0
    ("misaligned_a_200x256x1000", lambda: _uniform(200, 256, 1000, 200), 3, (1, 0, 0)),
]


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load()
    yield


@pytest.mark.parametrize("label,make,splits,offsets", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_the_oracle_twice(label, make, splits, offsets):
    A, B = make()
    want = oracle.ref_gemm(A, B)
    alloc = _call("alloc", A, B, splits, offsets)
    for call in range(2):
        got = _call("noalloc", A, B, splits, offsets)
        res = oracle.compare(got, want)
        assert res["pass"], f"{label} call {call}: {res}"
        assert np.array_equal(got.view(np.uint32), alloc.view(np.uint32)), \
            f"{label} call {call}: differs from the allocating path with {splits} splits"


def test_noalloc_automatic_splits_match_the_oracle_twice():
    A, B = make_workload(4)
    want = oracle.ref_gemm(A, B)
    for call in range(2):
        res = oracle.compare(_call("noalloc", A, B, 0), want)
        assert res["pass"], f"call {call}: {res}"


def test_noalloc_timeout_is_reported_then_cleared():
    # a barrier nothing completes, 20 ms limit, on the no-alloc fault word
    assert g.gemm_f32_noalloc_selftest_watchdog(20_000_000) == g.ERR_DEVICE_TIMEOUT
    assert g.gemm_f32_device_status(0) == g.ERR_DEVICE_TIMEOUT  # reported, kept
    assert g.gemm_f32_device_status(1) == g.ERR_DEVICE_TIMEOUT  # reported, cleared
    assert g.gemm_f32_device_status(0) == g.SUCCESS
    # the context is usable and the next call runs clean
    A, B = make_workload(1)
    res = oracle.compare(_call("noalloc", A, B, 2), oracle.ref_gemm(A, B))
    assert res["pass"], res
    assert g.gemm_f32_device_status(0) == g.SUCCESS


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 64 explicit splits of a 4096-wide output need 64 x 256 x 4096 x 4 bytes
    # of partials, far beyond the fixed scratch: refused before any launch
    st = g.gemm_f32_noalloc(1 << 32, 1 << 36, 1 << 40, 256, 4096, 65536, 64, 0)
    assert st == g.ERR_INVALID_VALUE
