"""gemm_f32_noalloc: the allocation-free entry point against gemm_f32_algo_splitk.

Some callers cannot let a library allocate device memory while they run (a
program that hands out its whole memory budget from its own pool, or a loop
that cannot absorb cudaFree's device-wide synchronisation).  For them the
library offers gemm_f32_noalloc, whose scratch is a fixed array compiled
into the library.  This test calls it twice in a row through the C ABI and
checks each result against the ordinary entry point's result on the same
inputs, within the parity tolerance used everywhere else.  The file is
named to be collected last and works both alone in a fresh process (where
its first call performs the per-device set-up) and after the other tests.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload

pytestmark = pytest.mark.gpu


def _run(entry, A, B, M, N, K, splits):
    import torch

    a = torch.from_numpy(A).cuda()
    b = torch.from_numpy(B).cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    if entry == "noalloc":
        st = g.gemm_f32_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, splits,
                                s.cuda_stream)
    else:
        st = g.gemm_f32_algo_splitk(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                    g.ALGO_FFMA, splits, s.cuda_stream)
    g.check(st, entry)
    s.synchronize()
    return c.cpu().numpy()


def test_noalloc_matches_the_allocating_entry_point_twice():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available()
    g.load()
    cases = [
        (make_workload(4), 256, 256, 65536, 0),   # deep K: split partials in the scratch
        (make_workload(1), 1025, 1023, 1000, 2),  # ragged: padded B copy plus 2 splits
    ]
    for (A, B), M, N, K, splits in cases:
        got = _run("noalloc", A, B, M, N, K, splits)
        want = _run("alloc", A, B, M, N, K, splits)
        res = oracle.compare(got, want)
        assert res["pass"], f"{M}x{N}x{K}: {res}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    g.load()
    # 64 explicit splits of a 4096-wide output need 64 x 256 x 4096 x 4 bytes
    # of partials, far beyond the fixed scratch: refused before any launch
    st = g.gemm_f32_noalloc(1 << 32, 1 << 36, 1 << 40, 256, 4096, 65536, 64, 0)
    assert st == g.ERR_INVALID_VALUE
