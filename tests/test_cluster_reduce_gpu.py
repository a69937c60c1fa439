"""GPU parity of the CUDA-core kernel's in-cluster split-K reduction: for
2..4 K splits the splits of one output tile run as a thread-block cluster
and add their partial tiles through distributed shared memory, split 0
first, with no workspace and no reduction kernel.

Against the oracle within 1e-3 + 1e-3 |C_ref| (NaN guard bands around C);
against the workspace reduction (gemm_f32_noalloc: same kernel, partials in
a scratch array, summed by the reduction kernel in the same split order),
bit for bit.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload

from . import _gpu
from .test_gemm_gpu import _check, _ex_case

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 16 << 20  # GEMM_F32_NOALLOC_SCRATCH_BYTES in gemm_f32.h


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load()
    yield
    g.gemm_f32_release()


@pytest.mark.parametrize("splits,want", [(2, 1), (3, 1), (4, 1), (5, 0), (8, 0), (1, 0)])
def test_plan(splits, want):
    M, N, K = 300, 260, 4000
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_FFMA, splits, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["cluster_reduce"] == want, p
    if want:
        assert p["workspace_bytes"] == 0 and p["kernels"] == 1, p


def test_auto_reduces_in_cluster():
    # the CUDA-core plan for 1000 x 1000 x 250 (64 tiles): 4 splits, in a cluster
    M, N, K = 1000, 1000, 250
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_FFMA, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["splits"] == 4 and p["cluster_reduce"] == 1
    A, B = make_workload(2, M=M, N=N, K=K)
    _check(_gpu.run(A, B, g.ALGO_FFMA), oracle.ref_gemm(A, B), label="ffma 1000x1000x250")
    # AUTO's choice there for a transposed A (staged operands: the split and
    # transpose in one pass): the staged tensor-core kernel, 2 splits, in a
    # cluster
    st, p = g.gemm_f32_plan_ex(1, 0, M, N, K, M, N, N, g.ALGO_AUTO)
    assert st == 0 and p["algo"] == g.ALGO_3XTF32 and p["splits"] == 2 and p["cluster_reduce"] == 1
    _ex_case(M, N, K, 1, 0, 0, 1.0, 0.0, g.ALGO_AUTO)
    # A's base 4 bytes off a 16-byte boundary: a padded copy of A, then the
    # kernel with B's split in tensor memory
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=(1 << 32) + 4, B=1 << 36, C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and p["stage_a"] == 1, p
    _check(_gpu.run(A, B, g.ALGO_AUTO, offsets=(1, 0, 0)), oracle.ref_gemm(A, B),
           label="auto 1000x1000x250, A misaligned")
    _check(_gpu.run(A, B, g.ALGO_AUTO), oracle.ref_gemm(A, B), label="auto 1000x1000x250")


@pytest.mark.parametrize("splits", [2, 3, 4, 8])
@pytest.mark.parametrize("shape", [(300, 260, 4000), (129, 1000, 2049), (1025, 1023, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_parity_and_equal_to_workspace_reduction(shape, splits):
    M, N, K = shape
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run(A, B, g.ALGO_FFMA, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"cluster reduce {shape} s{splits}")
    # the workspace path of the same kernel (narrow tiles at these sizes),
    # where its partials and padded copies fit the no-allocation scratch
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_FFMA, splits, A=1 << 32, B=1 << 36, C=1 << 40)
    assert p["tile_n"] == 128
    ld4 = lambda x: (x + 3) // 4 * 4
    need = 4 * (splits * M * ld4(N) + (M * ld4(K) if K % 4 else 0) + (K * ld4(N) if N % 4 else 0))
    if need > NOALLOC_SCRATCH_BYTES:
        return
    t = _gpu.torch()
    a = t.from_numpy(A).cuda()
    b = t.from_numpy(B).cuda()
    c = t.empty((M, N), device="cuda")
    s = t.cuda.current_stream()
    g.check(g.gemm_f32_noalloc(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, splits,
                               s.cuda_stream), "noalloc")
    s.synchronize()
    W = c.cpu().numpy()
    assert np.array_equal(C.view(np.uint32), W.view(np.uint32)), "differs from the workspace sum"


def test_wide_tiles_in_cluster():
    M, N, K = 384, 700, 3000
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_FFMA, g.TILE_128x256, 3)
    _check(C, oracle.ref_gemm(A, B), label="wide tiles, 3 splits in a cluster")


def test_alpha_beta_applied_by_the_cluster_reduction():
    _ex_case(200, 300, 5000, 0, 0, 3, -0.75, 1.5, g.ALGO_FFMA, splits=4)
    _ex_case(200, 300, 5000, 1, 1, 0, 2.0, 0.0, g.ALGO_FFMA, splits=3, c_nan=True)


def test_quantised_exact_in_cluster():
    A, B = make_workload(0)
    C = _gpu.run(A, B, g.ALGO_FFMA, 4)
    _check(C, oracle.ref_gemm(A, B), exact=True, label="quantised 512^3, 4 splits in a cluster")


# ---- the single-CTA tensor-core (3xTF32) kernel: 2..8 splits, one unit per CTA ----

def _configured(A, B, tile, splits):
    return _gpu.run_configured(A, B, g.ALGO_3XTF32, tile, splits)


@pytest.mark.parametrize("tile,splits", [(g.TILE_128x128, 2), (g.TILE_128x128, 3),
                                         (g.TILE_128x128, 5), (g.TILE_128x128, 8),
                                         (g.TILE_128x256, 3)])
def test_3xtf32_cluster_equals_split_order_sum_of_partials(tile, splits):
    # Each split's partial is the same kernel run alone on that K range (same
    # tile, same MMAs, same promotion chunks), so the cluster's result must be
    # those partials added in split order, bit for bit.
    M, N, K = 300, 260, 3000
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, tile, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["cluster_reduce"] == 1, p
    assert p["workspace_bytes"] > 0 and p["kernels"] == 2, p  # staging + GEMM, no reduction
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _configured(A, B, tile, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"3xtf32 cluster {tile}/{splits}")
    kb = (K + 31) // 32
    per = (kb + splits - 1) // splits
    total = None
    for s in range(splits):
        k0, k1 = s * per * 32, min(K, (s + 1) * per * 32)
        part = _configured(np.ascontiguousarray(A[:, k0:k1]), np.ascontiguousarray(B[k0:k1]),
                           tile, 1)
        total = part if total is None else (total + part).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), total.view(np.uint32)), \
        "cluster sum differs from the split-order sum of the partials"


def test_3xtf32_auto_ragged_plan_reduces_in_cluster():
    # AUTO's staged plan for the ragged shape (a transposed A keeps the
    # operands staged): 2 splits added in a cluster
    st, p = g.gemm_f32_plan_ex(1, 0, 1025, 1023, 1000, 1025, 1023, 1023, g.ALGO_AUTO)
    assert st == 0 and p["algo"] == g.ALGO_3XTF32 and p["splits"] == 2 and p["cluster_reduce"] == 1


def test_3xtf32_more_units_than_sms_uses_the_workspace():
    # 40 x 40 tiles x 2 splits = 3200 units: persistent CTAs take several
    # units each, so the partials go through the workspace
    st, p = g.gemm_f32_plan_config(5120, 5120, 4096, g.ALGO_3XTF32, g.TILE_128x128, 2,
                                   A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["cluster_reduce"] == 0, p


def test_3xtf32_cluster_alpha_beta():
    _ex_case(300, 260, 3000, 0, 0, 5, 0.5, -1.25, g.ALGO_3XTF32, splits=4)


def test_3xtf32_clusters_that_do_not_all_fit_use_the_workspace():
    # 21 tiles of 128 x 256 in clusters of 7: fewer such clusters fit on the
    # device at once (15 on a 152-SM GB300), so a caller's 7-way split goes
    # through the workspace instead of running the clusters in two waves,
    # and AUTO picks a plan whose clusters do fit (with K >= 8192 it prefers
    # 128 x 256 tiles: 21 tiles in 6 splits, 21 clusters of 6 against the 23
    # that fit; earlier 128 x 128 tiles in 3 splits)
    if _gpu.torch().cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("cluster capacities measured on a 152-SM part")
    M, N, K = 101, 5159, 61036
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, g.TILE_128x256, 7,
                                   A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["splits"] == 7 and p["cluster_reduce"] == 0, p
    # (AUTO's staged plan: a transposed A keeps the operands staged; row-major
    # ones, with N odd, take the kernels with B's split in tensor memory
    # after a padded copy of B)
    st, p = g.gemm_f32_plan_ex(1, 0, M, N, K, M, N, N, g.ALGO_AUTO)
    assert st == 0 and p["tile_m"] == 128 and 2 <= p["splits"] <= 8, p
    assert p["cluster_reduce"] == 1, p
    tiles = ((M + 127) // 128) * ((N + p["tile_n"] - 1) // p["tile_n"])
    capacity = {2: 76, 3: 46, 4: 36, 5: 28, 6: 23, 7: 15, 8: 15}[p["splits"]]
    assert tiles <= capacity, (tiles, capacity, p)
