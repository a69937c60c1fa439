"""GPU parity of the 3xTF32 kernel that holds B's TF32 split in tensor memory
(GEMM_F32_TILE_128x128_TMEM): each 128 x 128 tile is computed transposed,
D[n][m] = sum_k B[k][n] A[m][k], with B^T as the MMA's tensor-memory operand.

Against the oracle, elementwise within 1e-3 + 1e-3 |C_ref| ("Lecture 12:
final project", section 4) with NaN guard bands around C; bit-exact on the
quantised workload; bit for bit against the staged 128 x 128 kernel without
split-K (the same high and low parts, the same three products per K step in
the same order, the same 128-deep promotion chunks: only the roles of the
operands in the MMA are swapped); and run to run with split-K.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload

from . import _gpu
from .test_gemm_gpu import _check, _ex_case

pytestmark = pytest.mark.gpu

TMEM = g.TILE_128x128_TMEM

# ragged in M, N (not a multiple of the 32-column B boxes) and K; several
# rounds of the persistent grid; K shorter than one stage
SHAPES = [(128, 128, 32), (300, 200, 40), (1, 1, 1), (129, 33, 7), (2304, 2304, 512),
          (2305, 2049, 1000), (2560, 2330, 77), (1025, 1023, 1000), (513, 4100, 333)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load()
    yield
    g.gemm_f32_release()


def _sample(M, N, seed, n=3000):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([np.arange(M), rng.integers(0, M, n), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, M), rng.integers(0, N, n), np.arange(N)])
    return rows, cols


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_parity_and_equal_to_staged(shape):
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, TMEM, 1, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and (p["tile_m"], p["tile_n"]) == (128, 128), p
    # read in place unless a row stride is not a multiple of 16 bytes
    assert p["stage_a"] == (K % 4 != 0) and p["stage_b"] == (N % 4 != 0), p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, 1)
    if M * N <= 300 * 300:
        _check(C, oracle.ref_gemm(A, B), label=f"tmem {shape}")
    else:
        rows, cols = _sample(M, N, M * 3 + N + K)
        _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label=f"tmem {shape}")
    S = _gpu.run_configured(A, B, g.ALGO_3XTF32, g.TILE_128x128, 1)
    assert np.array_equal(C.view(np.uint32), S.view(np.uint32)), \
        f"differs from the staged kernel at {np.argwhere(C.view(np.uint32) != S.view(np.uint32))[:5]}"


@pytest.mark.parametrize("splits", [2, 5, 16, 38])
def test_split_k_parity_and_determinism(splits):
    M, N, K = 256, 256, 16384
    A, B = make_workload(4, M=M, N=N, K=K)
    C1 = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, splits)
    _check(C1, oracle.ref_gemm(A, B), label=f"tmem split-K {splits}")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, splits)
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


def test_deep_k_workload_auto():
    # 256 x 256 x 65536: AUTO's plan is this kernel with split-K, the
    # partials added inside the kernel (one launch, no reduction kernel)
    A, B = make_workload(4)
    st, p = g.gemm_f32_plan(256, 256, 65536, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and p["splits"] > 1, p
    assert p["reduce_in_kernel"] == 1 and p["kernels"] == 1, p
    C = _gpu.run(A, B, g.ALGO_AUTO)
    _check(C, oracle.ref_gemm(A, B), label="tmem deep K (AUTO)")
    # deterministic from call to call (the counters reset themselves)
    for _ in range(3):
        C2 = _gpu.run(A, B, g.ALGO_AUTO)
        assert np.array_equal(C.view(np.uint32), C2.view(np.uint32))


@pytest.mark.parametrize("shape,splits", [((256, 256, 16384), 16), ((300, 200, 40000), 20),
                                          ((129, 384, 20490), 17)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_in_kernel_reduction_equals_split_order_sum(shape, splits):
    # each split's partial is the same kernel run alone on that K range (same
    # MMAs, same promotion chunks from the start of the range), so the
    # in-kernel reduction must equal those partials added in split order
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, TMEM, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["reduce_in_kernel"] == 1, p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem in-kernel reduction {shape} s{splits}")
    kb = (K + 31) // 32
    per = (kb + splits - 1) // splits
    total = None
    for s in range(splits):
        k0, k1 = s * per * 32, min(K, (s + 1) * per * 32)
        part = _gpu.run_configured(np.ascontiguousarray(A[:, k0:k1]),
                                   np.ascontiguousarray(B[k0:k1]), g.ALGO_3XTF32, TMEM, 1)
        total = part if total is None else (total + part).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), total.view(np.uint32)), \
        "in-kernel sum differs from the split-order sum of the partials"


@pytest.mark.parametrize("shape,splits", [((300, 260, 3000), 2), ((300, 260, 3000), 3),
                                          ((300, 260, 3000), 8), ((1025, 1023, 1000), 2),
                                          ((129, 384, 2049), 4)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_cluster_split_equals_split_order_sum(shape, splits):
    # 2..8 splits with one unit per CTA: the splits of a tile run as one
    # cluster and add their partials through distributed shared memory, no
    # workspace and no reduction launch; each split's partial is the same
    # kernel run alone on its K range, so C must equal those partials added
    # in split order, bit for bit
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, TMEM, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["cluster_reduce"] == 1, p
    assert p["reduce_in_kernel"] == 0, p
    assert p["kernels"] == 1 + p["stage_a"] + p["stage_b"], p
    if not p["stage_a"] and not p["stage_b"]:
        assert p["workspace_bytes"] == 0, p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem cluster split {shape} s{splits}")
    kb = (K + 31) // 32
    per = (kb + splits - 1) // splits
    total = None
    for s in range(splits):
        k0, k1 = s * per * 32, min(K, (s + 1) * per * 32)
        part = _gpu.run_configured(np.ascontiguousarray(A[:, k0:k1]),
                                   np.ascontiguousarray(B[k0:k1]), g.ALGO_3XTF32, TMEM, 1)
        total = part if total is None else (total + part).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), total.view(np.uint32)), \
        "cluster sum differs from the split-order sum of the partials"
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, splits)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


@pytest.mark.parametrize("pad", [0, 1, 4])
def test_cluster_split_general_form(pad):
    # the ragged workload's AUTO plan (N odd: B padded, then this kernel with
    # 2 splits added in a cluster), with alpha/beta applied where the cluster
    # writes C: element by element (pad 0, 4: a row stride that is not a
    # multiple of 4) or by 16-byte words (pad 1: ldc 1024)
    M, N, K = 1025, 1023, 1000
    st, p = g.gemm_f32_plan_ex(0, 0, M, N, K, K + pad, N + pad, N + pad, g.ALGO_AUTO, 0,
                               A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and (p["tile_m"], p["tile_n"]) == (128, 128), p
    assert p["splits"] == 2 and p["cluster_reduce"] == 1, p
    _ex_case(M, N, K, 0, 0, pad, -0.75, 1.5, g.ALGO_AUTO)
    _ex_case(M, N, K, 0, 0, pad, 2.0, 0.0, g.ALGO_AUTO, c_nan=True)  # beta 0: C never read


def test_more_units_than_sms_uses_the_reduction_kernel():
    # 40 x 40 tiles x 2 splits: CTAs take several units, so the partials go
    # through the workspace and the reduction kernel
    st, p = g.gemm_f32_plan_config(5120, 5120, 4096, g.ALGO_3XTF32, TMEM, 2, A=1 << 32,
                                   B=1 << 36, C=1 << 40)
    assert st == 0 and p["reduce_in_kernel"] == 0 and p["kernels"] == 2, p
    M, N, K = 1280, 1408, 1024  # 110 tiles x 2 splits = 220 units > 152 SMs
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, TMEM, 2, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["reduce_in_kernel"] == 0, p
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, 2)
    rows, cols = _sample(M, N, 17)
    _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label="tmem s2 workspace")


@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_operands(offsets):
    # operands TMA cannot read in place get padded copies first
    M, N, K = 700, 900, 300
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, 0, offsets=offsets)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem, offsets {offsets}")


def test_quantised_exact():
    A, B = make_workload(0)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, 0)
    _check(C, oracle.ref_gemm(A, B), exact=True, label="quantised 512^3, tmem")


@pytest.mark.parametrize("pad", [0, 4])
def test_general_form_alpha_beta(pad):
    # alpha/beta and leading dimensions on shapes AUTO sends to this kernel
    # (operands read in place), with and without split-K
    _ex_case(520, 300, 2000, 0, 0, pad, 0.5, -0.75, g.ALGO_AUTO)
    _ex_case(256, 256, 20000, 0, 0, pad, -1.5, 0.25, g.ALGO_AUTO)
    _ex_case(300, 200, 96, 0, 0, pad, 2.0, 0.0, g.ALGO_AUTO, c_nan=True)  # beta 0: C not read


def test_split_reconstructs_each_operand():
    # a 0/1 selection operand makes C reproduce each element of the other
    # operand through the whole split-and-multiply path: to 2^-20 relative,
    # which a tensor-core read that rounded the word would miss by up to 2^-11
    rng = np.random.default_rng(11)
    M, N, K = 256, 256, 256
    X = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-6, 6, (M, K)))).astype(np.float32)
    I = np.eye(K, N, dtype=np.float32)
    C = _gpu.run_configured(X, I, g.ALGO_3XTF32, TMEM, 1)
    assert np.allclose(C, X, rtol=2.0 ** -20, atol=0), np.max(np.abs(C - X) / np.abs(X))
    Y = (rng.standard_normal((K, N)) * np.exp(rng.uniform(-6, 6, (K, N)))).astype(np.float32)
    C = _gpu.run_configured(np.eye(M, K, dtype=np.float32), Y, g.ALGO_3XTF32, TMEM, 1)
    assert np.allclose(C, Y, rtol=2.0 ** -20, atol=0), np.max(np.abs(C - Y) / np.abs(Y))


# ---- the CTA-pair form: 256 x 256 tiles, N = 256 MMAs, one accumulator ----
PAIR = g.TILE_256x256_TMEM


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pair_parity_and_equal_to_single(shape):
    # the same products per output in the same order as the single-CTA form;
    # its promotion chunks are 256 deep (the single form's 128), so the bits
    # agree where K fits in one chunk of either
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, PAIR, 1, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and (p["tile_m"], p["tile_n"]) == (256, 256), p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 1)
    if M * N <= 300 * 300:
        _check(C, oracle.ref_gemm(A, B), label=f"tmem pair {shape}")
    else:
        rows, cols = _sample(M, N, M * 5 + N + K)
        _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols),
               label=f"tmem pair {shape}")
    if K <= 128:
        S = _gpu.run_configured(A, B, g.ALGO_3XTF32, TMEM, 1)
        assert np.array_equal(C.view(np.uint32), S.view(np.uint32)), \
            f"differs from the single-CTA form at {np.argwhere(C.view(np.uint32) != S.view(np.uint32))[:5]}"


@pytest.mark.parametrize("splits", [2, 7])
def test_pair_split_k(splits):
    # 9 tiles x 2 or 7 splits, one unit per cluster: below 16 splits the
    # partials go to the reduction kernel
    M, N, K = 520, 700, 6000
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, PAIR, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["reduce_in_kernel"] == 0, p
    assert p["kernels"] == 2, p
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem pair split-K {splits}")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, splits)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


@pytest.mark.parametrize("shape,splits", [((256, 256, 16384), 16), ((300, 200, 40000), 20),
                                          ((129, 384, 20490), 17), ((256, 256, 65536), 76)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_pair_in_kernel_reduction_equals_split_order_sum(shape, splits):
    # the CTA pair's in-kernel reduction (each CTA of each split sums a band
    # of the tile's rows) equals the per-split partials, each the pair kernel
    # run alone on its K range, added in split order
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, PAIR, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["reduce_in_kernel"] == 1, p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem pair in-kernel reduction {shape} s{splits}")
    kb = (K + 31) // 32
    per = (kb + splits - 1) // splits
    total = None
    for s in range(splits):
        k0, k1 = s * per * 32, min(K, (s + 1) * per * 32)
        part = _gpu.run_configured(np.ascontiguousarray(A[:, k0:k1]),
                                   np.ascontiguousarray(B[k0:k1]), g.ALGO_3XTF32, PAIR, 1)
        total = part if total is None else (total + part).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), total.view(np.uint32)), \
        "in-kernel sum differs from the split-order sum of the partials"
    # the counters reset themselves: the next calls give the same bits
    for _ in range(2):
        C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, splits)
        assert np.array_equal(C.view(np.uint32), C2.view(np.uint32))


def test_pair_more_units_than_clusters_uses_the_reduction_kernel():
    # 64 pair tiles x 2 splits = 128 units: clusters take several units, so
    # the partials go through the workspace and the reduction kernel
    M, N, K = 2048, 2048, 4096
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, PAIR, 2, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == 2 and p["reduce_in_kernel"] == 0 and p["kernels"] == 2, p
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 2)
    rows, cols = _sample(M, N, 23)
    _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label="tmem pair s2 workspace")


def test_pair_quantised_exact_and_misaligned():
    A, B = make_workload(0)
    _check(_gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 0), oracle.ref_gemm(A, B), exact=True,
           label="quantised 512^3, tmem pair")
    M, N, K = 700, 900, 300
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 0, offsets=(3, 2, 1))
    _check(C, oracle.ref_gemm(A, B), label="tmem pair, misaligned operands")



@pytest.mark.parametrize("shape", [(2304, 2304, 512), (4096, 4096, 1024), (2560, 2330, 777)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_tail_split(shape):
    # tiles beyond a whole number of rounds of the persistent grid: the
    # partly idle last round's tiles are cut into K shares, added by the
    # fix-up kernel in share order
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, PAIR, 0, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == 1 and p["kernels"] >= 2, p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 0)
    rows, cols = _sample(M, N, M + 3 * N + K)
    _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label=f"tmem pair tail {shape}")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 0)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


WIDE = g.TILE_256x128_TMEM


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_wide_parity_and_equal_to_pair(shape):
    # the wide single-CTA form (256 x 128 tiles, 16-deep stages with A in
    # 64-byte swizzle) issues, per output, the pair form's MMAs in the same
    # order with the same 256-deep promotion chunks: bit-equal to it without
    # split-K
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, WIDE, 1, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and (p["tile_m"], p["tile_n"], p["tile_k"]) == \
        (256, 128, 16), p
    assert p["stage_a"] == (K % 4 != 0) and p["stage_b"] == (N % 4 != 0), p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, 1)
    if M * N <= 300 * 300:
        _check(C, oracle.ref_gemm(A, B), label=f"tmem wide {shape}")
    else:
        rows, cols = _sample(M, N, M * 7 + N + K)
        _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols),
               label=f"tmem wide {shape}")
    P = _gpu.run_configured(A, B, g.ALGO_3XTF32, PAIR, 1)
    assert np.array_equal(C.view(np.uint32), P.view(np.uint32)), \
        f"differs from the pair form at {np.argwhere(C.view(np.uint32) != P.view(np.uint32))[:5]}"


@pytest.mark.parametrize("splits", [2, 7])
def test_wide_split_k(splits):
    M, N, K = 520, 700, 6000
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, WIDE, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["reduce_in_kernel"] == 0, p
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem wide split-K {splits}")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, splits)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


@pytest.mark.parametrize("shape,splits", [((256, 256, 16384), 16), ((300, 200, 40000), 20),
                                          ((256, 256, 65536), 76)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_wide_in_kernel_reduction_equals_split_order_sum(shape, splits):
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, WIDE, splits, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["reduce_in_kernel"] == 1, p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"tmem wide in-kernel reduction {shape} s{splits}")
    kb = (K + 15) // 16
    per = (kb + splits - 1) // splits
    total = None
    for s in range(splits):
        k0, k1 = s * per * 16, min(K, (s + 1) * per * 16)
        part = _gpu.run_configured(np.ascontiguousarray(A[:, k0:k1]),
                                   np.ascontiguousarray(B[k0:k1]), g.ALGO_3XTF32, WIDE, 1)
        total = part if total is None else (total + part).astype(np.float32)
    assert np.array_equal(C.view(np.uint32), total.view(np.uint32)), \
        "in-kernel sum differs from the split-order sum of the partials"
    for _ in range(2):
        C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, splits)
        assert np.array_equal(C.view(np.uint32), C2.view(np.uint32))


def test_wide_quantised_exact_and_misaligned():
    A, B = make_workload(0)
    _check(_gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, 0), oracle.ref_gemm(A, B), exact=True,
           label="quantised 512^3, tmem wide")
    M, N, K = 700, 900, 300
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, WIDE, 0, offsets=(3, 2, 1))
    _check(C, oracle.ref_gemm(A, B), label="tmem wide, misaligned operands")


@pytest.mark.parametrize("alpha,beta", [(0.5, -0.75), (1.0, 1.0)])
def test_wide_general_form_through_auto(alpha, beta):
    # alpha/beta and padded leading dimensions on a shape AUTO sends to the
    # wide form with its partials added inside the kernel (19 splits of 8
    # tiles: one round), so that the in-kernel reduction applies alpha/beta
    from .test_gemm_gpu import _ex_case
    M, N, K = 512, 512, 16384
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and (p["tile_m"], p["tile_n"]) == (256, 128), p
    assert p["reduce_in_kernel"] == 1 and p["kernels"] == 1, p
    _ex_case(M, N, K, 0, 0, 4, alpha, beta, g.ALGO_AUTO)
