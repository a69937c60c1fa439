"""GPU parity of the 3xTF32 kernels that split A and B into TF32 hi/lo parts
in shared memory (the CTA pair, GEMM_F32_TILE_256x256_PAIR_SPLIT, and the
single-CTA 128 x 128 tile, GEMM_F32_TILE_128x128_SPLIT) instead of reading
copies written by staging kernels.

Against the oracle, elementwise within 1e-3 + 1e-3 |C_ref| (NaN guard bands
around C); against the pre-split pair kernel, bit for bit when neither splits
K: both give the tensor core the same high parts (the fp32 words, which it
reads truncated to TF32) and low parts lo = tf32(x - trunc(x)), and issue the
same MMAs in the same order, promoted in the same 128-deep chunks.
"""

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle
from seeded_inputs import make_workload

from . import _gpu
from .test_gemm_gpu import _check

pytestmark = pytest.mark.gpu

SPLIT = g.TILE_256x256_PAIR_SPLIT
PRESPLIT = g.TILE_256x256_PAIR

# ragged in M, N (not a multiple of the 32-column B boxes) and K; several
# rounds of the persistent grid with a K-split tail (2304^2: 81 tiles)
SHAPES = [(256, 256, 32), (300, 200, 40), (2304, 2304, 512), (2305, 2049, 1000),
          (2560, 2330, 77), (1025, 1023, 1000), (513, 4100, 333)]


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
def test_parity_and_equal_to_presplit(shape):
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, SPLIT, 0, A=1 << 32, B=1 << 36,
                                   C=1 << 40)
    assert st == 0 and p["split_in_kernel"] == 1 and (p["tile_m"], p["tile_n"]) == (256, 256)
    # read in place unless a row stride is not a multiple of 16 bytes
    assert p["stage_a"] == (K % 4 != 0) and p["stage_b"] == (N % 4 != 0), p
    A, B = make_workload(2, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT)
    rows, cols = _sample(M, N, M * 7 + N + K)
    _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label=f"split {shape}")
    # bit for bit against the staged pair kernel, both without split-K (the
    # two kernels' stages are 32 and 16 deep, so their split-K boundaries
    # differ; their 128-deep promotion chunks coincide)
    C1 = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT, 1)
    C0 = _gpu.run_configured(A, B, g.ALGO_3XTF32, PRESPLIT, 1)
    assert np.array_equal(C1.view(np.uint32), C0.view(np.uint32)), \
        f"differs from the pre-split kernel at {np.argwhere(C1.view(np.uint32) != C0.view(np.uint32))[:5]}"


@pytest.mark.parametrize("splits", [2, 7])
def test_split_k(splits):
    M, N, K = 600, 700, 5000
    A, B = make_workload(4, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"split-in-kernel, {splits} K splits")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT, splits)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


def test_deep_k_one_tile():
    # one output tile, K spread over many clusters (split-K with workspace)
    M, N, K = 256, 256, 65536
    A, B = make_workload(4, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT, 0)
    _check(C, oracle.ref_gemm(A, B), label="256x256x65536 split in kernel")


@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_operands_are_staged(offsets):
    M, N, K = 700, 900, 300   # row strides of A and B are multiples of 16 bytes
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, SPLIT, 0,
                                   A=(1 << 32) + 4 * offsets[0], B=(1 << 36) + 4 * offsets[1],
                                   C=(1 << 40) + 4 * offsets[2])
    assert st == 0 and p["stage_a"] == (offsets[0] % 4 != 0) and \
        p["stage_b"] == (offsets[1] % 4 != 0), p
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT, 0, offsets=offsets)
    _check(C, oracle.ref_gemm(A, B), label=f"split in kernel, offsets {offsets}")


def test_quantised_exact():
    A, B = make_workload(0)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SPLIT, 0)
    _check(C, oracle.ref_gemm(A, B), exact=True, label="quantised 512^3, split in kernel")


# want: 1 the single-CTA form with B in tensor memory, 2 its pair form, 3 its
# wide single-CTA form, 23 either of the last two (the model's near-ties: per
# SM the two run at the same rate, on tiles of different size), 12 the
# single-CTA or pair form after padded copies (a row stride not a multiple
# of 16 bytes)
@pytest.mark.parametrize("shape,want", [((65536, 256, 1024), 2),
                                        ((2048, 2048, 2048), 23), ((8192, 8192, 8192), 2),
                                        ((1025, 1023, 1000), 12), ((512, 512, 512), 1),
                                        ((384, 384, 20000), 1), ((177, 4459, 16098), 12),
                                        ((9000, 200, 8190), 12), ((9000, 200, 8192), 23),
                                        ((2560, 2560, 2560), 2), ((3072, 3072, 3072), 23),
                                        ((4096, 4096, 4096), 2), ((1024, 1024, 8192), 23),
                                        ((2304, 2304, 512), 2), ((386, 358, 15342), 12),
                                        ((89, 1216, 24336), 1), ((2900, 2900, 1024), 23),
                                        ((1536, 1536, 4096), 23), ((512, 512, 4096), 1),
                                        ((1792, 1792, 4096), 23), ((512, 512, 16384), 3)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_auto_b_in_tensor_memory_rule(shape, want):
    # AUTO takes a kernel with B's split in tensor memory for row-major A and
    # B: the single-CTA 128 x 128 form, the CTA pair or the wide single-CTA
    # form, as its model times them (each with its own split-K factor: 512^2
    # x 4096, 9 splits of 16 single tiles; 512^2 x 16384, 19 splits of 8 wide
    # tiles; 256 x 256 x 65536 in the deep-K test); a row stride that is not
    # a multiple of 16 bytes (1025 x 1023, 177 x 4459, 9000 x 200 x 8190,
    # 386 x 358 x 15342) first gets a padded copy, and the wide form is not
    # offered on copies
    M, N, K = shape
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["algo"] == g.ALGO_3XTF32 and p["b_in_tmem"] == 1, p
    forms = {1: [(128, 128)], 2: [(256, 256)], 3: [(256, 128)], 23: [(256, 256), (256, 128)],
             12: [(128, 128), (256, 256)]}[want]
    assert (p["tile_m"], p["tile_n"]) in forms and p["split_in_kernel"] == 1, p
    assert p["stage_a"] == (K % 4 != 0) and p["stage_b"] == (N % 4 != 0), p
    # the single-CTA form adds 2..8 splits inside a cluster (one unit per CTA)
    assert p["cluster_reduce"] == 0 or (
        (p["tile_m"], p["tile_n"]) == (128, 128) and 2 <= p["splits"] <= 8), p
    # A misaligned by 4 bytes: a padded copy of A, then the single-CTA or
    # pair form
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=(1 << 32) + 4, B=1 << 36, C=1 << 40)
    assert st == 0 and p["b_in_tmem"] == 1 and p["stage_a"] == 1, p
    assert (p["tile_m"], p["tile_n"]) in ((128, 128), (256, 256)), p
    # transposed A: staged unless C has 3M elements or more
    st, p = g.gemm_f32_plan_ex(1, 0, M, N, K, M, N, N, g.ALGO_AUTO)
    assert st == 0 and p["b_in_tmem"] == (M * N >= 3_000_000), p


def test_auto_skinny_parity():
    # AUTO on a tall, narrow, deep product read in place (B's split in
    # tensor memory; ragged M)
    M, N, K = 9000, 200, 8192
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["split_in_kernel"] == 1, p
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run(A, B, g.ALGO_AUTO)
    rows, cols = _sample(M, N, 5)
    _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label="auto skinny")


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
def test_general_form_through_the_in_kernel_split(ta, tb):
    # alpha/beta, leading dimensions and (staged) transposes on a shape AUTO
    # sends, read in place, to the kernel with B's split in tensor memory
    from .test_gemm_gpu import _ex_case
    M, N, K = 1024, 256, 16384
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and p["split_in_kernel"] == 1, p
    _ex_case(M, N, K, ta, tb, 4, -0.75, 1.25, g.ALGO_AUTO)


def _full_mantissa_values(n, rng):
    """fp32 values with all 23 mantissa bits in play: random words over
    exponents 2^-20 .. 2^20 of both signs, plus words whose low 13 bits sit at
    and around the TF32 rounding tie (0x0fff, 0x1000, 0x1001) for even and odd
    TF32 mantissas."""
    special = []
    for m in (0, 1, 2, 3, 1022, 1023):
        for low in (0x0001, 0x0fff, 0x1000, 0x1001, 0x1fff):
            for e in (0, 5, -7):
                for sign in (0, 1):
                    special.append((sign << 31) | ((127 + e) << 23) | (m << 13) | low)
    words = (rng.integers(0, 2, n, dtype=np.uint32) << 31) | \
            (rng.integers(107, 148, n, dtype=np.uint32) << 23) | \
            rng.integers(0, 1 << 23, n, dtype=np.uint32)
    words[:len(special)] = np.array(special, dtype=np.uint32)
    return words.view(np.float32)


@pytest.mark.parametrize("tile", [g.TILE_128x128, PRESPLIT, SPLIT, g.TILE_128x128_SPLIT],
                         ids=["single-cta-staged", "pair-staged", "pair-split", "single-cta-split"])
def test_split_reconstructs_each_operand(tile):
    # With a 0/1 selection matrix as the other operand, C reproduces one
    # operand's elements through the TF32 split: hi (the fp32 word itself,
    # read by the tensor core as trunc(x)) plus lo = tf32(x - trunc(x)).
    # That sum is within 2^-22 |x| of x, and the tensor core's two-term
    # accumulation adds at most one fp32 ulp, so |C - x| <= 2^-20 |x| holds.
    # A tensor core that rounded the word instead of truncating it would be
    # off by up to 2^-11 |x|: the bound pins the reading the split relies on.
    rng = np.random.default_rng(11)
    M = N = 256
    K = 64
    X = _full_mantissa_values(M * K, rng).reshape(M, K)
    S = np.zeros((K, N), dtype=np.float32)
    S[np.arange(N) % K, np.arange(N)] = 1.0          # column n selects k = n % K
    want_a = X[:, np.arange(N) % K].astype(np.float64)
    got_a = _gpu.run_configured(X, S, g.ALGO_3XTF32, tile, 1).astype(np.float64)
    assert np.all(np.abs(got_a - want_a) <= 2.0 ** -20 * np.abs(want_a)), \
        float(np.max(np.abs(got_a - want_a) / np.abs(want_a)))
    # the other side: B split (and, staged, transposed) the same way
    Y = _full_mantissa_values(K * N, rng).reshape(K, N)
    T = np.zeros((M, K), dtype=np.float32)
    T[np.arange(M), np.arange(M) % K] = 1.0          # row m selects k = m % K
    want_b = Y[np.arange(M) % K, :].astype(np.float64)
    got_b = _gpu.run_configured(T, Y, g.ALGO_3XTF32, tile, 1).astype(np.float64)
    assert np.all(np.abs(got_b - want_b) <= 2.0 ** -20 * np.abs(want_b)), \
        float(np.max(np.abs(got_b - want_b) / np.abs(want_b)))


@pytest.mark.parametrize("tile", [PRESPLIT, SPLIT], ids=["pair-staged", "pair-split"])
@pytest.mark.parametrize("shape", [(256, 200, 64), (300, 200, 1000), (520, 100, 96),
                                   (257, 1028, 64), (700, 452, 300)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_output_boxes(tile, shape):
    # Both pair kernels write C through shared memory with TMA stores of 32-row
    # x 16-column boxes.  A ragged N leaves one box partly inside C followed by
    # boxes wholly outside it (not issued); a ragged M leaves warps whose rows
    # are all outside.  Every element is compared, and a second run must give
    # the same bits (a slab reused before its store had read it would not).
    M, N, K = shape
    A, B = make_workload(3, M=M, N=N, K=K)
    want = oracle.ref_gemm(A, B)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, tile, 1)
    _check(C, want, label=f"pair output boxes {shape}")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, tile, 1)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run identical"


def test_pair_output_boxes_alpha():
    # alpha without beta: the staged pair kernel scales the values it stages
    # for the TMA stores; ragged N (2900 = 11 * 256 + 84) and a padded row
    # stride; a transposed A keeps it on staged operands (and AUTO's plan for
    # the operands read in place, a form with B in tensor memory and N = 256
    # MMAs, the CTA pair or the wide single-CTA one, runs too)
    from .test_gemm_gpu import _ex_case
    M, N, K = 2900, 2900, 1024
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and (p["tile_m"], p["tile_n"]) in ((256, 256), (256, 128)), p
    _ex_case(M, N, K, 1, 0, 4, 0.5, 0.0, g.ALGO_AUTO)
    _ex_case(M, N, K, 0, 0, 4, 0.5, 0.0, g.ALGO_AUTO)


@pytest.mark.parametrize("shape,algo,ta", [((2900, 2900, 1024), g.ALGO_AUTO, 1),
                                           ((300, 200, 40), g.ALGO_3XTF32, 1),
                                           ((520, 100, 2000), g.ALGO_3XTF32, 1)],
                         ids=["pair", "single-128", "single-ragged-m"])
def test_output_boxes_with_beta(shape, algo, ta):
    # alpha and beta: the kernels load each 32 x 16 box of the old C into
    # their shared-memory slab (TMA, clipped boxes zero-filled outside C),
    # replace it by alpha v + beta C and store it back (a transposed A keeps
    # these shapes on the staged kernels)
    from .test_gemm_gpu import _ex_case
    M, N, K = shape
    _ex_case(M, N, K, ta, 0, 4, 0.5, -0.75, algo)
    _ex_case(M, N, K, ta, 0, 0, 1.0, 1.0, algo)


def test_pair_output_ragged_row_in_padded_stride():
    # N % 4 != 0 with a row stride that is a multiple of 4 (ldc = N + 2): the
    # columns past N (the padding) must come back untouched, so the kernel may
    # not store the last row piece as a whole 16-byte unit
    from .test_gemm_gpu import _ex_case
    M, N, K = 2900, 2902, 1024
    st, p = g.gemm_f32_plan(M, N, K, g.ALGO_AUTO, 0, A=1 << 32, B=1 << 36, C=1 << 40)
    assert st == 0 and (p["tile_m"], p["tile_n"]) in ((256, 256), (256, 128)), p
    _ex_case(M, N, K, 1, 0, 2, 1.0, 0.0, g.ALGO_AUTO)  # staged pair, TMA stores
    _ex_case(M, N, K, 0, 0, 2, 1.0, 0.0, g.ALGO_AUTO)  # B in tensor memory


SINGLE_SPLIT = g.TILE_128x128_SPLIT


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_single_cta_split_parity_and_equal_to_staged(shape):
    # the single-CTA 128 x 128 kernel splitting in shared memory: against the
    # oracle, and bit for bit against the staged 128 x 128 kernel without
    # split-K (the same high and low parts, the same MMAs in the same order,
    # the same 128-deep promotion chunks)
    M, N, K = shape
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, SINGLE_SPLIT, 1, A=1 << 32,
                                   B=1 << 36, C=1 << 40)
    assert st == 0 and p["split_in_kernel"] == 1 and (p["tile_m"], p["tile_n"]) == (128, 128)
    assert p["stage_a"] == (K % 4 != 0) and p["stage_b"] == (N % 4 != 0), p
    A, B = make_workload(2, M=M, N=N, K=K)
    C1 = _gpu.run_configured(A, B, g.ALGO_3XTF32, SINGLE_SPLIT, 1)
    rows, cols = _sample(M, N, M * 5 + N + K)
    _check(C1[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols),
           label=f"single-CTA split {shape}")
    C0 = _gpu.run_configured(A, B, g.ALGO_3XTF32, g.TILE_128x128, 1)
    assert np.array_equal(C1.view(np.uint32), C0.view(np.uint32)), \
        f"differs from the staged kernel at {np.argwhere(C1.view(np.uint32) != C0.view(np.uint32))[:5]}"


@pytest.mark.parametrize("splits", [2, 4, 8, 12])
def test_single_cta_split_with_split_k(splits):
    # 2..8: the K splits of a tile added inside a cluster; 12: through the
    # workspace and the reduction kernel
    M, N, K = 300, 260, 3000
    st, p = g.gemm_f32_plan_config(M, N, K, g.ALGO_3XTF32, SINGLE_SPLIT, splits, A=1 << 32,
                                   B=1 << 36, C=1 << 40)
    assert st == 0 and p["splits"] == splits and p["split_in_kernel"] == 1, p
    assert p["cluster_reduce"] == (1 if splits <= 8 else 0), p
    A, B = make_workload(4, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SINGLE_SPLIT, splits)
    _check(C, oracle.ref_gemm(A, B), label=f"single-CTA split, {splits} K splits")
    C2 = _gpu.run_configured(A, B, g.ALGO_3XTF32, SINGLE_SPLIT, splits)
    assert np.array_equal(C.view(np.uint32), C2.view(np.uint32)), "not run-to-run deterministic"


@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_single_cta_split_misaligned_operands(offsets):
    M, N, K = 700, 900, 300
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SINGLE_SPLIT, 0, offsets=offsets)
    _check(C, oracle.ref_gemm(A, B), label=f"single-CTA split, offsets {offsets}")


def test_single_cta_split_quantised_exact():
    A, B = make_workload(0)
    C = _gpu.run_configured(A, B, g.ALGO_3XTF32, SINGLE_SPLIT, 0)
    _check(C, oracle.ref_gemm(A, B), exact=True, label="quantised 512^3, single-CTA split")


def test_auto_skinny_deep_parity():
    # few flops per operand element, read in place: B's split in tensor memory
    M, N, K = 89, 1216, 24336
    A, B = make_workload(1, M=M, N=N, K=K)
    C = _gpu.run(A, B, g.ALGO_AUTO)
    rows, cols = _sample(M, N, 9)
    _check(C[rows, cols], oracle.ref_gemm_entries(A, B, rows, cols), label="auto skinny deep")
