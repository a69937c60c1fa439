"""Pins of the CPU oracle against values fixed by arithmetic alone.

The oracle follows the double-accumulation golden reference of "Lecture 12:
final project" (section 3).  None of these tests re-types that loop: each
expected value comes from exact integer or rational arithmetic, a closed
form, or an invariant, chosen so that a plausible slip in the oracle (float
accumulation, a transposed operand, a wrong index, a dropped term, truncating
instead of rounding) fails at least one of them.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from seeded_inputs import make_workload, quantised_fill, uniform_stream


def _exact_round(values) -> np.ndarray:
    """Round exact rationals to float32: each must be exact in double first."""
    out = []
    for v in values:
        d = float(v)
        assert Fraction(d) == v, "test input chosen so the exact sum fits a double"
        out.append(np.float32(d))
    return np.array(out, dtype=np.float32)


def _rng(seed):
    return np.random.default_rng(seed)


def test_one_by_one_is_rounded_product():
    rng = _rng(1)
    for _ in range(200):
        a = np.float32(rng.standard_normal() * 10.0 ** int(rng.integers(-5, 5)))
        b = np.float32(rng.standard_normal() * 10.0 ** int(rng.integers(-5, 5)))
        c = oracle.ref_gemm(np.array([[a]], np.float32), np.array([[b]], np.float32))
        exact = Fraction(float(a)) * Fraction(float(b))
        assert c[0, 0] == _exact_round([exact])[0]


@pytest.mark.parametrize("shape", [(37, 29, 53), (1, 64, 3), (64, 1, 17), (5, 7, 1)])
def test_quantised_inputs_match_exact_integer_product(shape):
    M, N, K = shape
    A = quantised_fill(M * K, 11).reshape(M, K)
    B = quantised_fill(K * N, 12).reshape(K, N)
    # entries are multiples of 1/4: scale to integers, multiply exactly in int64
    Ai = np.rint(A * 4).astype(np.int64)
    Bi = np.rint(B * 4).astype(np.int64)
    exact = (Ai @ Bi).astype(np.float64) / 16.0
    got = oracle.ref_gemm(A, B)
    assert np.array_equal(got, exact.astype(np.float32))


def test_quantised_512_workload_is_exact():
    A, B = make_workload(0)
    Ai = np.rint(A * 4).astype(np.int64)
    Bi = np.rint(B * 4).astype(np.int64)
    exact = ((Ai @ Bi).astype(np.float64) / 16.0).astype(np.float32)
    got = oracle.ref_gemm(A, B)
    assert np.array_equal(got, exact)
    # |C| <= 512 on a 1/16 grid: 14 significant bits, exact in float32
    assert np.abs(exact).max() <= 512


@pytest.mark.parametrize("shape", [(5, 7, 1000), (3, 4, 65536), (9, 1, 1)])
def test_all_ones_gives_k(shape):
    M, N, K = shape
    C = oracle.ref_gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
    assert np.all(C == np.float32(K))


def test_identity_and_permutation_are_exact():
    v, _ = uniform_stream(23 * 31 + 31 * 19, 777)
    A = v[: 23 * 31].reshape(23, 31)
    B = v[23 * 31:].reshape(31, 19)
    assert np.array_equal(oracle.ref_gemm(A, np.eye(31, dtype=np.float32)), A)
    assert np.array_equal(oracle.ref_gemm(np.eye(23, dtype=np.float32), A), A)
    perm = _rng(2).permutation(31)
    P = np.zeros((31, 31), np.float32)
    P[np.arange(31), perm] = 1.0  # (P @ B)[i] = B[perm[i]]
    assert np.array_equal(oracle.ref_gemm(P, B), B[perm])
    Q = np.zeros((19, 19), np.float32)
    q = _rng(3).permutation(19)
    Q[q, np.arange(19)] = 1.0  # (B @ Q)[:, j] = B[:, q[j]]
    assert np.array_equal(oracle.ref_gemm(B, Q), B[:, q])


def test_power_of_two_diagonal_scales_rows():
    v, _ = uniform_stream(12 * 10, 99)
    B = v.reshape(12, 10)
    d = np.array([2.0 ** e for e in range(-6, 6)], np.float32)
    C = oracle.ref_gemm(np.diag(d).astype(np.float32), B)
    assert np.array_equal(C, (B * d[:, None]).astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (7, 13, 17), (17, 5, 13), (3, 17, 2),
                                   (13, 7, 11)])
def test_bruteforce_tiny_dyadic(M, N, K):
    rng = _rng(M * 100 + N * 10 + K)
    Ai = rng.integers(-1024, 1025, size=(M, K))
    Bi = rng.integers(-1024, 1025, size=(K, N))
    A = (Ai / 256.0).astype(np.float32)
    B = (Bi / 256.0).astype(np.float32)
    exact = [sum(Fraction(int(Ai[i, k]) * int(Bi[k, j]), 65536) for k in range(K))
             for i in range(M) for j in range(N)]
    want = _exact_round(exact).reshape(M, N)
    assert np.array_equal(oracle.ref_gemm(A, B), want)


def _ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def test_general_floats_agree_with_correctly_rounded_sum():
    # fsum returns the correctly rounded double of the exact sum of the (exact)
    # double products; rounding that to float32 can differ from the oracle's
    # double-accumulated value only when the two doubles straddle a float32
    # rounding boundary, i.e. by at most one float32 ulp and rarely.
    rng = _rng(5)
    M, N, K = 24, 20, 300
    A = (rng.standard_normal((M, K)) * np.exp(rng.uniform(-8, 8, (M, K)))).astype(np.float32)
    B = (rng.standard_normal((K, N)) * np.exp(rng.uniform(-8, 8, (K, N)))).astype(np.float32)
    Ad, Bd = A.astype(np.float64), B.astype(np.float64)
    want = np.array([[np.float32(math.fsum(Ad[i, :] * Bd[:, j])) for j in range(N)]
                     for i in range(M)], dtype=np.float32)
    got = oracle.ref_gemm(A, B)
    dist = _ulp_distance(got, want)
    assert dist.max() <= 1
    assert np.mean(dist == 0) >= 0.99


def test_double_accumulation_survives_cancellation():
    # float accumulation would give 1 + 2^-30 -> 1 -> 0
    A = np.array([[1.0, 2.0 ** -30, -1.0]], np.float32)
    B = np.ones((3, 1), np.float32)
    assert oracle.ref_gemm(A, B)[0, 0] == np.float32(2.0 ** -30)


@pytest.mark.parametrize("terms", [
    [1.0, 2.0 ** -24, 2.0 ** -40],  # above the midpoint: rounds up
    [1.0, 2.0 ** -24],              # exact tie, even neighbour is 1.0
    [1.0, 3 * 2.0 ** -24],          # exact tie, even neighbour is 1 + 2^-22
    [-1.0, -(2.0 ** -24), -(2.0 ** -45)],
])
def test_final_conversion_rounds_to_nearest_even(terms):
    A = np.array([terms], np.float32)
    B = np.ones((len(terms), 1), np.float32)
    exact = sum(Fraction(t) for t in terms)
    assert oracle.ref_gemm(A, B)[0, 0] == _exact_round([exact])[0]


def test_transpose_invariant_bitwise():
    v, _ = uniform_stream(33 * 47 + 47 * 21, 31337)
    A = v[: 33 * 47].reshape(33, 47)
    B = v[33 * 47:].reshape(47, 21)
    C = oracle.ref_gemm(A, B)
    Ct = oracle.ref_gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T))
    assert C.shape == (33, 21)
    assert np.array_equal(Ct.T, C)


def test_linearity_exact_on_quantised():
    M, N, K = 19, 23, 41
    A = quantised_fill(M * K, 5).reshape(M, K)
    B1 = quantised_fill(K * N, 6).reshape(K, N)
    B2 = quantised_fill(K * N, 7).reshape(K, N)
    lhs = oracle.ref_gemm(A, B1 + B2)
    rhs = oracle.ref_gemm(A, B1) + oracle.ref_gemm(A, B2)
    assert np.array_equal(lhs, rhs)


def test_zero_row_and_column_give_zero_output():
    v, _ = uniform_stream(10 * 12 + 12 * 9, 4242)
    A = v[:120].reshape(10, 12).copy()
    B = v[120:].reshape(12, 9).copy()
    A[3, :] = 0
    B[:, 5] = 0
    C = oracle.ref_gemm(A, B)
    assert np.all(C[3, :] == 0) and np.all(C[:, 5] == 0)
    assert np.count_nonzero(C) == 9 * 8


def test_k_zero_and_empty_shapes():
    C = oracle.ref_gemm(np.zeros((4, 0), np.float32), np.zeros((0, 3), np.float32))
    assert C.shape == (4, 3) and np.all(C == 0)
    assert oracle.ref_gemm(np.zeros((0, 5), np.float32), np.zeros((5, 3), np.float32)).shape == (0, 3)


def test_entries_and_rows_match_full_product():
    A, B = make_workload(1, M=67, N=45, K=129)
    C = oracle.ref_gemm(A, B)
    rng = _rng(9)
    r = rng.integers(0, 67, 500)
    c = rng.integers(0, 45, 500)
    assert np.array_equal(oracle.ref_gemm_entries(A, B, r, c), C[r, c])
    assert np.array_equal(oracle.ref_gemm_rows(A, B, 10, 7), C[10:17])


def test_thread_count_does_not_change_bits():
    A, B = make_workload(2, M=96, N=80, K=777)
    assert np.array_equal(oracle.ref_gemm(A, B, nthreads=1), oracle.ref_gemm(A, B, nthreads=3))


# ---------------------------------------------------------------------------
# comparator
# ---------------------------------------------------------------------------
def test_comparator_tolerance_edges_and_nan():
    ref = np.array([0.0, 100.0, -2.0], np.float32)
    ok = ref + np.array([1e-3 * 0.999, 0.1009, -0.0029], np.float32)
    assert oracle.compare(ok, ref)["pass"]
    bad = ref.copy()
    bad[1] = 100.2
    res = oracle.compare(bad, ref)
    assert not res["pass"] and res["first_bad"] == 1
    for poison in (np.nan, np.inf, -np.inf):
        g = ref.copy()
        g[2] = poison
        assert not oracle.compare(g, ref)["pass"]


# ---------------------------------------------------------------------------
# general form: transposes, leading dimensions, alpha and beta
# ---------------------------------------------------------------------------
def test_general_form_reduces_to_plain_product():
    A, B = make_workload(1, M=37, N=29, K=41)
    C = oracle.ref_gemm(A, B)
    got = oracle.ref_gemm_ex(0, 0, 37, 29, 41, 1.0, A, 41, B, 29, 0.0,
                             np.full(37 * 29, np.nan, np.float32), 29)
    assert np.array_equal(got.reshape(37, 29), C)


def test_transposed_storage_gives_same_bits():
    A, B = make_workload(2, M=23, N=19, K=31)
    C = oracle.ref_gemm(A, B)
    At = np.ascontiguousarray(A.T)  # K x M storage
    Bt = np.ascontiguousarray(B.T)  # N x K storage
    for ta, tb, a, lda, b, ldb in ((1, 0, At, 23, B, 19), (0, 1, A, 31, Bt, 31),
                                   (1, 1, At, 23, Bt, 31)):
        got = oracle.ref_gemm_ex(ta, tb, 23, 19, 31, 1.0, a, lda, b, ldb, 0.0,
                                 np.zeros(23 * 19, np.float32), 19)
        assert np.array_equal(got.reshape(23, 19), C), (ta, tb)


def test_leading_dimensions_pick_the_right_submatrix():
    # embed A (5 x 7) in a 5 x 11 buffer and C (5 x 3) in a 5 x 8 buffer
    A = quantised_fill(5 * 7, 3).reshape(5, 7)
    B = quantised_fill(7 * 3, 4).reshape(7, 3)
    Abuf = np.full((5, 11), 1e30, np.float32)
    Abuf[:, :7] = A
    Cbuf = np.full((5, 8), 7.0, np.float32)
    got = oracle.ref_gemm_ex(0, 0, 5, 3, 7, 1.0, Abuf, 11, B, 3, 0.0, Cbuf, 8).reshape(5, 8)
    Ai = np.rint(A * 4).astype(np.int64)
    Bi = np.rint(B * 4).astype(np.int64)
    assert np.array_equal(got[:, :3], ((Ai @ Bi) / 16.0).astype(np.float32))
    assert np.all(got[:, 3:] == 7.0)


def test_alpha_beta_exact_on_dyadic_values():
    # quantised inputs, alpha and beta powers of two, C old on a 1/16 grid:
    # every step is exact, so the result is alpha S + beta C exactly
    A = quantised_fill(9 * 13, 5).reshape(9, 13)
    B = quantised_fill(13 * 6, 6).reshape(13, 6)
    Cold = (quantised_fill(9 * 6, 7) / 4).astype(np.float32).reshape(9, 6)
    S = (np.rint(A * 4).astype(np.int64) @ np.rint(B * 4).astype(np.int64)) / 16.0
    got = oracle.ref_gemm_ex(0, 0, 9, 6, 13, 0.5, A, 13, B, 6, -2.0, Cold, 6).reshape(9, 6)
    assert np.array_equal(got, (0.5 * S - 2.0 * Cold).astype(np.float32))


def _round_f32(x: Fraction) -> np.float32:
    """The float32 nearest an exact rational, ties to even (normal range).

    Works on the rational itself, so no intermediate double rounding can hide
    a second rounding in the oracle.
    """
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127, "chosen inputs stay in float32's normal range"
    scaled = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return np.float32(sign * m * 2.0 ** (e - 23))  # m * 2^(e-23) is exact in double


def test_round_f32_helper_against_numpy_on_doubles():
    # on values that are doubles, numpy's double -> float32 cast is correctly
    # rounded, so the helper must agree with it everywhere, ties included
    rng = _rng(17)
    vals = list(rng.standard_normal(2000) * 2.0 ** rng.integers(-40, 40, 2000))
    vals += [1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, -(1.0 + 2.0 ** -24), 1.0 - 2.0 ** -25]
    for v in vals:
        assert _round_f32(Fraction(float(v))) == np.float32(v), v


def test_alpha_beta_rounded_once_near_cancellation():
    # alpha = fl32(1/3), beta = -alpha and an old C one part in 2^9 to 2^14
    # away from S: alpha*S + beta*C nearly cancels, so rounding alpha*S to
    # float32 before the add (a double rounding) changes the result by far
    # more than an ulp of it.  Every double step the general form takes is
    # exact here (S has <= 23 significant bits, alpha*S <= 47, beta*C <= 48,
    # and the two products lie within a factor of two of each other), so the
    # expected value is the exact rational result rounded once.
    M, N, K = 6, 5, 7
    rng = _rng(23)
    Ai = rng.integers(-1024, 1025, size=(M, K))
    Bi = rng.integers(-1024, 1025, size=(K, N))
    A = (Ai / 256.0).astype(np.float32)
    B = (Bi / 256.0).astype(np.float32)
    S = [[sum(Fraction(int(Ai[i, k]) * int(Bi[k, j]), 65536) for k in range(K))
          for j in range(N)] for i in range(M)]
    alpha = np.float32(1.0 / 3.0)
    beta = -alpha
    Cold = np.empty((M, N), np.float32)
    for i in range(M):
        for j in range(N):
            s = S[i][j] if S[i][j] != 0 else Fraction(1)
            delta = Fraction(int(rng.integers(1, 32)), 2 ** int(rng.integers(9, 15)))
            Cold[i, j] = np.float32(float(s * (1 + delta)))
    want = np.empty((M, N), np.float32)
    twice = np.empty((M, N), np.float32)
    for i in range(M):
        for j in range(N):
            exact = Fraction(float(alpha)) * S[i][j] + Fraction(float(beta)) * Fraction(float(Cold[i, j]))
            want[i, j] = _round_f32(exact)
            rounded_first = Fraction(float(_round_f32(Fraction(float(alpha)) * S[i][j])))
            twice[i, j] = _round_f32(rounded_first + Fraction(float(beta)) * Fraction(float(Cold[i, j])))
    # the case has teeth: a double rounding differs on most entries
    assert np.mean(want != twice) > 0.5
    got = oracle.ref_gemm_ex(0, 0, M, N, K, float(alpha), A, K, B, N, float(beta), Cold, N)
    assert np.array_equal(got.reshape(M, N), want)


def test_alpha_beta_general_values_within_one_ulp_of_exact():
    # general alpha, beta, operands and old C: the exact rational alpha*S +
    # beta*C rounded once, against which the oracle's double arithmetic may
    # differ by at most one float32 ulp, and rarely
    M, N, K = 9, 8, 23
    rng = _rng(29)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    Cold = rng.standard_normal((M, N)).astype(np.float32)
    alpha, beta = np.float32(0.7071), np.float32(-1.3)
    want = np.empty((M, N), np.float32)
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
            want[i, j] = _round_f32(Fraction(float(alpha)) * s
                                    + Fraction(float(beta)) * Fraction(float(Cold[i, j])))
    got = oracle.ref_gemm_ex(0, 0, M, N, K, float(alpha), A, K, B, N, float(beta), Cold, N)
    dist = _ulp_distance(got.reshape(M, N), want)
    assert dist.max() <= 1
    assert np.mean(dist == 0) >= 0.95


def test_beta_zero_never_reads_c():
    A, B = make_workload(1, M=4, N=5, K=6)
    got = oracle.ref_gemm_ex(0, 0, 4, 5, 6, 1.0, A, 6, B, 5, 0.0,
                             np.full(20, np.nan, np.float32), 5)
    assert np.isfinite(got).all()
    # beta != 0 with a NaN in C propagates it
    got = oracle.ref_gemm_ex(0, 0, 4, 5, 6, 1.0, A, 6, B, 5, 1.0,
                             np.full(20, np.nan, np.float32), 5)
    assert np.isnan(got).all()
