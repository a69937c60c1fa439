"""The C-ABI library: it loads, exports what the header declares, and its host
logic (argument validation and the edge rules) holds without touching a GPU.
"""

import ctypes
import os
import re

import pytest

import dense_fp32_gemm_row_gb300 as g
from dense_fp32_gemm_row_gb300 import build as gbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gemm_f32.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(gemm_f32\w*)\s*\(", text,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load()


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("gemm_f32", "gemm_f32_algo", "gemm_f32_algo_splitk", "gemm_f32_plan",
                 "gemm_f32_release", "gemm_f32_status_string", "gemm_f32_device_status",
                 "gemm_f32_selftest_watchdog", "gemm_f32_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(g.library_path())
    for name in _declared_functions():
        assert hasattr(raw, name), f"{name} declared in gemm_f32.h but not exported"


def test_status_strings_and_version(lib):
    assert g.gemm_f32_status_string(0) == "success"
    assert "invalid" in g.gemm_f32_status_string(g.ERR_INVALID_VALUE)
    assert "timed out" in g.gemm_f32_status_string(g.ERR_DEVICE_TIMEOUT)
    assert "captured" in g.gemm_f32_status_string(g.ERR_CAPTURE)
    assert g.gemm_f32_status_string(-99) == "unknown status"
    assert g.gemm_f32_version() >= 100


FAKE_A, FAKE_B, FAKE_C = 0x7000_0000_0000, 0x7100_0000_0000, 0x7200_0000_0000


@pytest.mark.parametrize("M,N,K", [(-1, 4, 4), (4, -1, 4), (4, 4, -1)])
def test_negative_dimension_is_invalid(lib, M, N, K):
    assert g.gemm_f32(FAKE_A, FAKE_B, FAKE_C, M, N, K) == g.ERR_INVALID_VALUE


def test_null_pointer_with_extent_is_invalid(lib):
    assert g.gemm_f32(0, FAKE_B, FAKE_C, 4, 4, 4) == g.ERR_INVALID_VALUE
    assert g.gemm_f32(FAKE_A, 0, FAKE_C, 4, 4, 4) == g.ERR_INVALID_VALUE
    assert g.gemm_f32(FAKE_A, FAKE_B, 0, 4, 4, 4) == g.ERR_INVALID_VALUE


def test_unknown_algo_and_bad_splits_are_invalid(lib):
    assert g.gemm_f32_algo(FAKE_A, FAKE_B, FAKE_C, 4, 4, 4, 3) == g.ERR_INVALID_VALUE
    assert g.gemm_f32_algo(FAKE_A, FAKE_B, FAKE_C, 4, 4, 4, -1) == g.ERR_INVALID_VALUE
    assert g.gemm_f32_algo_splitk(FAKE_A, FAKE_B, FAKE_C, 4, 4, 4, 1, -1) == g.ERR_INVALID_VALUE
    assert g.gemm_f32_algo_splitk(FAKE_A, FAKE_B, FAKE_C, 4, 4, 4, 1,
                                  g.MAX_SPLITS + 1) == g.ERR_INVALID_VALUE


def test_output_overlapping_an_input_is_invalid(lib):
    M = N = K = 8
    assert g.gemm_f32(FAKE_A, FAKE_B, FAKE_A + 4 * 10, M, N, K) == g.ERR_INVALID_VALUE
    assert g.gemm_f32(FAKE_A, FAKE_B, FAKE_B - 4 * 10, M, N, K) == g.ERR_INVALID_VALUE
    assert g.gemm_f32(FAKE_A, FAKE_B, FAKE_A, M, N, K) == g.ERR_INVALID_VALUE


def test_misaligned_float_pointer_is_invalid(lib):
    assert g.gemm_f32(FAKE_A + 2, FAKE_B, FAKE_C, 4, 4, 4) == g.ERR_INVALID_VALUE


def test_empty_output_is_a_no_op_without_a_device(lib):
    # M == 0 or N == 0: success, nothing launched, pointers never looked at
    assert g.gemm_f32(0, 0, 0, 0, 5, 7) == g.SUCCESS
    assert g.gemm_f32(0, 0, 0, 5, 0, 7) == g.SUCCESS
    assert g.gemm_f32(FAKE_A, FAKE_B, FAKE_C, 0, 0, 0) == g.SUCCESS


@pytest.mark.skipif(_has_gpu(), reason="checks the no-device answer; a GPU is present")
def test_no_device_is_unsupported_not_a_fallback(lib):
    assert g.gemm_f32(FAKE_A, FAKE_B, FAKE_C, 4, 4, 4) == g.ERR_UNSUPPORTED_DEVICE
    st, _ = g.gemm_f32_plan(64, 64, 64)
    assert st == g.ERR_UNSUPPORTED_DEVICE
    assert g.gemm_f32_device_status(0) == g.ERR_UNSUPPORTED_DEVICE


def test_matmul_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        g.matmul(torch.zeros(2, 3), torch.zeros(3, 4))


def test_general_entry_validates_layout(lib):
    A, B, C = FAKE_A, FAKE_B, FAKE_C
    ex = g.gemm_f32_ex
    # transpose flags must be 0 or 1
    assert ex(2, 0, 4, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4) == g.ERR_INVALID_VALUE
    # leading dimensions below their minimum
    assert ex(0, 0, 4, 5, 6, 1.0, A, 5, B, 5, 0.0, C, 5) == g.ERR_INVALID_VALUE   # lda < K
    assert ex(1, 0, 4, 5, 6, 1.0, A, 3, B, 5, 0.0, C, 5) == g.ERR_INVALID_VALUE   # lda < M
    assert ex(0, 0, 4, 5, 6, 1.0, A, 6, B, 4, 0.0, C, 5) == g.ERR_INVALID_VALUE   # ldb < N
    assert ex(0, 1, 4, 5, 6, 1.0, A, 6, B, 5, 0.0, C, 5) == g.ERR_INVALID_VALUE   # ldb < K
    assert ex(0, 0, 4, 5, 6, 1.0, A, 6, B, 5, 0.0, C, 4) == g.ERR_INVALID_VALUE   # ldc < N
    # C overlapping A through A's leading dimension
    assert ex(0, 0, 4, 4, 4, 1.0, A, 1000, B, 4, 0.0, A + 4 * 2000, 4) == g.ERR_INVALID_VALUE
    # empty output: success without a device
    assert ex(0, 0, 0, 5, 6, 1.0, 0, 6, 0, 5, 0.0, 0, 5) == g.SUCCESS


def test_tune_configuration_space():
    # the sweep tool's grid: every (algo, tile, splits) once; --quick keeps
    # the tensor-core tiles with the library's own split choice
    from dense_fp32_gemm_row_gb300 import tune
    full = list(tune._configs(g))
    assert len(full) == len(set(full)) == (2 + 8) * len(tune.SPLITS)
    assert {a for a, _, _ in full} == {g.ALGO_FFMA, g.ALGO_3XTF32}
    quick = list(tune._configs(g, quick=True))
    assert quick == [(g.ALGO_3XTF32, t, 0) for t in (g.TILE_128x128, g.TILE_128x256,
                                                       g.TILE_256x256_PAIR,
                                                       g.TILE_256x256_PAIR_SPLIT,
                                                       g.TILE_128x128_SPLIT,
                                                       g.TILE_128x128_TMEM,
                                                       g.TILE_256x256_TMEM,
                                                       g.TILE_256x128_TMEM)]


def test_host_fault_injection_arms_and_disarms(lib):
    # the testing aid is host-only: arming and disarming need no device
    assert g.gemm_f32_inject_host_fault(g.INJECT_WORKSPACE) == g.SUCCESS
    assert g.gemm_f32_inject_host_fault(g.INJECT_DESCRIPTOR) == g.SUCCESS
    assert g.gemm_f32_inject_host_fault(g.INJECT_NONE) == g.SUCCESS
    assert g.gemm_f32_inject_host_fault(3) == g.ERR_INVALID_VALUE
    assert g.gemm_f32_inject_host_fault(-1) == g.ERR_INVALID_VALUE
