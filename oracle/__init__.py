"""CPU oracle for row-major FP32 GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the package smoke check and the benchmark's CPU-baseline leg
may import this module.  The CUDA library never calls it, and the two share
no code: the oracle is a plain C triple loop (``ref_gemm.c``) compiled with
gcc, loaded here through ctypes.

What it computes ("Lecture 12: final project", runguoli.com ECE408 notes l12,
section 3 "CPU golden reference"): ``C[i][j] = float(sum_k double(A[i][k]) *
double(B[k][j]))``, k ascending, double accumulation, one final
round-to-nearest conversion.  See ``ref_gemm.c`` for the details.

Every function here is pinned by ``tests/test_oracle.py`` against values fixed
by arithmetic alone (exact integer products, closed forms, exact rational
brute force, invariants); none is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_gemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libref_gemm.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``ref_gemm.c`` into ``oracle/_build/libref_gemm.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    f32p = ctypes.POINTER(ctypes.c_float)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.ref_gemm.argtypes = [f32p, f32p, f32p, i64, i64, i64, ctypes.c_int]
    lib.ref_gemm.restype = None
    lib.ref_gemm_entries.argtypes = [f32p, f32p, i64, i64, i64, i64p, i64p, i64, f32p,
                                     ctypes.c_int]
    lib.ref_gemm_entries.restype = None
    lib.ref_gemm_rows.argtypes = [f32p, f32p, i64, i64, i64, i64, i64, f32p, ctypes.c_int]
    lib.ref_gemm_rows.restype = None
    lib.ref_gemm_ex.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, ctypes.c_double, f32p,
                                i64, f32p, i64, ctypes.c_double, f32p, i64, ctypes.c_int]
    lib.ref_gemm_ex.restype = None
    lib.ref_max_threads.argtypes = []
    lib.ref_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle takes float32 inputs, got {a.dtype}")
    return a


def _ptr(a: np.ndarray, t=ctypes.c_float):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _shapes(A: np.ndarray, B: np.ndarray) -> tuple[int, int, int]:
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {A.shape} x {B.shape}")
    return A.shape[0], B.shape[1], A.shape[1]


def ref_gemm(A: np.ndarray, B: np.ndarray, nthreads: int = 0) -> np.ndarray:
    """Full ``C = A @ B`` by the oracle's definition (float32 result)."""
    A, B = _f32(A), _f32(B)
    M, N, K = _shapes(A, B)
    C = np.empty((M, N), dtype=np.float32)
    if M and N:
        _load().ref_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(nthreads))
    return C


def ref_gemm_entries(A: np.ndarray, B: np.ndarray, rows, cols, nthreads: int = 0) -> np.ndarray:
    """``C[rows[t], cols[t]]`` for each t, one dot product each."""
    A, B = _f32(A), _f32(B)
    M, N, K = _shapes(A, B)
    r = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    c = np.ascontiguousarray(cols, dtype=np.int64).ravel()
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("entry index out of range")
    out = np.empty(r.size, dtype=np.float32)
    if r.size:
        _load().ref_gemm_entries(_ptr(A), _ptr(B), M, N, K, _ptr(r, ctypes.c_int64),
                                 _ptr(c, ctypes.c_int64), r.size, _ptr(out), int(nthreads))
    return out


def ref_gemm_rows(A: np.ndarray, B: np.ndarray, row0: int, nrows: int,
                  nthreads: int = 0) -> np.ndarray:
    """Rows ``row0 .. row0+nrows-1`` of ``C`` (an ``nrows x N`` array)."""
    A, B = _f32(A), _f32(B)
    M, N, K = _shapes(A, B)
    if row0 < 0 or nrows < 0 or row0 + nrows > M:
        raise IndexError("row range out of bounds")
    out = np.empty((nrows, N), dtype=np.float32)
    if nrows and N:
        _load().ref_gemm_rows(_ptr(A), _ptr(B), M, N, K, int(row0), int(nrows), _ptr(out),
                              int(nthreads))
    return out


def ref_gemm_ex(transa: int, transb: int, M: int, N: int, K: int, alpha: float,
                A: np.ndarray, lda: int, B: np.ndarray, ldb: int, beta: float,
                C: np.ndarray, ldc: int, nthreads: int = 0) -> np.ndarray:
    """General form C = alpha op(A) op(B) + beta C on flat row-major buffers.

    ``A``, ``B`` and ``C`` are flat float32 arrays holding the matrices with
    the given leading dimensions; returns a new flat copy of ``C`` with the
    M x N block updated (elements outside it are left as they were).
    """
    A = _f32(np.ravel(A))
    B = _f32(np.ravel(B))
    out = _f32(np.ravel(C)).copy()
    need_a = ((K - 1) * lda + M if transa else (M - 1) * lda + K) if M and K else 0
    need_b = ((N - 1) * ldb + K if transb else (K - 1) * ldb + N) if K and N else 0
    need_c = (M - 1) * ldc + N if M and N else 0
    if A.size < need_a or B.size < need_b or out.size < need_c:
        raise ValueError("buffer smaller than its leading dimension implies")
    if M and N:
        _load().ref_gemm_ex(int(transa), int(transb), M, N, K, float(alpha), _ptr(A), lda,
                            _ptr(B), ldb, float(beta), _ptr(out), ldc, int(nthreads))
    return out


def max_threads() -> int:
    """Threads the oracle's OpenMP loop uses by default."""
    return int(_load().ref_max_threads())


# ---------------------------------------------------------------------------
# comparator ("Lecture 12: final project", section 4, verify)
# ---------------------------------------------------------------------------
def compare(got: np.ndarray, ref: np.ndarray, atol: float = 1e-3, rtol: float = 1e-3) -> dict:
    """Elementwise ``|got - ref| <= atol + rtol*|ref|``; NaN or Inf in ``got`` fails.

    The page's comparator tests ``err > tol`` and so lets a NaN pass; here the
    test is ``not (err <= tol)``, which fails it.  Returns pass flag, max abs
    and max relative error (relative only where ``|ref| > 1e-30``), the worst
    ratio ``err / tol`` and the first failing flat index (-1 if none).
    """
    g = np.asarray(got, dtype=np.float64).ravel()
    e = np.asarray(ref, dtype=np.float64).ravel()
    if g.shape != e.shape:
        raise ValueError("shape mismatch")
    if g.size == 0:
        return {"pass": True, "max_abs": 0.0, "max_rel": 0.0, "worst_ratio": 0.0, "first_bad": -1}
    with np.errstate(invalid="ignore"):
        ad = np.abs(g - e)
        tol = atol + rtol * np.abs(e)
        ok = ad <= tol
        nz = np.abs(e) > 1e-30
        rel = np.where(nz, ad / np.where(nz, np.abs(e), 1.0), 0.0)
    bad = np.flatnonzero(~ok)
    finite = np.isfinite(ad)
    return {
        "pass": bool(bad.size == 0),
        "max_abs": float(np.max(np.where(finite, ad, np.inf))),
        "max_rel": float(np.max(np.where(finite, rel, np.inf))),
        "worst_ratio": float(np.max(np.where(finite, ad / tol, np.inf))),
        "first_bad": int(bad[0]) if bad.size else -1,
    }
