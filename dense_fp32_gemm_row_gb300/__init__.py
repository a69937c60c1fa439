"""GB300-native single-precision GEMM: ``C = A @ B``, row-major, any M/N/K.

A thin ctypes binding over ``libgemmf32.so`` (declared in
``include/gemm_f32.h``).  The functions carry the C names and only marshal
arguments: every step of the computation runs in the library's CUDA kernels
on the GPU.  There is no CPU fallback: if the library is missing or the
device is not an sm_103 GPU, the calls raise.

Raw entry points (pointers and the stream are plain integers)::

    gemm_f32(A_ptr, B_ptr, C_ptr, M, N, K, stream) -> status
    gemm_f32_algo(A_ptr, B_ptr, C_ptr, M, N, K, algo, stream) -> status
    gemm_f32_algo_splitk(A_ptr, B_ptr, C_ptr, M, N, K, algo, splits, stream) -> status

Tensor convenience (torch CUDA tensors, float32, row-major contiguous)::

    matmul(A, B, out=None, algo=ALGO_AUTO, splits=0, stream=None) -> C
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "ALGO_AUTO", "ALGO_FFMA", "ALGO_3XTF32", "ALGOS", "MAX_SPLITS",
    "SUCCESS", "ERR_INVALID_VALUE", "ERR_UNSUPPORTED_DEVICE", "ERR_WORKSPACE",
    "ERR_DEVICE_TIMEOUT", "ERR_DESCRIPTOR", "ERR_CAPTURE", "GemmError",
    "library_path", "load", "gemm_f32", "gemm_f32_algo", "gemm_f32_algo_splitk",
    "gemm_f32_algo_splitk_ev", "gemm_f32_noalloc", "gemm_f32_host", "gemm_f32_ex",
    "gemm_f32_configured", "gemm_f32_plan_config", "Config", "TILE_AUTO", "TILE_128x128",
    "TILE_128x256", "TILE_256x256_PAIR", "TILE_256x256_PAIR_SPLIT", "TILE_128x128_SPLIT",
    "TILE_128x128_TMEM", "TILE_256x256_TMEM", "TILE_256x128_TMEM",
    "gemm_f32_plan", "gemm_f32_plan_ex", "gemm_f32_device_status", "gemm_f32_selftest_watchdog",
    "gemm_f32_noalloc_selftest_watchdog", "gemm_f32_inject_host_fault", "INJECT_NONE",
    "INJECT_WORKSPACE", "INJECT_DESCRIPTOR",
    "gemm_f32_release", "gemm_f32_status_string", "gemm_f32_version", "matmul", "check",
]

ALGO_AUTO = 0
ALGO_FFMA = 1
ALGO_3XTF32 = 2
ALGOS = {"auto": ALGO_AUTO, "ffma": ALGO_FFMA, "3xtf32": ALGO_3XTF32}
MAX_SPLITS = 256

SUCCESS = 0
ERR_INVALID_VALUE = -1
ERR_UNSUPPORTED_DEVICE = -2
ERR_WORKSPACE = -3
ERR_DEVICE_TIMEOUT = -4
ERR_DESCRIPTOR = -5
ERR_CAPTURE = -6

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libgemmf32.so")
_lib = None
_lock = threading.Lock()


class GemmError(RuntimeError):
    """A non-zero status from libgemmf32."""

    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: status {status} ({gemm_f32_status_string(status)})")


TILE_AUTO = 0
TILE_128x128 = 1
TILE_128x256 = 2
TILE_256x256_PAIR = 3
TILE_256x256_PAIR_SPLIT = 4
TILE_128x128_SPLIT = 5
TILE_128x128_TMEM = 6
TILE_256x256_TMEM = 7
TILE_256x128_TMEM = 8


class Config(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_int), ("tile", ctypes.c_int), ("splits", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("algo", ctypes.c_int), ("splits", ctypes.c_int), ("tile_m", ctypes.c_int),
        ("tile_n", ctypes.c_int), ("tile_k", ctypes.c_int), ("stages", ctypes.c_int),
        ("ctas", ctypes.c_int), ("stage_a", ctypes.c_int), ("stage_b", ctypes.c_int),
        ("kernels", ctypes.c_int), ("workspace_bytes", ctypes.c_longlong),
        ("split_in_kernel", ctypes.c_int), ("cluster_reduce", ctypes.c_int),
        ("ctas_per_sm", ctypes.c_int), ("threads_per_cta", ctypes.c_int),
        ("b_in_tmem", ctypes.c_int), ("reduce_in_kernel", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libgemmf32.so (built in-tree); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing; build it with "
                "`python -m dense_fp32_gemm_row_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        lib.gemm_f32.argtypes = [vp, vp, vp, i, i, i, vp]
        lib.gemm_f32_algo.argtypes = [vp, vp, vp, i, i, i, i, vp]
        lib.gemm_f32_algo_splitk.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.gemm_f32_algo_splitk_ev.argtypes = [vp, vp, vp, i, i, i, i, i, vp, vp, vp]
        lib.gemm_f32_plan.argtypes = [i, i, i, i, i, vp, vp, vp, ctypes.POINTER(PlanInfo)]
        lib.gemm_f32_plan_ex.argtypes = [i, i, i, i, i, vp, ll, vp, ll, vp, ll, i, i,
                                         ctypes.POINTER(PlanInfo)]
        lib.gemm_f32_noalloc.argtypes = [vp, vp, vp, i, i, i, i, vp]
        lib.gemm_f32_host.argtypes = [vp, vp, vp, i, i, i, i, vp]
        lib.gemm_f32_configured.argtypes = [vp, vp, vp, i, i, i, ctypes.POINTER(Config), vp]
        lib.gemm_f32_plan_config.argtypes = [i, i, i, ctypes.POINTER(Config), vp, vp, vp,
                                             ctypes.POINTER(PlanInfo)]
        f = ctypes.c_float
        lib.gemm_f32_ex.argtypes = [i, i, i, i, i, f, vp, ll, vp, ll, f, vp, ll, i, i, vp]
        lib.gemm_f32_device_status.argtypes = [i]
        lib.gemm_f32_selftest_watchdog.argtypes = [ll, vp]
        lib.gemm_f32_noalloc_selftest_watchdog.argtypes = [ll, vp]
        lib.gemm_f32_inject_host_fault.argtypes = [i]
        lib.gemm_f32_release.argtypes = []
        lib.gemm_f32_status_string.argtypes = [i]
        lib.gemm_f32_status_string.restype = ctypes.c_char_p
        lib.gemm_f32_version.argtypes = []
        for name in ("gemm_f32", "gemm_f32_algo", "gemm_f32_algo_splitk",
                     "gemm_f32_algo_splitk_ev", "gemm_f32_plan", "gemm_f32_plan_ex",
                     "gemm_f32_noalloc",
                     "gemm_f32_host", "gemm_f32_ex", "gemm_f32_configured", "gemm_f32_plan_config",
                     "gemm_f32_device_status", "gemm_f32_selftest_watchdog",
                     "gemm_f32_noalloc_selftest_watchdog", "gemm_f32_inject_host_fault",
                     "gemm_f32_release",
                     "gemm_f32_version"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _p(x):
    return None if x is None or x == 0 else ctypes.c_void_p(int(x))


def gemm_f32(A, B, C, M, N, K, stream=0) -> int:
    return load().gemm_f32(_p(A), _p(B), _p(C), M, N, K, _p(stream))


def gemm_f32_algo(A, B, C, M, N, K, algo, stream=0) -> int:
    return load().gemm_f32_algo(_p(A), _p(B), _p(C), M, N, K, algo, _p(stream))


def gemm_f32_algo_splitk(A, B, C, M, N, K, algo, splits, stream=0) -> int:
    return load().gemm_f32_algo_splitk(_p(A), _p(B), _p(C), M, N, K, algo, splits, _p(stream))


def gemm_f32_algo_splitk_ev(A, B, C, M, N, K, algo, splits, stream=0, main_begin=None,
                            main_end=None) -> int:
    """``main_begin``/``main_end``: raw cudaEvent_t handles (e.g. ``torch.cuda.Event().cuda_event``)."""
    return load().gemm_f32_algo_splitk_ev(_p(A), _p(B), _p(C), M, N, K, algo, splits, _p(stream),
                                          _p(main_begin), _p(main_end))


def gemm_f32_ex(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, algo=ALGO_AUTO,
                splits=0, stream=0) -> int:
    """C = alpha op(A) op(B) + beta C, row-major with leading dimensions (see gemm_f32.h)."""
    return load().gemm_f32_ex(int(transa), int(transb), M, N, K, float(alpha), _p(A), int(lda),
                              _p(B), int(ldb), float(beta), _p(C), int(ldc), int(algo),
                              int(splits), _p(stream))


def gemm_f32_configured(A, B, C, M, N, K, algo, tile=TILE_AUTO, splits=0, stream=0) -> int:
    """C = A @ B with a forced kernel configuration (algorithm, tile, split-K)."""
    cfg = Config(int(algo), int(tile), int(splits))
    return load().gemm_f32_configured(_p(A), _p(B), _p(C), M, N, K, ctypes.byref(cfg), _p(stream))


def gemm_f32_plan_config(M, N, K, algo, tile=TILE_AUTO, splits=0, A=0, B=0, C=0):
    cfg = Config(int(algo), int(tile), int(splits))
    info = PlanInfo()
    st = load().gemm_f32_plan_config(M, N, K, ctypes.byref(cfg), _p(A), _p(B), _p(C),
                                     ctypes.byref(info))
    return st, info.as_dict()


def gemm_f32_host(A, B, C, M, N, K, algo=ALGO_AUTO, stream=0) -> int:
    """C = A @ B with HOST pointers; copies overlap the GEMM by row panels (asynchronous)."""
    return load().gemm_f32_host(_p(A), _p(B), _p(C), M, N, K, algo, _p(stream))


def gemm_f32_noalloc(A, B, C, M, N, K, splits=0, stream=0) -> int:
    """The FFMA split-K GEMM with scratch from a fixed device array; allocates nothing."""
    return load().gemm_f32_noalloc(_p(A), _p(B), _p(C), M, N, K, splits, _p(stream))


def gemm_f32_plan(M, N, K, algo=ALGO_AUTO, splits=0, A=0, B=0, C=0) -> tuple[int, dict]:
    info = PlanInfo()
    st = load().gemm_f32_plan(M, N, K, algo, splits, _p(A), _p(B), _p(C), ctypes.byref(info))
    return st, info.as_dict()


def gemm_f32_plan_ex(transa, transb, M, N, K, lda, ldb, ldc, algo=ALGO_AUTO, splits=0, A=0,
                     B=0, C=0) -> tuple[int, dict]:
    """The plan gemm_f32_ex would run for these transposes, sizes and leading
    dimensions (pointers optional: they only decide the alignment copies)."""
    info = PlanInfo()
    st = load().gemm_f32_plan_ex(int(transa), int(transb), M, N, K, _p(A), int(lda), _p(B),
                                 int(ldb), _p(C), int(ldc), int(algo), int(splits),
                                 ctypes.byref(info))
    return st, info.as_dict()


def gemm_f32_device_status(clear: int = 1) -> int:
    return load().gemm_f32_device_status(int(clear))


def gemm_f32_selftest_watchdog(timeout_ns: int, stream=0) -> int:
    return load().gemm_f32_selftest_watchdog(int(timeout_ns), _p(stream))


def gemm_f32_noalloc_selftest_watchdog(timeout_ns: int, stream=0) -> int:
    """Watchdog self-test on gemm_f32_noalloc's fault word (left set for the status call)."""
    return load().gemm_f32_noalloc_selftest_watchdog(int(timeout_ns), _p(stream))


INJECT_NONE = 0
INJECT_WORKSPACE = 1
INJECT_DESCRIPTOR = 2


def gemm_f32_inject_host_fault(kind: int) -> int:
    """Testing aid: the next workspace allocation (1) or descriptor encoding (2) fails; 0 disarms."""
    return load().gemm_f32_inject_host_fault(int(kind))


def gemm_f32_release() -> int:
    return load().gemm_f32_release()


def gemm_f32_status_string(status: int) -> str:
    try:
        return load().gemm_f32_status_string(int(status)).decode()
    except ImportError:
        return "library not loaded"


def gemm_f32_version() -> int:
    return load().gemm_f32_version()


def check(status: int, where: str = "gemm_f32") -> None:
    if status != SUCCESS:
        raise GemmError(status, where)


def matmul(A, B, out=None, algo=ALGO_AUTO, splits=0, stream=None):
    """``out = A @ B`` for float32 CUDA tensors, through ``gemm_f32_algo_splitk``.

    ``A`` is (M, K), ``B`` is (K, N), both row-major contiguous on the current
    device; ``out`` (M, N) is allocated if not given.  ``stream`` is a
    ``torch.cuda.Stream`` (default: the current stream).
    """
    import torch

    if isinstance(algo, str):
        algo = ALGOS[algo]
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}")
    for t in (A, B):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("A and B must be contiguous float32 CUDA tensors")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif out.shape != (M, N) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 (M, N) tensor")
    s = stream if stream is not None else torch.cuda.current_stream(A.device)
    with torch.cuda.device(A.device):
        st = gemm_f32_algo_splitk(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, int(algo),
                                  int(splits), s.cuda_stream)
    check(st, "matmul")
    return out
