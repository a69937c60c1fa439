"""Seeded synthetic inputs for the five row-major FP32 GEMM workloads.

This module only draws numbers. It holds no matrix arithmetic, so both the CPU
oracle's tests and the CUDA path's tests can take their inputs from here
without sharing any of the method's code.

Generators (all deterministic, all vectorised with numpy, all bit-reproducible
on any host except the normal draw, whose transcendental functions come from
the host's libm through numpy):

* ``quantised_fill(n, seed)`` -- the lecture-5 host initialiser of
  "Lecture 5: tiled matrix multiply" (runguoli.com ECE408 notes, l5,
  ``fillMatrix`` in ``tiled_matmul_basic.cu``): element ``i`` is hashed as
  ``x = (i + 7919*seed) mod 2^32``, ``x = (1103515245*x + 12345) mod 2^32``,
  and mapped to ``(((x >> 16) & 7) - 3) / 4``, one of the eight values
  -0.75, -0.5, ..., 1.0.  Every value has at most three significant bits.
* ``uniform_stream(n, state)`` -- the lecture-12 project-template generator
  ("Lecture 12: final project", l12, section 6, ``frand``): a 32-bit LCG
  ``s <- 1664525*s + 1013904223 (mod 2^32)`` that is advanced *before* each
  draw; the draw is ``((s >> 8) & 0xFFFFFF) / 2^24 * 2 - 1``, an exact float in
  [-1, 1) on a 2^-23 grid.  The matrices are filled A first, then B, from one
  continuing stream.
* ``normal_stream(n, state)`` -- N(0,1) draws for the 8192^3 workload.  The
  pages give no normal generator; this is the plainest reading on top of the
  same LCG: Box-Muller on pairs ``u = (((s >> 8) & 0xFFFFFF) + 1) / 2^24`` in
  (0, 1], ``r = sqrt(-2 ln u1)``, values ``r cos(2 pi u2)`` then
  ``r sin(2 pi u2)``, computed in double and rounded once to float32.

``make_workload(index)`` returns ``(A, B)`` for one of the five workloads in
``WORKLOADS``; the seeds are the page's seeds (1 and 2 for the quantised
case, 20250612 plus the workload index for the LCG streams).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "LCG_MUL",
    "LCG_ADD",
    "quantised_fill",
    "lcg_states",
    "uniform_stream",
    "normal_stream",
    "make_workload",
    "workload_by_name",
]

LCG_MUL = np.uint32(1664525)
LCG_ADD = np.uint32(1013904223)
_MASK32 = 0xFFFFFFFF


@dataclass(frozen=True)
class Workload:
    """One synthetic GEMM problem: shapes, value distribution and seeds."""

    index: int
    name: str
    M: int
    N: int
    K: int
    dist: str  # "quantised" | "uniform" | "normal"
    seed: int  # LCG start state, or the A seed of the quantised fill
    seed_b: int | None = None  # quantised fill only: the B seed

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


WORKLOADS: tuple[Workload, ...] = (
    Workload(0, "quantised_512", 512, 512, 512, "quantised", 1, 2),
    Workload(1, "ragged_1025x1023x1000", 1025, 1023, 1000, "uniform", 20250612 + 1),
    Workload(2, "square_2048", 2048, 2048, 2048, "uniform", 20250612 + 2),
    Workload(3, "square_8192_normal", 8192, 8192, 8192, "normal", 20250612 + 3),
    Workload(4, "deep_k_256x256x65536", 256, 256, 65536, "uniform", 20250612 + 4),
)


def workload_by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name or str(w.index) == str(name):
            return w
    raise KeyError(name)


# ---------------------------------------------------------------------------
# quantised hash fill (lecture 5)
# ---------------------------------------------------------------------------
def quantised_fill(n: int, seed: int) -> np.ndarray:
    """``n`` float32 values of the lecture-5 hash fill for ``seed``."""
    i = np.arange(n, dtype=np.uint64)
    x = (i + np.uint64((seed * 7919) & _MASK32)) & np.uint64(_MASK32)
    x = (x * np.uint64(1103515245) + np.uint64(12345)) & np.uint64(_MASK32)
    q = ((x >> np.uint64(16)) & np.uint64(7)).astype(np.int64) - 3
    return (q.astype(np.float32) * np.float32(0.25)).astype(np.float32)


# ---------------------------------------------------------------------------
# the lecture-12 LCG, vectorised by jump-ahead
# ---------------------------------------------------------------------------
_BLOCK = 1 << 16


def _jump_tables(block: int) -> tuple[np.ndarray, np.ndarray]:
    """mul[i], add[i] such that state after i+1 steps = mul[i]*s0 + add[i]."""
    mul = np.empty(block, dtype=np.uint64)
    add = np.empty(block, dtype=np.uint64)
    m, a = 1, 0
    a_lcg, c_lcg = int(LCG_MUL), int(LCG_ADD)
    for i in range(block):
        m = (m * a_lcg) & _MASK32
        a = (a * a_lcg + c_lcg) & _MASK32
        mul[i] = m
        add[i] = a
    return mul, add


_TABLES: dict[int, tuple[np.ndarray, np.ndarray]] = {}


def lcg_states(n: int, state: int) -> tuple[np.ndarray, int]:
    """The next ``n`` LCG states after ``state`` (each advanced before use).

    Returns ``(states[uint32, n], new_state)``.
    """
    if n == 0:
        return np.empty(0, dtype=np.uint32), state
    block = min(_BLOCK, n)
    if block not in _TABLES:
        # tables for the full block size are reused for any shorter tail
        _TABLES[block] = _jump_tables(block)
    mul, add = _TABLES[block]
    out = np.empty(n, dtype=np.uint32)
    s = np.uint64(state & _MASK32)
    mask = np.uint64(_MASK32)
    for start in range(0, n, block):
        cnt = min(block, n - start)
        seg = (mul[:cnt] * s + add[:cnt]) & mask
        out[start:start + cnt] = seg
        s = np.uint64(seg[-1])
    return out, int(s)


def uniform_stream(n: int, state: int) -> tuple[np.ndarray, int]:
    """``n`` draws of the lecture-12 ``frand`` from ``state``: float32 in [-1, 1)."""
    s, state = lcg_states(n, state)
    j = ((s >> np.uint32(8)) & np.uint32(0xFFFFFF)).astype(np.float64)
    v = j / 16777216.0 * 2.0 - 1.0  # exact in float64 and in float32
    return v.astype(np.float32), state


def normal_stream(n: int, state: int) -> tuple[np.ndarray, int]:
    """``n`` N(0,1) draws by Box-Muller on the LCG; consumes 2*ceil(n/2) states."""
    pairs = (n + 1) // 2
    s, state = lcg_states(2 * pairs, state)
    u = (((s >> np.uint32(8)) & np.uint32(0xFFFFFF)).astype(np.float64) + 1.0) / 16777216.0
    u1 = u[0::2]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return z[:n].astype(np.float32), state


def make_workload(w: Workload | int | str, *, M: int | None = None, N: int | None = None,
                  K: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Row-major ``A[M,K]`` and ``B[K,N]`` (float32, C-contiguous) for a workload.

    ``M``, ``N`` and ``K`` may override the workload's shape (same distribution
    and seeds, the element index runs over the overridden matrix).
    """
    if not isinstance(w, Workload):
        w = workload_by_name(str(w))
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    if w.dist == "quantised":
        A = quantised_fill(M * K, w.seed)
        B = quantised_fill(K * N, w.seed_b)
    elif w.dist == "uniform":
        A, st = uniform_stream(M * K, w.seed)
        B, _ = uniform_stream(K * N, st)
    elif w.dist == "normal":
        A, st = normal_stream(M * K, w.seed)
        B, _ = normal_stream(K * N, st)
    else:
        raise ValueError(w.dist)
    return A.reshape(M, K), B.reshape(K, N)
