"""Helpers for the GPU parity tests: upload, call through the C ABI with
guard bands around C, download, and compare with the oracle."""

from __future__ import annotations

import numpy as np

import dense_fp32_gemm_row_gb300 as g

GUARD = 4096  # floats of sentinel before and after C
SENTINEL_BITS = np.uint32(0x7FC0DEAD)  # a quiet NaN with a distinctive payload


def torch():
    import torch as _t
    return _t


def upload(a: np.ndarray, offset: int = 0):
    """Device copy of ``a``; ``offset`` floats of padding in front (misaligns the pointer)."""
    t = torch()
    flat = np.ascontiguousarray(a, dtype=np.float32).ravel()
    buf = t.empty(flat.size + offset + 1, dtype=t.float32, device="cuda")
    view = buf[offset:offset + flat.size]
    view.copy_(t.from_numpy(flat))
    return buf, view


def run(A: np.ndarray, B: np.ndarray, algo: int = g.ALGO_AUTO, splits: int = 0,
        offsets=(0, 0, 0), stream=None, check_guards: bool = True) -> np.ndarray:
    """C = A @ B on the GPU through gemm_f32_algo_splitk; returns C as numpy."""
    t = torch()
    M, K = A.shape
    N = B.shape[1]
    _, a = upload(A, offsets[0])
    _, b = upload(B, offsets[1])
    cbuf = t.empty(M * N + 2 * GUARD + offsets[2], dtype=t.float32, device="cuda")
    cbuf.view(t.int32).fill_(int(SENTINEL_BITS.view(np.int32)))
    c = cbuf[GUARD + offsets[2]:GUARD + offsets[2] + M * N]
    s = stream if stream is not None else t.cuda.current_stream()
    st = g.gemm_f32_algo_splitk(a.data_ptr() if a.numel() else 0,
                                b.data_ptr() if b.numel() else 0,
                                c.data_ptr() if c.numel() else 0, M, N, K, algo, splits,
                                s.cuda_stream)
    g.check(st, "gemm_f32_algo_splitk")
    s.synchronize()
    g.check(g.gemm_f32_device_status(1), "device status")
    host = cbuf.cpu().numpy()
    if check_guards:
        lo = host[:GUARD + offsets[2]].view(np.uint32)
        hi = host[GUARD + offsets[2] + M * N:].view(np.uint32)
        assert np.all(lo == SENTINEL_BITS), "write before C"
        assert np.all(hi == SENTINEL_BITS), "write after C"
    return host[GUARD + offsets[2]:GUARD + offsets[2] + M * N].reshape(M, N).copy()


def run_configured(A: np.ndarray, B: np.ndarray, algo: int, tile: int, splits: int = 0,
                   offsets=(0, 0, 0)) -> np.ndarray:
    """C = A @ B through gemm_f32_configured (forced kernel configuration),
    with the same guard bands as ``run``."""
    t = torch()
    M, K = A.shape
    N = B.shape[1]
    _, a = upload(A, offsets[0])
    _, b = upload(B, offsets[1])
    cbuf = t.empty(M * N + 2 * GUARD + offsets[2], dtype=t.float32, device="cuda")
    cbuf.view(t.int32).fill_(int(SENTINEL_BITS.view(np.int32)))
    c = cbuf[GUARD + offsets[2]:GUARD + offsets[2] + M * N]
    s = t.cuda.current_stream()
    g.check(g.gemm_f32_configured(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, algo, tile,
                                  splits, s.cuda_stream), "gemm_f32_configured")
    s.synchronize()
    g.check(g.gemm_f32_device_status(1), "device status")
    host = cbuf.cpu().numpy()
    assert np.all(host[:GUARD + offsets[2]].view(np.uint32) == SENTINEL_BITS), "write before C"
    assert np.all(host[GUARD + offsets[2] + M * N:].view(np.uint32) == SENTINEL_BITS), \
        "write after C"
    return host[GUARD + offsets[2]:GUARD + offsets[2] + M * N].reshape(M, N).copy()
