"""The seeded generators against scalar restatements of their definitions.

The vectorised generators in ``seeded_inputs`` jump the LCG ahead in blocks;
these tests walk the same recurrences one step at a time in plain Python and
compare, across a block boundary.  Frozen digests of the LCG-based workloads
catch any later change of the streams.
"""

import hashlib
import json
import math
import os

import numpy as np
import pytest

from seeded_inputs import (WORKLOADS, lcg_states, make_workload, normal_stream, quantised_fill,
                           uniform_stream)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "generator_sha256.json")


def _scalar_lcg(state, n):
    out = []
    for _ in range(n):
        state = (state * 1664525 + 1013904223) & 0xFFFFFFFF
        out.append(state)
    return out, state


def test_quantised_fill_matches_scalar_hash():
    for seed in (1, 2, 3, 4):
        got = quantised_fill(3000, seed)
        want = []
        for i in range(3000):
            x = (i + seed * 7919) & 0xFFFFFFFF
            x = (x * 1103515245 + 12345) & 0xFFFFFFFF
            want.append((((x >> 16) & 7) - 3) * 0.25)
        assert np.array_equal(got, np.array(want, np.float32))
    assert set(np.unique(quantised_fill(100000, 1)).tolist()) <= {k / 4 for k in range(-3, 5)}


def test_lcg_states_cross_block_boundary():
    n = (1 << 16) + 4321
    got, end = lcg_states(n, 20250612)
    want, wend = _scalar_lcg(20250612, n)
    assert end == wend
    assert np.array_equal(got, np.array(want, np.uint32))


def test_uniform_stream_matches_frand():
    got, st = uniform_stream(5000, 20250612)
    states, st2 = _scalar_lcg(20250612, 5000)
    want = [((s >> 8) & 0xFFFFFF) / 16777216.0 * 2.0 - 1.0 for s in states]
    assert st == st2
    assert np.array_equal(got, np.array(want, np.float32))
    assert got.min() >= -1.0 and got.max() < 1.0
    # continuing the stream equals one long draw (A then B)
    a, st = uniform_stream(777, 5)
    b, _ = uniform_stream(555, st)
    ab, _ = uniform_stream(1332, 5)
    assert np.array_equal(np.concatenate([a, b]), ab)


def test_normal_stream_matches_scalar_box_muller():
    got, st = normal_stream(4001, 20250615)
    states, st2 = _scalar_lcg(20250615, 4002)
    assert st == st2
    want = []
    for p in range(2001):
        u1 = (((states[2 * p] >> 8) & 0xFFFFFF) + 1) / 16777216.0
        u2 = (((states[2 * p + 1] >> 8) & 0xFFFFFF) + 1) / 16777216.0
        r = math.sqrt(-2.0 * math.log(u1))
        want += [r * math.cos(2 * math.pi * u2), r * math.sin(2 * math.pi * u2)]
    want = np.array(want[:4001], np.float32)
    # numpy's vectorised libm and Python's scalar libm may differ in the last
    # double bit; after rounding to float32 at most one ulp can move
    ulps = np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    big, _ = normal_stream(200000, 1)
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1.0) < 0.01


def _digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


@pytest.mark.parametrize("index", [0, 1, 2, 4])
def test_workload_streams_are_frozen(index):
    with open(GOLDEN) as f:
        golden = json.load(f)
    A, B = make_workload(index)
    w = WORKLOADS[index]
    assert A.shape == (w.M, w.K) and B.shape == (w.K, w.N)
    assert A.dtype == np.float32 and A.flags.c_contiguous
    assert golden[w.name] == {"A": _digest(A), "B": _digest(B)}
