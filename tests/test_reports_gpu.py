"""The sweep and scaling-report tools, checked against the CPU oracle.

The design-space sweep (the library's counterpart of the sweep program of
"Lecture 12: final project") runs here with the oracle as its correctness
gate on two small shapes, and every configuration it times must pass it.
The scaling report (``bench.py --curve``, the counterpart of that page's
roofline report program) runs on two small sizes; its CSV must carry the
report's columns, an occupancy for the library's kernels and an oracle check
that passed for every kernel, cuBLAS included.
"""

import csv
import io
import os
import subprocess
import sys

import numpy as np
import pytest

import dense_fp32_gemm_row_gb300 as g
import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _oracle_check(a, b, c):
    want = oracle.ref_gemm(a.cpu().numpy(), b.cpu().numpy())
    return oracle.compare(c.cpu().numpy(), want)["pass"]


def test_sweep_with_the_oracle_as_its_gate():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available()
    from dense_fp32_gemm_row_gb300 import tune

    out = io.StringIO()
    rows = tune.sweep([(300, 260, 1000), (256, 256, 4096)], repeats=1, out=out, quick=False,
                      check=_oracle_check)
    assert rows, "no configuration ran"
    bad = [r for r in rows if r["check"] != "pass"]
    assert not bad, bad
    assert all(r["tflops"] > 0 for r in rows)
    # every shape has the library's own choice and a ranked best
    text = out.getvalue()
    assert text.count("# 300x260x1000: best") == 1 and text.count("# 256x256x4096: best") == 1
    g.gemm_f32_release()


def test_curve_report_columns_and_oracle_check():
    env = dict(os.environ)
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--curve",
                           "--curve-sizes", "128,300", "--steps", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    rows = list(csv.DictReader(io.StringIO(proc.stdout)))
    assert [r["kernel"] for r in rows] == ["ffma", "3xtf32", "cublas"] * 2
    assert {int(r["size"]) for r in rows} == {128, 300}
    for r in rows:
        assert r["check"] == "pass", r
        assert int(r["checked"]) == int(r["size"]) ** 2
        assert float(r["ms"]) > 0 and float(r["tflops"]) > 0
        n = int(r["size"])
        assert np.isclose(float(r["ai"]), 2.0 * n ** 3 / (12.0 * n * n), rtol=0.01)
        if r["kernel"] != "cublas":
            assert 0.0 < float(r["occup"]) <= 1.0, r
