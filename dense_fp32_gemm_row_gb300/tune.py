"""Design-space sweep of the GEMM kernels: try, check, time, rank.

    python -m dense_fp32_gemm_row_gb300.tune [--shapes 2048x2048x2048,...]
                                             [--repeats 10] [--csv out.csv]
                                             [--quick]

The library-side counterpart of the sweep program of "Lecture 12: final
project" (block size x tile depth x coarsening, each combination checked for
correctness before it is timed, then ranked).  Here the configuration space
is the library's own: algorithm (CUDA-core FFMA or 3xTF32 tensor cores) x
tile (128x128, 128x256, and for 3xTF32 the 256x256 two-CTA tile, fed by
staging kernels or splitting its operands in shared memory, and a 128x128
tile that splits in shared memory too) x split-K factor.  Every configuration
runs once through ``gemm_f32_configured`` and must pass a correctness check
before it is timed.  From the command line that check is cuBLAS SGEMM (TF32
off) within 1e-3 + 1e-3 |ref| on every output: this module belongs to the
library and does not load the test suite's CPU oracle.  ``sweep(check=...)``
takes any other check, and the test suite runs the sweep with the oracle as
its check.  Timing is the median of ``--repeats`` calls (CUDA events, L2
flushed between calls when the inputs fit in it; the configurations of a
shape are timed round-robin, one call each per round, each round starting
at the next configuration).  The library's own choice
(``gemm_f32``, AUTO) is timed alongside so the table shows how far AUTO is
from the best configuration per shape.

Prints one CSV row per configuration and a summary line per shape.
``--quick`` narrows the space to the tensor-core tiles with the library's
own split-K choice (splits = 0), the check of AUTO's tile rules.
"""

from __future__ import annotations

import argparse
import csv
import statistics
import sys

DEFAULT_SHAPES = ("512x512x512,1025x1023x1000,2048x2048x2048,4096x4096x4096,"
                  "256x256x65536,8192x8192x8192")
SPLITS = (1, 2, 4, 8, 16, 32, 64)


def _configs(g, quick: bool = False):
    if quick:
        for tile in (g.TILE_128x128, g.TILE_128x256, g.TILE_256x256_PAIR,
                     g.TILE_256x256_PAIR_SPLIT, g.TILE_128x128_SPLIT, g.TILE_128x128_TMEM,
                     g.TILE_256x256_TMEM, g.TILE_256x128_TMEM):
            yield g.ALGO_3XTF32, tile, 0
        return
    for algo, tiles in ((g.ALGO_FFMA, (g.TILE_128x128, g.TILE_128x256)),
                        (g.ALGO_3XTF32, (g.TILE_128x128, g.TILE_128x256, g.TILE_256x256_PAIR,
                                         g.TILE_256x256_PAIR_SPLIT, g.TILE_128x128_SPLIT,
                                         g.TILE_128x128_TMEM, g.TILE_256x256_TMEM,
                                         g.TILE_256x128_TMEM))):
        for tile in tiles:
            for splits in SPLITS:
                yield algo, tile, splits


def sweep(shapes, repeats: int, out=sys.stdout, quick: bool = False, check=None) -> list[dict]:
    """Check, time and rank every configuration on each (M, N, K) shape.

    ``check(a, b, c) -> bool`` decides whether the output ``c`` of ``a @ b``
    (device tensors) is correct; the default compares it with cuBLAS SGEMM.
    """
    import torch

    import dense_fp32_gemm_row_gb300 as g

    g.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    names = {g.ALGO_FFMA: "ffma", g.ALGO_3XTF32: "3xtf32", g.ALGO_AUTO: "auto"}
    tiles = {0: "auto", 1: "128x128", 2: "128x256", 3: "256x256pair", 4: "256x256pair-split",
             5: "128x128-split", 6: "128x128-tmem", 7: "256x256pair-tmem", 8: "256x128-tmem"}
    writer = csv.writer(out)
    writer.writerow(["shape", "algo", "tile", "splits", "ctas", "kernels", "ms", "tflops",
                     "check", "rank"])
    rows = []
    for shape in shapes:
        M, N, K = shape
        gen = torch.Generator(device=dev).manual_seed(M * 31 + N * 7 + K)
        a = torch.rand((M, K), device=dev, generator=gen) * 2 - 1
        b = torch.rand((K, N), device=dev, generator=gen) * 2 - 1
        c = torch.empty((M, N), device=dev)
        if check is None:
            prev = torch.backends.cuda.matmul.allow_tf32
            torch.backends.cuda.matmul.allow_tf32 = False
            ref = a @ b
            torch.backends.cuda.matmul.allow_tf32 = prev

            def passes(c=c, ref=ref):
                return bool(((c - ref).abs() <= 1e-3 + 1e-3 * ref.abs()).all().item())
        else:
            def passes(c=c, a=a, b=b):
                return bool(check(a, b, c))
        fits_l2 = 4 * (M * K + K * N) < 256 * 1024 * 1024
        flops = 2.0 * M * N * K

        def timed_once(call):
            if fits_l2:
                flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1)

        # every configuration is checked first, then all passing ones are
        # timed round-robin (one call each per round), so that none is
        # favoured or penalised by its place in the order (clock and cache
        # state drift over a shape's run)
        results, calls = [], []
        candidates = [(g.ALGO_AUTO, 0, 0)] + list(_configs(g, quick))
        for algo, tile, splits in candidates:
            st, plan = (g.gemm_f32_plan(M, N, K, algo, splits, a.data_ptr(), b.data_ptr(),
                                        c.data_ptr()) if algo == g.ALGO_AUTO else
                        g.gemm_f32_plan_config(M, N, K, algo, tile, splits, a.data_ptr(),
                                               b.data_ptr(), c.data_ptr()))
            if st != 0 or (splits and plan["splits"] != splits):
                continue  # not a distinct configuration (e.g. more splits than K blocks)

            def call(algo=algo, tile=tile, splits=splits):
                if algo == g.ALGO_AUTO:
                    g.check(g.gemm_f32(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                       stream.cuda_stream), "gemm_f32")
                else:
                    g.check(g.gemm_f32_configured(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N,
                                                  K, algo, tile, splits, stream.cuda_stream),
                            "gemm_f32_configured")

            c.fill_(float("nan"))
            call()
            stream.synchronize()
            ok = passes()
            results.append({"shape": f"{M}x{N}x{K}", "algo": names[algo],
                            "tile": tiles[tile] if algo != g.ALGO_AUTO else
                            f"{plan['tile_m']}x{plan['tile_n']}"
                            + ("-tmem" if plan.get("b_in_tmem") else
                               "-split" if plan.get("split_in_kernel") else ""),
                            "splits": plan["splits"], "ctas": plan["ctas"],
                            "kernels": plan["kernels"], "ms": float("nan"), "tflops": 0.0,
                            "check": "pass" if ok else "FAIL", "auto": algo == g.ALGO_AUTO})
            calls.append(call if ok else None)
        live = [i for i, cl in enumerate(calls) if cl is not None]
        for i in live:
            for _ in range(2):
                calls[i]()
        times = {i: [] for i in live}
        for r in range(repeats):
            # each round starts at the next configuration: the first call of
            # a round measured slower (by 2-10 us on calls of ~20 us), and
            # the rotation spreads that over all of them
            k = r % len(live)
            for i in live[k:] + live[:k]:
                times[i].append(timed_once(calls[i]))
        for i in live:
            ms = statistics.median(times[i])
            results[i]["ms"] = ms
            results[i]["tflops"] = flops / (ms * 1e-3) / 1e12
        ranked = sorted((r for r in results if r["check"] == "pass" and not r["auto"]),
                        key=lambda r: r["ms"])
        for i, r in enumerate(ranked):
            r["rank"] = i + 1
        for r in results:
            writer.writerow([r["shape"], r["algo"], r["tile"], r["splits"], r["ctas"],
                             r["kernels"], f"{r['ms']:.4f}", f"{r['tflops']:.2f}", r["check"],
                             r.get("rank", "auto" if r["auto"] else "")])
        auto = next(r for r in results if r["auto"])
        if ranked:
            best = ranked[0]
            print(f"# {best['shape']}: best {best['algo']} {best['tile']} splits {best['splits']}"
                  f" {best['ms']:.4f} ms ({best['tflops']:.1f} TFLOPS); auto {auto['tile']} "
                  f"splits {auto['splits']} {auto['ms']:.4f} ms "
                  f"({100 * best['ms'] / auto['ms']:.0f}% of best)", file=out, flush=True)
        rows += results
    return rows


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--shapes", default=DEFAULT_SHAPES)
    ap.add_argument("--repeats", type=int, default=10)
    ap.add_argument("--csv", default=None, help="also write the table to this file")
    ap.add_argument("--quick", action="store_true",
                    help="3xTF32 tiles with the library's split-K choice only")
    args = ap.parse_args(argv)
    shapes = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",") if s]
    if args.csv:
        with open(args.csv, "w") as f:
            sweep(shapes, args.repeats, out=f, quick=args.quick)
        with open(args.csv) as f:
            sys.stdout.write(f.read())
    else:
        sweep(shapes, args.repeats, quick=args.quick)
    return 0


if __name__ == "__main__":
    sys.exit(main())
