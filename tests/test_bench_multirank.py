"""The benchmark's multi-rank arithmetic on CPU: two gloo ranks.

Under torchrun every rank runs an independent replica of the GEMM; the
harness takes the max of the per-rank times and reports the total work of
all ranks over that time.  This runs those reductions with world size 2 on
the gloo backend, no GPU involved.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    w, r, _ = bench.dist_env()
    assert (w, r) == (world, rank)
    dist = bench.dist_init(w, "gloo")
    try:
        # rank-dependent per-rank times (ms) and work
        t_ms = 10.0 + 5.0 * rank
        tmax = bench.reduce_max(t_ms, w)
        units = bench.reduce_sum(1.0, w)
        bench.barrier(w)
        q.put((rank, tmax, units))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_total_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    for _, tmax, units in got:
        assert tmax == 15.0 and units == 2.0


def test_single_process_reductions_are_identity():
    import bench

    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.reduce_sum(2.0, 1) == 2.0
    bench.barrier(1)


def test_clock_summary_parses_nvidia_smi_csv():
    import bench

    text = ("index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], x, a, b, c, d\n"
            "0, 1980, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
            "0, 2010, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active\n"
            "0, 300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    s = bench.ClockSampler.summarise(text)
    assert s["samples"] == 3 and s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == 1995.0  # median of the samples under load
    assert s["reasons"] == ["sw_power_cap"]
